"""Host-buffer forward through the C ABI: pipelined calls give the same bits as the
device-buffer forward."""
import pytest
import torch

import dit_inputs as di
import diffusion_transformer_block_gb300 as kd
from gpu_helpers import make_block, upload

pytestmark = pytest.mark.gpu


def test_forward_host_matches_device_forward():
    cfg = di.CONFIGS["small_a"]
    cases = [di.make_case(cfg.replace(seed=cfg.seed + i)) for i in range(3)]
    blk = make_block(cfg)
    try:
        t, _, _ = upload(blk, cases[0])
        ms = blk.timestep_embed(t)
        kd.krea_dit_block_enable_host_io(blk.handle)
        ref = []
        for c in cases:
            ref.append(blk.forward(c.dev["x_img"].cuda(), c.dev["x_txt"].cuda(), cfg.B, cfg.img_h, cfg.img_w,
                                   cfg.n_txt, ms).cpu())
        outs = [torch.full((cfg.B, cfg.L, cfg.d), float("nan"), dtype=torch.bfloat16).pin_memory() for _ in cases]
        ins = [(c.dev["x_img"].contiguous().pin_memory(), c.dev["x_txt"].contiguous().pin_memory()) for c in cases]
        stream = torch.cuda.current_stream()
        for (xi, xt), o in zip(ins, outs):  # three calls in flight: staging sets alternate
            kd.krea_dit_block_forward_host(blk.handle, xi, xt, cfg.B, cfg.img_h, cfg.img_w, cfg.n_txt, ms,
                                           blk._wstruct, o, stream)
        kd.krea_dit_block_host_sync(blk.handle)
        for r, o in zip(ref, outs):
            assert torch.equal(r, o)
        # refused before enable / bad sizes: nothing enqueued
        assert kd.lib().krea_dit_block_forward_host(blk.handle, kd._ptr(ins[0][0]), kd._ptr(ins[0][1]), cfg.B + 1,
                                                    cfg.img_h, cfg.img_w, cfg.n_txt, kd._ptr(ms),
                                                    kd.ctypes.byref(blk._wstruct), kd._ptr(outs[0]), None) == \
            kd.KREA_DIT_ERR_EXCEEDS_CREATE_LIMITS
    finally:
        blk.close()
