"""Canary-padded buffers: no kernel writes past the extent of its call.

compute-sanitizer is not available on the GPU pool, so out-of-range writes are looked
for directly. A handle created for a larger call first runs that larger call (so every
workspace buffer has a known extent of T_big rows), then every workspace buffer is
filled with a byte pattern, and a smaller call with a ragged shape (L not a multiple of
the 128-row tiles, T not a multiple of the 256-row GEMM tiles) runs on the same handle
with an output buffer that is itself padded with the pattern. Afterwards everything past
the small call's extent must still hold the pattern, byte for byte, and the small call's
result must match the fp64 oracle.
"""
import numpy as np
import pytest
import torch

import dit_inputs as di
import diffusion_transformer_block_gb300 as kd
from diffusion_transformer_block_gb300.runner import _DevView
from gpu_helpers import check_parity, make_block, run_gpu, upload

pytestmark = pytest.mark.gpu

PATTERN = 0x5A  # every byte of a canary region


def _byte_view(ptr: int, nbytes: int) -> torch.Tensor:
    return torch.as_tensor(_DevView(ptr, (nbytes,), "|u1"), device="cuda")


@pytest.mark.parametrize("name", ["small_a", "small_b"])
def test_no_write_past_the_call(name):
    cfg = di.CONFIGS[name]  # ragged: L = 116 (small_a), 357 (small_b)
    big = cfg.replace(img_h=cfg.img_h + 8, img_w=cfg.img_w + 4, n_txt=cfg.n_txt + 21, seed=cfg.seed + 100)
    blk = make_block(big)
    try:
        # the large call fixes each buffer's full extent
        run_gpu(di.make_case(big), blk=blk)
        names = ("XN", "Q", "K", "VT", "G", "OG", "H1", "HN", "HMID")
        full = {n: kd.krea_dit_block_workspace(blk.handle, n) for n in names}
        for n, (ptr, nbytes) in full.items():
            _byte_view(ptr, nbytes).fill_(PATTERN)
        case = di.make_case(cfg)
        t, x_img, x_txt = upload(blk, case)
        ms = blk.timestep_embed(t)
        n_out = cfg.B * cfg.L * cfg.d
        pad = 4096  # elements of canary after the output
        out_buf = torch.empty(n_out + pad, device="cuda", dtype=torch.bfloat16)
        out_buf.view(torch.uint8).fill_(PATTERN)
        out = out_buf[:n_out].view(cfg.B, cfg.L, cfg.d)
        blk.forward(x_img, x_txt, cfg.B, cfg.img_h, cfg.img_w, cfg.n_txt, ms, out=out)
        torch.cuda.synchronize()
        st, site = kd.krea_dit_block_device_status(blk.handle)
        assert st == kd.KREA_DIT_OK and site == 0
        # the output's padding is untouched
        tail = out_buf[n_out:].view(torch.uint8)
        assert bool((tail == PATTERN).all()), "a kernel wrote past the end of the output"
        # workspace past the small call's extent is untouched
        for n, (ptr, nbytes) in full.items():
            _, used = kd.krea_dit_block_workspace(blk.handle, n)
            assert 0 < used < nbytes, n
            rest = _byte_view(ptr + used, nbytes - used)
            bad = int((rest != PATTERN).sum().item())
            assert bad == 0, f"{n}: {bad} bytes written past the call's extent ({used} of {nbytes} used)"
        # and the small call is right: a second, ordinary call on the same handle gives the
        # same output bit for bit, and its output and intermediates match the oracle
        got = out.double().cpu().numpy()
        again = run_gpu(case, blk=blk)
        for b in range(cfg.B):
            np.testing.assert_array_equal(got[b], again["out"][b])
        check_parity(case, again)
    finally:
        blk.close()
