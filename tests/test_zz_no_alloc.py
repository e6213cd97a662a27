"""The allocation-free timestep embedding, through the C ABI, against the fp64 oracle
and against the handle-based entry point.

Callers that cannot allocate device memory (a serving runtime that owns the whole
device through its own pool, a latency-critical loop that must not block on the
allocator) use krea_dit_timestep_embed_noalloc, whose scratch is a fixed library-owned
device array. This file is collected last so that a failure here leaves every other
test already run.
"""
import numpy as np
import pytest
import torch

import dit_inputs as di
import diffusion_transformer_block_gb300 as kd
import oracle
from gpu_helpers import make_block

pytestmark = pytest.mark.gpu

TOL = 1e-5  # the timestep-embedding tolerance of the handle-based test (x RMS)


def _inputs(cfg):
    case = di.make_case(cfg)
    tw = {k: case.dev["temb." + k].cuda().contiguous() for k in ("w1", "b1", "w2", "b2")}
    return case, tw, case.dev["t"].cuda()


def _err_vs(out: torch.Tensor, ref: np.ndarray) -> float:
    got = out.double().cpu().numpy()
    return float(np.abs(got - ref).max() / np.sqrt(np.mean(ref ** 2)))


def test_noalloc_matches_oracle_and_handle_entry_point_twice():
    cfg = di.CONFIGS["small_c"]
    case, tw, t = _inputs(cfg)
    ref_oracle = oracle.mod_shared_for(case)
    blk = make_block(cfg)
    try:
        blk.set_temb_weights({k: v for k, v in tw.items()})
        ref = blk.timestep_embed(t).clone()
    finally:
        blk.close()
    wstruct = kd.make_temb_weights(tw)
    outs = [torch.full((cfg.B, 6, cfg.d), float("nan"), device="cuda") for _ in range(2)]
    torch.cuda.synchronize()
    free_after = []
    for out in outs:  # two calls in a row share the scratch array
        kd.krea_dit_timestep_embed_noalloc(t, cfg.B, cfg.d, wstruct, out, torch.cuda.current_stream())
        torch.cuda.synchronize()
        free_after.append(torch.cuda.mem_get_info()[0])
    rms = ref.pow(2).mean().sqrt().item()
    for out in outs:
        assert torch.isfinite(out).all()
        assert (out - ref).abs().max().item() <= TOL * rms
        assert _err_vs(out, ref_oracle) <= TOL
    # the second call allocated nothing on the device
    assert free_after[1] == free_after[0]


def test_noalloc_other_width_matches_oracle_then_rejects_oversize():
    case, tw, t = _inputs(di.CONFIGS["small_a"])
    # width 512 with B = 2 fits; the same call with a batch past the scratch is refused
    assert case.cfg.d == 512 and case.cfg.B == 2
    wstruct = kd.make_temb_weights(tw)
    out = torch.zeros(2, 6, 512, device="cuda")
    kd.krea_dit_timestep_embed_noalloc(t, 2, 512, wstruct, out, torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    assert _err_vs(out, oracle.mod_shared_for(case)) <= TOL
    too_many = kd.KREA_DIT_NOALLOC_SCRATCH_FLOATS // (256 + 512) + 1
    big_t = torch.rand(too_many, device="cuda")
    big_out = torch.zeros(too_many, 6, 512, device="cuda")
    st = kd.lib().krea_dit_timestep_embed_noalloc(kd._ptr(big_t), too_many, 512, kd.ctypes.byref(wstruct),
                                                  kd._ptr(big_out), None)
    assert st == kd.KREA_DIT_ERR_SCRATCH_TOO_SMALL
    torch.cuda.synchronize()
    assert big_out.abs().max().item() == 0.0
