"""Host-side error handling through the C ABI on a GPU (nothing here faults the GPU:
every bad argument is rejected on the host before anything is enqueued)."""
import time

import pytest
import torch

import dit_inputs as di
import diffusion_transformer_block_gb300 as kd
from gpu_helpers import make_block, upload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def setup():
    cfg = di.CONFIGS["small_a"]
    case = di.make_case(cfg)
    blk = make_block(cfg)
    t, x_img, x_txt = upload(blk, case)
    ms = blk.timestep_embed(t)
    yield cfg, blk, x_img, x_txt, ms
    blk.close()


def _fwd(blk, x_img, x_txt, B, h, w, nt, ms, out):
    return kd.lib().krea_dit_block_forward(blk.handle, kd._ptr(x_img), kd._ptr(x_txt), B, h, w, nt, kd._ptr(ms),
                                           kd.ctypes.byref(blk._wstruct), kd._ptr(out), None)


def test_rejections(setup):
    cfg, blk, x_img, x_txt, ms = setup
    out = torch.empty(cfg.B, cfg.L, cfg.d, device="cuda", dtype=torch.bfloat16)
    args = (cfg.img_h, cfg.img_w, cfg.n_txt)
    assert _fwd(blk, x_img, x_txt, cfg.B + 1, *args, ms, out) == kd.KREA_DIT_ERR_EXCEEDS_CREATE_LIMITS
    assert _fwd(blk, x_img, x_txt, cfg.B, cfg.img_h + 1, cfg.img_w, cfg.n_txt, ms, out) == \
        kd.KREA_DIT_ERR_EXCEEDS_CREATE_LIMITS
    assert _fwd(blk, x_img, x_txt, -1, *args, ms, out) == kd.KREA_DIT_ERR_INVALID_ARG
    assert _fwd(blk, None, x_txt, cfg.B, *args, ms, out) == kd.KREA_DIT_ERR_INVALID_ARG
    assert _fwd(blk, x_img, x_txt, cfg.B, *args, None, out) == kd.KREA_DIT_ERR_INVALID_ARG
    big = torch.empty(cfg.B * cfg.L * cfg.d + 8, device="cuda", dtype=torch.bfloat16)
    assert _fwd(blk, x_img, x_txt, cfg.B, *args, ms, big[1:]) == kd.KREA_DIT_ERR_MISALIGNED
    # output aliasing an input
    assert _fwd(blk, x_img, x_txt, cfg.B, *args, ms, x_img) == kd.KREA_DIT_ERR_INVALID_ARG
    st, site = kd.krea_dit_block_device_status(blk.handle)
    assert st == kd.KREA_DIT_OK and site == 0


def test_empty_calls_are_noops(setup):
    cfg, blk, x_img, x_txt, ms = setup
    out = torch.full((1,), 7.0, device="cuda")
    assert _fwd(blk, x_img, x_txt, 0, cfg.img_h, cfg.img_w, cfg.n_txt, ms, out) == kd.KREA_DIT_OK
    assert _fwd(blk, None, None, cfg.B, 0, 0, 0, ms, out) == kd.KREA_DIT_OK
    torch.cuda.synchronize()
    assert out.item() == 7.0


def test_injected_fault_enqueues_nothing(setup):
    cfg, blk, x_img, x_txt, ms = setup
    out = torch.zeros(cfg.B, cfg.L, cfg.d, device="cuda", dtype=torch.bfloat16)
    kd.krea_dit_block_inject_fault(blk.handle, 1)
    assert _fwd(blk, x_img, x_txt, cfg.B, cfg.img_h, cfg.img_w, cfg.n_txt, ms, out) == kd.KREA_DIT_ERR_INJECTED
    torch.cuda.synchronize()
    assert out.abs().max().item() == 0.0
    assert _fwd(blk, x_img, x_txt, cfg.B, cfg.img_h, cfg.img_w, cfg.n_txt, ms, out) == kd.KREA_DIT_OK
    torch.cuda.synchronize()
    assert out.abs().max().item() > 0.0


def test_bounded_wait_gives_up_and_the_handle_stays_usable(setup):
    """A wait on an mbarrier that nothing arrives at, through the same routine every
    tensor-core kernel waits with (limit 1 ms here instead of about a second), gives up:
    the call returns, the device status names the site, the tensor memory the waiting
    CTAs held is free again (the next forward's kernels allocate 512 columns per SM),
    and the next forward on the same handle gives the same result as before."""
    cfg, blk, x_img, x_txt, ms = setup
    before = blk.forward(x_img, x_txt, cfg.B, cfg.img_h, cfg.img_w, cfg.n_txt, ms).clone()
    torch.cuda.synchronize()
    assert kd.krea_dit_block_device_status(blk.handle) == (kd.KREA_DIT_OK, 0)
    for site in (kd.SITES["ATTN_MMA"], kd.SITES["GEMM_PRODUCER"], kd.SITES["ATTN_TEARDOWN"]):
        t0 = time.perf_counter()
        kd.krea_dit_block_selftest_wait(blk.handle, site, 1_000_000)
        st, got = kd.krea_dit_block_device_status(blk.handle)
        assert time.perf_counter() - t0 < 10.0
        assert st == kd.KREA_DIT_ERR_DEVICE_TIMEOUT and got == site
        assert kd.krea_dit_block_device_status(blk.handle) == (kd.KREA_DIT_OK, 0)  # read and cleared
        after = blk.forward(x_img, x_txt, cfg.B, cfg.img_h, cfg.img_w, cfg.n_txt, ms)
        torch.cuda.synchronize()
        assert torch.equal(after, before)
        assert kd.krea_dit_block_device_status(blk.handle) == (kd.KREA_DIT_OK, 0)
    # out-of-range arguments are rejected on the host
    L = kd.lib()
    assert L.krea_dit_block_selftest_wait(blk.handle, 0, 1_000_000, None) == kd.KREA_DIT_ERR_INVALID_ARG
    assert L.krea_dit_block_selftest_wait(blk.handle, 0x100, 1_000_000, None) == kd.KREA_DIT_ERR_INVALID_ARG
    assert L.krea_dit_block_selftest_wait(blk.handle, 1, 10, None) == kd.KREA_DIT_ERR_INVALID_ARG
    assert L.krea_dit_block_selftest_wait(blk.handle, 1, 2_000_000_000, None) == kd.KREA_DIT_ERR_INVALID_ARG


def test_timing_counts_launches(setup):
    cfg, blk, x_img, x_txt, ms = setup
    kd.krea_dit_block_set_timing(blk.handle, True)
    kd.krea_dit_block_timing_reset(blk.handle)
    for _ in range(3):
        blk.forward(x_img, x_txt, cfg.B, cfg.img_h, cfg.img_w, cfg.n_txt, ms)
    times = kd.krea_dit_block_kernel_times(blk.handle)
    kd.krea_dit_block_set_timing(blk.handle, False)
    assert set(times) == {"norm1_modulate", "qkvg_gemm_qknorm_rope", "attention_gate", "oproj_gemm_residual",
                          "norm2_modulate", "upgate_gemm_swiglu", "down_gemm_residual"}
    assert all(n == 3 and ms_ > 0 for ms_, n in times.values())


def test_create_rejects_bad_shapes():
    base = dict(max_batch=1, max_seq=16, d_model=256, n_q=4, n_kv=2, head_dim=128, ffn=512, img_h_max=4,
                img_w_max=4)
    for bad, code in [(dict(head_dim=64), kd.KREA_DIT_ERR_UNSUPPORTED_SHAPE),
                      (dict(d_model=200), kd.KREA_DIT_ERR_UNSUPPORTED_SHAPE),
                      (dict(n_kv=3), kd.KREA_DIT_ERR_UNSUPPORTED_SHAPE),
                      (dict(max_batch=0), kd.KREA_DIT_ERR_INVALID_ARG)]:
        cfg = kd.make_config(**{**base, **bad})
        h = kd.ctypes.c_void_p()
        assert kd.lib().krea_dit_block_create(kd.ctypes.byref(cfg), kd.ctypes.byref(h)) == code
        assert not h.value
