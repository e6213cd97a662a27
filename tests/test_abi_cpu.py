"""The C-ABI library builds, loads and exports every symbol its header declares; host-side
argument checks answer without a GPU (no compute call is made here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "krea_dit.h")


@pytest.fixture(scope="module")
def lib():
    import diffusion_transformer_block_gb300 as kd
    if not os.path.exists(kd.LIB_PATH):
        from diffusion_transformer_block_gb300 import build
        build.build()
    return kd


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^(?:int|size_t|const char\*)\s+(krea_dit_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("krea_dit_block_create", "krea_dit_block_destroy", "krea_dit_block_forward",
              "krea_dit_timestep_embed", "krea_dit_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    so = ctypes.CDLL(lib.LIB_PATH)
    for n in declared_functions():
        assert hasattr(so, n), n
    assert sorted(lib.EXPORTS) == declared_functions()


def test_status_strings(lib):
    assert lib.krea_dit_status_string(0) == "ok"
    for code in range(-9, 0):
        assert lib.krea_dit_status_string(code) != "unknown status"
    assert lib.krea_dit_status_string(-99) == "unknown status"


def test_host_checks_without_gpu(lib):
    L = lib.lib()
    h = ctypes.c_void_p(123)
    assert L.krea_dit_block_create(None, ctypes.byref(h)) == lib.KREA_DIT_ERR_INVALID_ARG
    assert h.value is None
    bad = lib.make_config(max_batch=1, max_seq=8, d_model=100, n_q=2, n_kv=1, head_dim=128, ffn=256, img_h_max=2,
                          img_w_max=2)
    assert L.krea_dit_block_create(ctypes.byref(bad), ctypes.byref(h)) == lib.KREA_DIT_ERR_UNSUPPORTED_SHAPE
    bad = lib.make_config(max_batch=1, max_seq=8, d_model=256, n_q=2, n_kv=1, head_dim=64, ffn=256, img_h_max=2,
                          img_w_max=2)  # bf16 mode needs head_dim 128
    assert L.krea_dit_block_create(ctypes.byref(bad), ctypes.byref(h)) == lib.KREA_DIT_ERR_UNSUPPORTED_SHAPE
    assert L.krea_dit_block_forward(None, None, None, 1, 1, 1, 1, None, None, None, None) == \
        lib.KREA_DIT_ERR_INVALID_ARG
    assert L.krea_dit_block_destroy(None) == lib.KREA_DIT_OK
    names = lib.krea_dit_kernel_names()
    assert "attention_gate" in names and "upgate_gemm_swiglu" in names


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import diffusion_transformer_block_gb300 as kd
    monkeypatch.setattr(kd, "_lib", None)
    monkeypatch.setattr(kd, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        kd.lib()


def test_every_handle_call_rejects_a_null_handle(lib):
    """Each entry point that takes a handle answers INVALID_ARG for a null one, on the host,
    before any device work; the graph calls do the same for a null graph."""
    L = lib.lib()
    inv = lib.KREA_DIT_ERR_INVALID_ARG
    i = ctypes.c_int(0)
    p = ctypes.c_void_p(0)
    n = ctypes.c_size_t(0)
    calls = {
        "krea_dit_timestep_embed": lambda: L.krea_dit_timestep_embed(None, None, 1, None, None, None),
        "krea_dit_block_workspace": lambda: L.krea_dit_block_workspace(None, 0, ctypes.byref(p), ctypes.byref(n)),
        "krea_dit_block_set_timing": lambda: L.krea_dit_block_set_timing(None, 1),
        "krea_dit_block_timing_reset": lambda: L.krea_dit_block_timing_reset(None),
        "krea_dit_block_device_status": lambda: L.krea_dit_block_device_status(None, None, ctypes.byref(i)),
        "krea_dit_block_inject_fault": lambda: L.krea_dit_block_inject_fault(None, 0),
        "krea_dit_block_selftest_wait": lambda: L.krea_dit_block_selftest_wait(None, 1, 1000000, None),
        "krea_dit_block_enable_host_io": lambda: L.krea_dit_block_enable_host_io(None),
        "krea_dit_block_forward_host": lambda: L.krea_dit_block_forward_host(None, None, None, 1, 1, 1, 1, None, None,
                                                                             None, None),
        "krea_dit_block_host_sync": lambda: L.krea_dit_block_host_sync(None),
        "krea_dit_block_forward_joint": lambda: L.krea_dit_block_forward_joint(None, None, 1, 1, 1, 1, None, None, None,
                                                                               None),
        "krea_dit_stack_forward": lambda: L.krea_dit_stack_forward(None, None, 1, 1, 1, 1, None, None, 1, None),
        "krea_dit_graph_launch": lambda: L.krea_dit_graph_launch(None, None),
        "krea_dit_block_enable_backward": lambda: L.krea_dit_block_enable_backward(None),
        "krea_dit_stack_graph_create": lambda: L.krea_dit_stack_graph_create(None, None, 1, 1, 1, 1, None, None, 1, None,
                                                                             ctypes.byref(p)),
        "krea_dit_weights8_quantize": lambda: L.krea_dit_weights8_quantize(None, None, None, None),
        "krea_dit_block_backward": lambda: L.krea_dit_block_backward(None, None, None, 1, 1, 1, 1, None, None, None,
                                                                     None, None),
        "krea_dit_block_forward8": lambda: L.krea_dit_block_forward8(None, None, None, 1, 1, 1, 1, None, None, None,
                                                                     None, None),
        "krea_dit_weights4_quantize": lambda: L.krea_dit_weights4_quantize(None, None, None, None),
        "krea_dit_block_forward4": lambda: L.krea_dit_block_forward4(None, None, None, 1, 1, 1, 1, None, None, None,
                                                                     None, None),
    }
    for name, call in calls.items():
        assert call() == inv, name


def test_nvfp4_scale_bytes(lib):
    """ceil(rows / 128) * 128 rows of cols / 16 one-byte scales (host arithmetic only)."""
    f = lib.krea_dit_nvfp4_scale_bytes
    assert f(9216, 3072) == 9216 * 192
    assert f(1, 64) == 128 * 4
    assert f(130, 128) == 256 * 8
    assert f(0, 64) == 0 and f(5, 0) == 0
