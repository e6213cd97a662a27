"""Python binding of the GB300 Krea 2 single-stream DiT block library (libkrea_dit.so).

Argument marshalling only: every step of the block runs in the library's CUDA kernels.
Functions carry the C ABI's names (see include/krea_dit.h for the operation, layouts,
ownership and errors); they accept raw device addresses (int) or torch tensors (their
``data_ptr()``), and raise ``KreaDitError`` on a non-zero status. There is no fallback:
if the shared library is missing, importing the binding's functions raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, List, Optional, Tuple

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkrea_dit.so")

KREA_DIT_OK = 0
KREA_DIT_ERR_INVALID_ARG = -1
KREA_DIT_ERR_UNSUPPORTED_SHAPE = -2
KREA_DIT_ERR_MISALIGNED = -3
KREA_DIT_ERR_EXCEEDS_CREATE_LIMITS = -4
KREA_DIT_ERR_CUDA = -5
KREA_DIT_ERR_NO_DEVICE = -6
KREA_DIT_ERR_DEVICE_TIMEOUT = -7
KREA_DIT_ERR_INJECTED = -8
KREA_DIT_ERR_SCRATCH_TOO_SMALL = -9
KREA_DIT_NOALLOC_SCRATCH_FLOATS = 262144
# sites of the bounded on-device waits (krea_dit_block_device_status)
SITES = {"GEMM_PRODUCER": 0x01, "GEMM_MMA": 0x02, "GEMM_EPILOGUE": 0x04, "GEMM_TEARDOWN": 0x08, "ATTN_LOAD": 0x10,
         "ATTN_MMA": 0x20, "ATTN_SOFTMAX": 0x40, "ATTN_TEARDOWN": 0x80}
KREA_DIT_BF16 = 0
KREA_DIT_FP32 = 1
KREA_DIT_FP8_TENSOR = 2
KREA_DIT_FP8_ROW = 3
KREA_DIT_NVFP4 = 4
BUFFERS = {"XN": 0, "Q": 1, "K": 2, "VT": 3, "G": 4, "OG": 5, "H1": 6, "HN": 7, "HMID": 8, "XN8": 9, "OG8": 10,
           "HN8": 11, "HMID8": 12, "DQ_XN": 13, "DQ_OG": 14, "DQ_HN": 15, "DQ_HMID": 16, "XN4": 17, "OG4": 18,
           "HN4": 19, "HMID4": 20, "SF_XN4": 21, "SF_OG4": 22, "SF_HN4": 23, "SF_HMID4": 24, "TS_XN4": 25,
           "TS_OG4": 26, "TS_HN4": 27, "TS_HMID4": 28}

# C symbols the header declares (checked by the CPU tests against the built library)
EXPORTS = [
    "krea_dit_block_create", "krea_dit_block_destroy", "krea_dit_timestep_embed", "krea_dit_block_forward",
    "krea_dit_status_string", "krea_dit_block_workspace", "krea_dit_block_set_timing",
    "krea_dit_block_kernel_times", "krea_dit_block_timing_reset", "krea_dit_block_device_status",
    "krea_dit_block_inject_fault", "krea_dit_kernel_names", "krea_dit_timestep_embed_noalloc",
    "krea_dit_block_enable_host_io", "krea_dit_block_forward_host", "krea_dit_block_host_sync",
    "krea_dit_block_forward_joint", "krea_dit_stack_forward", "krea_dit_stack_graph_create", "krea_dit_graph_launch",
    "krea_dit_graph_destroy", "krea_dit_weights8_quantize", "krea_dit_block_forward8",
    "krea_dit_block_enable_backward", "krea_dit_block_backward", "krea_dit_block_selftest_wait",
    "krea_dit_nvfp4_scale_bytes", "krea_dit_weights4_quantize", "krea_dit_block_forward4",
]


class KreaDitError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: status {status} ({krea_dit_status_string(status)})")


class krea_dit_config(ctypes.Structure):
    _fields_ = [("max_batch", ctypes.c_int), ("max_seq", ctypes.c_int), ("d_model", ctypes.c_int),
                ("n_q", ctypes.c_int), ("n_kv", ctypes.c_int), ("head_dim", ctypes.c_int), ("ffn", ctypes.c_int),
                ("img_h_max", ctypes.c_int), ("img_w_max", ctypes.c_int), ("eps", ctypes.c_float),
                ("rope_base", ctypes.c_float), ("gate_on", ctypes.c_int), ("mode", ctypes.c_int)]


class krea_dit_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "w_qkvg", "w_o", "w_gate", "w_up", "w_down", "norm1_w", "norm2_w", "q_norm_w", "k_norm_w", "mod_bias")]


class krea_dit_weights4(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "w_qkvg", "w_o", "w_gate", "w_up", "w_down", "sf_qkvg", "sf_o", "sf_gate", "sf_up", "sf_down", "ts_qkvg",
        "ts_o", "ts_gate", "ts_up", "ts_down")]


class krea_dit_weights8(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "w_qkvg", "w_o", "w_gate", "w_up", "w_down", "dq_qkvg", "dq_o", "dq_gate", "dq_up", "dq_down")]


class krea_dit_grads(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "d_x_txt", "d_x_img", "d_w_qkvg", "d_w_o", "d_w_gate", "d_w_up", "d_w_down", "d_norm1_w", "d_norm2_w",
        "d_q_norm_w", "d_k_norm_w", "d_mod_bias", "d_mod_shared")]


class krea_dit_temb_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("w1", "b1", "w2", "b2")]


_lib: Optional[ctypes.CDLL] = None


def lib() -> ctypes.CDLL:
    """Load libkrea_dit.so (built in-tree by ``__graft_entry__.build()``); raise if absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build the CUDA library first (__graft_entry__.build())")
        L = ctypes.CDLL(LIB_PATH)
        vp, ci, cf = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        L.krea_dit_block_create.argtypes = [ctypes.POINTER(krea_dit_config), ctypes.POINTER(vp)]
        L.krea_dit_block_destroy.argtypes = [vp]
        L.krea_dit_timestep_embed.argtypes = [vp, vp, ci, ctypes.POINTER(krea_dit_temb_weights), vp, vp]
        L.krea_dit_block_forward.argtypes = [vp, vp, vp, ci, ci, ci, ci, vp, ctypes.POINTER(krea_dit_weights), vp, vp]
        L.krea_dit_status_string.argtypes = [ci]
        L.krea_dit_status_string.restype = ctypes.c_char_p
        L.krea_dit_block_workspace.argtypes = [vp, ci, ctypes.POINTER(vp), ctypes.POINTER(ctypes.c_size_t)]
        L.krea_dit_block_set_timing.argtypes = [vp, ci]
        L.krea_dit_block_timing_reset.argtypes = [vp]
        L.krea_dit_block_kernel_times.argtypes = [vp, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_double),
                                                  ctypes.POINTER(ci), ci, ctypes.POINTER(ci)]
        L.krea_dit_block_device_status.argtypes = [vp, vp, ctypes.POINTER(ci)]
        L.krea_dit_block_inject_fault.argtypes = [vp, ci]
        L.krea_dit_block_selftest_wait.argtypes = [vp, ci, ctypes.c_longlong, vp]
        L.krea_dit_kernel_names.argtypes = [ctypes.POINTER(ctypes.c_char_p), ci]
        L.krea_dit_timestep_embed_noalloc.argtypes = [vp, ci, ci, ctypes.POINTER(krea_dit_temb_weights), vp, vp]
        L.krea_dit_block_enable_host_io.argtypes = [vp]
        L.krea_dit_block_forward_host.argtypes = L.krea_dit_block_forward.argtypes
        L.krea_dit_block_host_sync.argtypes = [vp]
        L.krea_dit_block_forward_joint.argtypes = [vp, vp, ci, ci, ci, ci, vp, ctypes.POINTER(krea_dit_weights), vp, vp]
        L.krea_dit_stack_forward.argtypes = [vp, vp, ci, ci, ci, ci, vp, ctypes.POINTER(krea_dit_weights), ci, vp]
        L.krea_dit_stack_graph_create.argtypes = [vp, vp, ci, ci, ci, ci, vp, ctypes.POINTER(krea_dit_weights), ci, vp,
                                                  ctypes.POINTER(vp)]
        L.krea_dit_graph_launch.argtypes = [vp, vp]
        L.krea_dit_graph_destroy.argtypes = [vp]
        L.krea_dit_weights8_quantize.argtypes = [vp, ctypes.POINTER(krea_dit_weights), ctypes.POINTER(krea_dit_weights8),
                                                 vp]
        L.krea_dit_nvfp4_scale_bytes.argtypes = [ci, ci]
        L.krea_dit_nvfp4_scale_bytes.restype = ctypes.c_size_t
        L.krea_dit_weights4_quantize.argtypes = [vp, ctypes.POINTER(krea_dit_weights), ctypes.POINTER(krea_dit_weights4),
                                                 vp]
        L.krea_dit_block_forward4.argtypes = [vp, vp, vp, ci, ci, ci, ci, vp, ctypes.POINTER(krea_dit_weights),
                                              ctypes.POINTER(krea_dit_weights4), vp, vp]
        L.krea_dit_block_enable_backward.argtypes = [vp]
        L.krea_dit_block_backward.argtypes = [vp, vp, vp, ci, ci, ci, ci, vp, ctypes.POINTER(krea_dit_weights), vp,
                                              ctypes.POINTER(krea_dit_grads), vp]
        L.krea_dit_block_forward8.argtypes = [vp, vp, vp, ci, ci, ci, ci, vp, ctypes.POINTER(krea_dit_weights),
                                              ctypes.POINTER(krea_dit_weights8), vp, vp]
        for name in EXPORTS:
            getattr(L, name)  # every declared symbol must resolve
            if name != "krea_dit_status_string":
                getattr(L, name).restype = ci
        _lib = L
    return _lib


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s) -> Optional[int]:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream  # torch.cuda.Stream


def _check(status: int, where: str) -> None:
    if status != KREA_DIT_OK:
        raise KreaDitError(status, where)


def krea_dit_status_string(status: int) -> str:
    return lib().krea_dit_status_string(status).decode()


def krea_dit_block_create(cfg: krea_dit_config) -> int:
    h = ctypes.c_void_p()
    _check(lib().krea_dit_block_create(ctypes.byref(cfg), ctypes.byref(h)), "krea_dit_block_create")
    return h.value


def krea_dit_block_destroy(handle: int) -> None:
    _check(lib().krea_dit_block_destroy(handle), "krea_dit_block_destroy")


def krea_dit_timestep_embed(handle: int, t, B: int, w: krea_dit_temb_weights, mod_shared, stream=None) -> None:
    _check(lib().krea_dit_timestep_embed(handle, _ptr(t), B, ctypes.byref(w), _ptr(mod_shared), _stream(stream)),
           "krea_dit_timestep_embed")


def krea_dit_timestep_embed_noalloc(t, B: int, d_model: int, w: krea_dit_temb_weights, mod_shared,
                                    stream=None) -> None:
    """Handle-free timestep embedding with fixed library-owned scratch (see the header)."""
    _check(lib().krea_dit_timestep_embed_noalloc(_ptr(t), B, d_model, ctypes.byref(w), _ptr(mod_shared),
                                                 _stream(stream)), "krea_dit_timestep_embed_noalloc")


def krea_dit_block_forward(handle: int, x_img, x_txt, B: int, img_h: int, img_w: int, n_txt: int, t_emb,
                           w: krea_dit_weights, out, stream=None) -> None:
    _check(lib().krea_dit_block_forward(handle, _ptr(x_img), _ptr(x_txt), B, img_h, img_w, n_txt, _ptr(t_emb),
                                        ctypes.byref(w), _ptr(out), _stream(stream)), "krea_dit_block_forward")


def krea_dit_weights8_quantize(handle: int, w: krea_dit_weights, q: krea_dit_weights8, stream=None) -> None:
    _check(lib().krea_dit_weights8_quantize(handle, ctypes.byref(w), ctypes.byref(q), _stream(stream)),
           "krea_dit_weights8_quantize")


def krea_dit_nvfp4_scale_bytes(rows: int, cols: int) -> int:
    return int(lib().krea_dit_nvfp4_scale_bytes(rows, cols))


def krea_dit_weights4_quantize(handle: int, w: krea_dit_weights, q: krea_dit_weights4, stream=None) -> None:
    _check(lib().krea_dit_weights4_quantize(handle, ctypes.byref(w), ctypes.byref(q), _stream(stream)),
           "krea_dit_weights4_quantize")


def krea_dit_block_forward4(handle: int, x_img, x_txt, B: int, img_h: int, img_w: int, n_txt: int, t_emb,
                            w: krea_dit_weights, q: krea_dit_weights4, out, stream=None) -> None:
    _check(lib().krea_dit_block_forward4(handle, _ptr(x_img), _ptr(x_txt), B, img_h, img_w, n_txt, _ptr(t_emb),
                                         ctypes.byref(w), ctypes.byref(q), _ptr(out), _stream(stream)),
           "krea_dit_block_forward4")


def krea_dit_block_forward8(handle: int, x_img, x_txt, B: int, img_h: int, img_w: int, n_txt: int, t_emb,
                            w: krea_dit_weights, q: krea_dit_weights8, out, stream=None) -> None:
    _check(lib().krea_dit_block_forward8(handle, _ptr(x_img), _ptr(x_txt), B, img_h, img_w, n_txt, _ptr(t_emb),
                                         ctypes.byref(w), ctypes.byref(q), _ptr(out), _stream(stream)),
           "krea_dit_block_forward8")


def krea_dit_block_enable_backward(handle: int) -> None:
    _check(lib().krea_dit_block_enable_backward(handle), "krea_dit_block_enable_backward")


def krea_dit_block_backward(handle: int, x_img, x_txt, B: int, img_h: int, img_w: int, n_txt: int, t_emb,
                            w: krea_dit_weights, d_out, g: krea_dit_grads, stream=None) -> None:
    _check(lib().krea_dit_block_backward(handle, _ptr(x_img), _ptr(x_txt), B, img_h, img_w, n_txt, _ptr(t_emb),
                                         ctypes.byref(w), _ptr(d_out), ctypes.byref(g), _stream(stream)),
           "krea_dit_block_backward")


def make_grads(t: Dict[str, object]) -> krea_dit_grads:
    """Gradient struct from a dict of device tensors keyed by the struct's field names
    (a missing key is passed as NULL)."""
    return krea_dit_grads(*[_ptr(t.get(n)) for n, _ in krea_dit_grads._fields_])


def krea_dit_block_enable_host_io(handle: int) -> None:
    _check(lib().krea_dit_block_enable_host_io(handle), "krea_dit_block_enable_host_io")


def krea_dit_block_forward_host(handle: int, x_img, x_txt, B: int, img_h: int, img_w: int, n_txt: int, t_emb,
                                w: krea_dit_weights, out, stream=None) -> None:
    """x_img, x_txt and out are host (ideally pinned) tensors or addresses."""
    _check(lib().krea_dit_block_forward_host(handle, _ptr(x_img), _ptr(x_txt), B, img_h, img_w, n_txt, _ptr(t_emb),
                                             ctypes.byref(w), _ptr(out), _stream(stream)),
           "krea_dit_block_forward_host")


def krea_dit_block_host_sync(handle: int) -> None:
    _check(lib().krea_dit_block_host_sync(handle), "krea_dit_block_host_sync")


def krea_dit_block_forward_joint(handle: int, x, B: int, img_h: int, img_w: int, n_txt: int, t_emb,
                                 w: krea_dit_weights, out, stream=None) -> None:
    _check(lib().krea_dit_block_forward_joint(handle, _ptr(x), B, img_h, img_w, n_txt, _ptr(t_emb), ctypes.byref(w),
                                              _ptr(out), _stream(stream)), "krea_dit_block_forward_joint")


def _weights_array(ws: List[krea_dit_weights]):
    arr = (krea_dit_weights * len(ws))(*ws)
    return arr


def krea_dit_stack_forward(handle: int, x, B: int, img_h: int, img_w: int, n_txt: int, t_emb,
                           ws: List[krea_dit_weights], stream=None) -> None:
    arr = _weights_array(ws)
    _check(lib().krea_dit_stack_forward(handle, _ptr(x), B, img_h, img_w, n_txt, _ptr(t_emb), arr, len(ws),
                                        _stream(stream)), "krea_dit_stack_forward")


def krea_dit_stack_graph_create(handle: int, x, B: int, img_h: int, img_w: int, n_txt: int, t_emb,
                                ws: List[krea_dit_weights], stream) -> int:
    arr = _weights_array(ws)
    g = ctypes.c_void_p()
    _check(lib().krea_dit_stack_graph_create(handle, _ptr(x), B, img_h, img_w, n_txt, _ptr(t_emb), arr, len(ws),
                                             _stream(stream), ctypes.byref(g)), "krea_dit_stack_graph_create")
    return g.value


def krea_dit_graph_launch(graph: int, stream=None) -> None:
    _check(lib().krea_dit_graph_launch(graph, _stream(stream)), "krea_dit_graph_launch")


def krea_dit_graph_destroy(graph: int) -> None:
    _check(lib().krea_dit_graph_destroy(graph), "krea_dit_graph_destroy")


def krea_dit_block_workspace(handle: int, which: str) -> Tuple[int, int]:
    p, n = ctypes.c_void_p(), ctypes.c_size_t()
    _check(lib().krea_dit_block_workspace(handle, BUFFERS[which], ctypes.byref(p), ctypes.byref(n)),
           "krea_dit_block_workspace")
    return p.value or 0, n.value


def krea_dit_block_set_timing(handle: int, enable: bool) -> None:
    _check(lib().krea_dit_block_set_timing(handle, int(bool(enable))), "krea_dit_block_set_timing")


def krea_dit_block_timing_reset(handle: int) -> None:
    _check(lib().krea_dit_block_timing_reset(handle), "krea_dit_block_timing_reset")


def krea_dit_block_kernel_times(handle: int) -> Dict[str, Tuple[float, int]]:
    cap = 64
    names = (ctypes.c_char_p * cap)()
    ms = (ctypes.c_double * cap)()
    cnt = (ctypes.c_int * cap)()
    n = ctypes.c_int()
    _check(lib().krea_dit_block_kernel_times(handle, names, ms, cnt, cap, ctypes.byref(n)),
           "krea_dit_block_kernel_times")
    return {names[i].decode(): (ms[i], cnt[i]) for i in range(n.value) if cnt[i] > 0}


def krea_dit_block_device_status(handle: int, stream=None) -> Tuple[int, int]:
    site = ctypes.c_int()
    st = lib().krea_dit_block_device_status(handle, _stream(stream), ctypes.byref(site))
    return st, site.value


def krea_dit_block_selftest_wait(handle: int, site: int, limit_ns: int, stream=None) -> None:
    _check(lib().krea_dit_block_selftest_wait(handle, site, limit_ns, _stream(stream)), "krea_dit_block_selftest_wait")


def krea_dit_block_inject_fault(handle: int, count: int) -> None:
    _check(lib().krea_dit_block_inject_fault(handle, count), "krea_dit_block_inject_fault")


def krea_dit_kernel_names() -> List[str]:
    cap = 64
    names = (ctypes.c_char_p * cap)()
    n = lib().krea_dit_kernel_names(names, cap)
    return [names[i].decode() for i in range(min(n, cap))]


def make_config(*, max_batch: int, max_seq: int, d_model: int, n_q: int, n_kv: int, head_dim: int, ffn: int,
                img_h_max: int, img_w_max: int, eps: float = 1e-6, rope_base: float = 10000.0, gate_on: bool = True,
                mode: int = KREA_DIT_BF16) -> krea_dit_config:
    return krea_dit_config(max_batch, max_seq, d_model, n_q, n_kv, head_dim, ffn, img_h_max, img_w_max, eps,
                           rope_base, int(bool(gate_on)), mode)


def make_weights(t: Dict[str, object]) -> krea_dit_weights:
    """Weights struct from a dict of device tensors keyed by the struct's field names
    (a missing key is passed as NULL)."""
    return krea_dit_weights(*[_ptr(t.get(n)) for n, _ in krea_dit_weights._fields_])


def make_weights8(t: Dict[str, object]) -> krea_dit_weights8:
    """8-bit weights struct from a dict of device tensors keyed by the struct's field names."""
    return krea_dit_weights8(*[_ptr(t[n]) for n, _ in krea_dit_weights8._fields_])


def make_weights4(t: Dict[str, object]) -> krea_dit_weights4:
    """NVFP4 weights struct from a dict of device tensors keyed by the struct's field names."""
    return krea_dit_weights4(*[_ptr(t[n]) for n, _ in krea_dit_weights4._fields_])


def make_temb_weights(t: Dict[str, object]) -> krea_dit_temb_weights:
    return krea_dit_temb_weights(*[_ptr(t[n]) for n, _ in krea_dit_temb_weights._fields_])
