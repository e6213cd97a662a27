"""fp64 CPU oracle of the block forward with NVFP4 GEMM operands.

TEST INFRASTRUCTURE ONLY (same rules as the rest of this package: the library never
imports it, and it shares no code with the CUDA path).

The Krea 2 Technical Report ("讨论与未来工作" / Discussion and future work) names
pretraining at NVFP4 precision as a next step; it gives no recipe. NVFP4 is the 4-bit
format with two-level scaling; the readings taken here:

* element: FP4 E2M1 (1 sign, 2 exponent bits with bias 1, 1 mantissa bit; no infinities
  or NaN): magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6. Round to nearest, ties to the value
  with an even mantissa bit, magnitudes above 6 saturate to 6;
* block scale: one positive FP8 E4M3 value per 16 consecutive elements along the
  reduction axis (K) of a row;
* tensor scale: one value per operand tensor, the power of two s_t = 2^j with j the
  smallest integer such that amax <= 448 * 6 * 2^j (amax = the tensor's largest
  magnitude; s_t = 1 when amax = 0), so that every block scale fits E4M3's range. A
  power of two (rather than amax / 2688 itself) keeps every division by s_t exact, so
  that the casts below are decided the same way in fp32 as in fp64;
* a block with largest magnitude a_b gets s_b = E4M3(a_b / (6 s_t)) (round to nearest
  even, saturating at 448); its elements become q_i = E2M1(x_i / (s_b s_t)) (q_i = 0
  when s_b = 0) and are dequantised as q_i s_b s_t;
* what is quantised: the four GEMMs of the block take both operands through the cast,
  as the 8-bit oracle (``oracle.gemm8``) does, an activation over all rows of the call
  being one tensor and each weight matrix (the fused [Q;K;V;G] projection one matrix)
  another; everything else is as in the bf16 block.
"""
from __future__ import annotations

from typing import Dict, Optional

import numpy as np

from .block import F64
from .gemm8 import block_forward8, round_to_e4m3

E2M1_VALUES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])  # codes 0..7 (magnitude bits)
E2M1_MAX = 6.0
E4M3_MAX = 448.0
BLOCK = 16


_CHUNK = 1 << 20  # elements per numpy pass over a large tensor (keeps temporaries in cache)


def _round_to_e2m1_flat(v: np.ndarray) -> np.ndarray:
    a = np.minimum(np.abs(v), E2M1_MAX)
    step = np.where(a < 2.0, 0.5, np.where(a < 4.0, 1.0, 2.0))
    lo = np.floor(a / step) * step  # the grid value at or below a
    hi = lo + step
    d_lo, d_hi = a - lo, hi - a
    # a tie keeps the neighbour whose mantissa bit is 0: 0, 1, 2 and 4
    lo_even = (lo == 0.0) | (lo == 1.0) | (lo == 2.0) | (lo == 4.0)
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & ~lo_even)
    r = np.where(pick_hi, np.minimum(hi, E2M1_MAX), lo)
    return np.copysign(r, v)


def round_to_e2m1(v) -> np.ndarray:
    """Nearest E2M1 value of each float64 input; a tie goes to the neighbour whose
    mantissa bit is 0 (codes 0, 2, 4, 6: 0, 1, 2, 4); magnitudes above 6 saturate to 6.
    In [0, 2) the spacing is 0.5, in [2, 4) it is 1, in [4, 6] it is 2. Elementwise (large
    inputs go through in slices of _CHUNK elements)."""
    v = np.asarray(v, F64)
    if v.size <= _CHUNK:
        return _round_to_e2m1_flat(v)
    flat = v.reshape(-1)
    out = np.empty_like(flat)
    for i in range(0, flat.size, _CHUNK):
        out[i:i + _CHUNK] = _round_to_e2m1_flat(flat[i:i + _CHUNK])
    return out.reshape(v.shape)


def tensor_scale(x) -> float:
    """s_t = 2^j, j the smallest integer with amax <= 2688 * 2^j; 1 for an all-zero
    tensor. With amax / 2688 = m 2^e (0.5 <= m < 1): j = e - 1 when m = 0.5, else e."""
    x = np.asarray(x, F64)
    amax = max(float(np.max(x, initial=0.0)), -float(np.min(x, initial=0.0)))
    if amax <= 0:
        return 1.0
    m, e = np.frexp(amax / (E4M3_MAX * E2M1_MAX))
    return float(np.ldexp(1.0, int(e) - 1 if m == 0.5 else int(e)))


def quantize(x, s_t: Optional[float] = None):
    """NVFP4 cast of x [R, K] (K a multiple of 16): returns (q [R, K] the E2M1 values,
    s_b [R, K/16] the E4M3 block scales, s_t the tensor scale), so that x is approximated
    by q * repeat(s_b, 16) * s_t."""
    x = np.asarray(x, F64)
    R, K = x.shape
    if K % BLOCK:
        raise ValueError("K must be a multiple of 16")
    st = tensor_scale(x) if s_t is None else float(s_t)
    q = np.empty((R, K))
    s_b = np.empty((R, K // BLOCK))
    rows = max(1, _CHUNK // max(K, 1))
    for r0 in range(0, R, rows):  # rows are independent once s_t is fixed
        blocks = x[r0:r0 + rows].reshape(-1, K // BLOCK, BLOCK)
        amax_b = np.max(np.abs(blocks), axis=-1)
        sb = round_to_e4m3(amax_b / (E2M1_MAX * st))
        denom = sb[..., None] * st
        q[r0:r0 + rows] = np.where(denom > 0, round_to_e2m1(blocks / np.where(denom > 0, denom, 1.0)),
                                   0.0).reshape(-1, K)
        s_b[r0:r0 + rows] = sb
    return q, s_b, st


def dequantized(x) -> np.ndarray:
    q, s_b, st = quantize(x)
    return q * np.repeat(s_b, BLOCK, axis=-1) * st


def block_forward4(x_txt, x_img, img_hw, mod_shared, w, *, n_q, n_kv, hd, eps=1e-6, rope_base=10000.0,
                   gate_on=True, store=None) -> Dict[str, list]:
    """The block forward with NVFP4 operands in the four GEMMs (all rows; an activation's
    tensor scale spans every row of the call). Same outputs as ``gemm8.block_forward8``
    (the dequantised operands under the keys xn8, og8, hn8, hmid8)."""
    return block_forward8(x_txt, x_img, img_hw, mod_shared, w, scaling="tensor", n_q=n_q, n_kv=n_kv, hd=hd, eps=eps,
                          rope_base=rope_base, gate_on=gate_on, store=store, deq=dequantized)


def run_case4(case, *, mod_shared: Optional[np.ndarray] = None, store=None) -> Dict[str, list]:
    """Timestep embedding plus the NVFP4 block forward for a seeded case."""
    from . import mod_shared_for

    cfg = case.cfg
    ms = mod_shared_for(case) if mod_shared is None else mod_shared
    return block_forward4(case.x_txt, case.x_img, (cfg.img_h, cfg.img_w), ms, case.w, n_q=cfg.n_q, n_kv=cfg.n_kv,
                          hd=cfg.hd, eps=cfg.eps, rope_base=cfg.rope_base, gate_on=cfg.gate_on, store=store)
