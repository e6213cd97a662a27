"""fp64 CPU oracle of the block forward with 8-bit GEMM operands.

TEST INFRASTRUCTURE ONLY (same rules as the rest of this package: the library never
imports it, and it shares no code with the CUDA path).

The Krea 2 Technical Report ("训练 › 预训练" / Training › Pretraining) trains the 256px
stage with 8-bit matrix multiplications under tensor-wise scaling and the 512px stage
under finer row-wise scaling; 1024px and later are bf16. The report names neither the
8-bit format nor the scale rule. Readings taken:

* format: e4m3 (4 exponent bits, bias 7, 3 mantissa bits, no infinities, largest
  finite value 448), round to nearest, ties to even, saturating at +-448;
* scale: a power of two 2^k per scaling group, k the largest integer with
  amax * 2^k <= 448 (amax = largest magnitude in the group; amax = 0 gives k = 0), so
  that scaling is exact and the cast to e4m3 is the only rounding; the dequantised
  value is q * 2^-k;
* groups: tensor-wise = one group per operand tensor (an activation over all B*L
  rows of the step; a weight matrix as a whole, the fused [Q;K;V;G] projection being
  one matrix); row-wise = one group per row along the reduction axis (a token's row
  of the activation, an output channel's row of the weight), so that the product of
  the two scales factors out of every dot product;
* what is quantised: the four GEMMs of the block (the fused QKV+gate projection, the
  attention output projection, the SwiGLU gate/up projections and the down
  projection) take both operands through the cast; everything else is as in the bf16
  block. An activation is cast from the value the bf16 block stores at that point.
"""
from __future__ import annotations

from typing import Dict, Optional, Sequence

import numpy as np

from .block import (
    F64,
    apply_rope_2d,
    gqa_attention,
    modulation,
    rope_angles,
    sigmoid,
    silu,
    storage_rounding,
    token_positions,
    zero_centred_rms_norm,
)

E4M3_MAX = 448.0
E4M3_MIN_EXP = -6  # exponent of the smallest normal value, 2^-6
E4M3_MANT = 3  # stored mantissa bits
K_MAX = 125  # cap on the scale exponent (keeps 2^k and 2^-k normal in fp32)


def round_to_e4m3(v) -> np.ndarray:
    """Nearest e4m3 value of each float64 input, ties to even, magnitudes above 448
    saturating to 448. In the binade [2^e, 2^(e+1)), e >= -6, the spacing is 2^(e-3);
    below 2^-6 (the subnormals) it is 2^-9."""
    v = np.asarray(v, F64)
    a = np.abs(v)
    _, e = np.frexp(a)  # a = m 2^e, 0.5 <= m < 1, so the binade exponent is e - 1
    exp = np.maximum(e - 1, E4M3_MIN_EXP)
    step = np.ldexp(1.0, exp - E4M3_MANT)
    r = np.rint(a / step) * step  # a / step is exact; rint ties to even
    return np.copysign(np.minimum(r, E4M3_MAX), v)


def scale_exponent(amax) -> np.ndarray:
    """Largest integer k with amax * 2^k <= 448 (0 where amax is 0), capped at 125.
    With amax = m 2^e, 0.5 <= m < 1: k = 9 - e when m <= 448/512 = 0.875, else 8 - e."""
    amax = np.asarray(amax, F64)
    m, e = np.frexp(amax)
    k = np.where(m <= 0.875, 9 - e, 8 - e)
    k = np.where(amax > 0, k, 0)
    return np.minimum(k, K_MAX).astype(np.int64)


def quantize(x, per_row: bool):
    """Scaled e4m3 cast of x [R, K]: returns (q, d) with q the e4m3 values [R, K] and d
    the dequantisation factors 2^-k ([R, 1] row-wise, a scalar array tensor-wise), so
    that x is approximated by q * d."""
    x = np.asarray(x, F64)
    a = np.abs(x)
    amax = a.max(axis=-1, keepdims=True) if per_row else a.max(initial=0.0)
    k = scale_exponent(amax)
    q = round_to_e4m3(np.ldexp(x, k))
    return q, np.ldexp(1.0, -k)


def dequantized(x, per_row: bool) -> np.ndarray:
    q, d = quantize(x, per_row)
    return q * d


def block_forward8(
    x_txt: np.ndarray,
    x_img: np.ndarray,
    img_hw: Sequence[int],
    mod_shared: np.ndarray,
    w: Dict[str, np.ndarray],
    *,
    scaling: str,
    n_q: int,
    n_kv: int,
    hd: int,
    eps: float = 1e-6,
    rope_base: float = 10000.0,
    gate_on: bool = True,
    store=None,
    deq=None,
) -> Dict[str, list]:
    """The block forward of ``block.block_forward`` with 8-bit GEMM operands.

    ``scaling`` is "tensor" or "row". Tensor-wise groups span every row of the step,
    so the block runs stage by stage over all batch elements (all rows; no row
    sampling). ``store`` rounds intermediates where an implementation stores them,
    as in ``block_forward``; an activation is cast to e4m3 from its stored value.
    Returns per-batch lists xn, q, k, v, g, o_g, h1, hn, hmid, out over all rows, plus
    the dequantised GEMM operands xn8, og8, hn8, hmid8 ([L, K] per batch element).

    ``deq`` (optional) replaces the cast: a function from a [R, K] operand (an
    activation over all rows of the step, or a weight matrix) to its dequantised values;
    ``scaling`` is then ignored. The NVFP4 oracle (``oracle.nvfp4``) uses it."""
    if deq is None and scaling not in ("tensor", "row"):
        raise ValueError(f"scaling must be 'tensor' or 'row', not {scaling!r}")
    per_row = scaling == "row"
    if deq is None:
        def deq(x):
            return dequantized(x, per_row)
    x_txt = np.asarray(x_txt, F64)
    x_img = np.asarray(x_img, F64)
    B, Nt, d = x_txt.shape
    H, W_ = int(img_hw[0]), int(img_hw[1])
    L = Nt + H * W_
    mod = modulation(mod_shared, w["mod_bias"])
    names = ("xn", "q", "k", "v", "g", "o_g", "h1", "hn", "hmid", "out")
    smap = store if isinstance(store, dict) else {n: store for n in names}
    rnd = {n: storage_rounding(smap.get(n)) for n in names}
    ang = rope_angles(token_positions(Nt, H, W_), hd, rope_base)

    def rows_of(per_b):  # per-batch [L, K] list -> [B*L, K]
        return np.concatenate(per_b, axis=0)

    def split(m):  # [B*L, K] -> per-batch list
        return [m[b * L:(b + 1) * L] for b in range(B)]

    def mat8(name):
        return deq(w[name])

    X = [np.concatenate([x_txt[b], x_img[b]], axis=0) for b in range(B)]

    # norm1 + modulation, stored, then cast for the fused projection
    xn = [rnd["xn"](zero_centred_rms_norm(X[b], w["norm1_w"], eps) * (1.0 + mod["scale_a"][b])
                    + mod["shift_a"][b]) for b in range(B)]
    xn8 = split(deq(rows_of(xn)))
    proj = split(rows_of(xn8) @ mat8("w_qkvg").T)

    qr, kr = n_q * hd, n_kv * hd
    res = {n: [] for n in ("q", "k", "v", "g", "o_g", "xn8", "og8")}
    for b in range(B):
        p = proj[b]

        def heads(m, n):
            return m.reshape(L, n, hd).transpose(1, 0, 2)

        q = zero_centred_rms_norm(heads(p[:, :qr], n_q), w["q_norm_w"], eps)
        k = zero_centred_rms_norm(heads(p[:, qr:qr + kr], n_kv), w["k_norm_w"], eps)
        v = rnd["v"](heads(p[:, qr + kr:qr + 2 * kr], n_kv))
        q, k = rnd["q"](apply_rope_2d(q, ang)), rnd["k"](apply_rope_2d(k, ang))
        o = gqa_attention(q, k, v).transpose(1, 0, 2).reshape(L, qr)
        if gate_on:
            g = rnd["g"](sigmoid(p[:, qr + 2 * kr:2 * qr + 2 * kr]))  # the gate value, as stored
            o_g = o * g
        else:
            g = np.zeros_like(o)
            o_g = o
        res["q"].append(q)
        res["k"].append(k)
        res["v"].append(v)
        res["g"].append(g)
        res["o_g"].append(rnd["o_g"](o_g))
        res["xn8"].append(xn8[b])

    # attention output projection + gated residual
    og8 = split(deq(rows_of(res["o_g"])))
    attn = split(rows_of(og8) @ mat8("w_o").T)
    h1 = [rnd["h1"](X[b] + mod["gate_a"][b] * attn[b]) for b in range(B)]
    hn = [rnd["hn"](zero_centred_rms_norm(h1[b], w["norm2_w"], eps) * (1.0 + mod["scale_m"][b])
                    + mod["shift_m"][b]) for b in range(B)]
    hn8 = split(deq(rows_of(hn)))
    hn_all = rows_of(hn8)
    hmid = split(silu(hn_all @ mat8("w_gate").T) * (hn_all @ mat8("w_up").T))
    hmid = [rnd["hmid"](m) for m in hmid]
    hmid8 = split(deq(rows_of(hmid)))
    down = split(rows_of(hmid8) @ mat8("w_down").T)
    out = [rnd["out"](h1[b] + mod["gate_m"][b] * down[b]) for b in range(B)]

    res["og8"] = og8
    res.update(xn=xn, h1=h1, hn=hn, hmid=hmid, out=out, hn8=hn8, hmid8=hmid8, rows=[np.arange(L)] * B)
    return res


def run_case8(case, scaling: str, *, mod_shared: Optional[np.ndarray] = None, store=None) -> Dict[str, list]:
    """Timestep embedding plus the 8-bit block forward for a seeded case."""
    from . import mod_shared_for

    cfg = case.cfg
    ms = mod_shared_for(case) if mod_shared is None else mod_shared
    return block_forward8(
        case.x_txt, case.x_img, (cfg.img_h, cfg.img_w), ms, case.w, scaling=scaling,
        n_q=cfg.n_q, n_kv=cfg.n_kv, hd=cfg.hd, eps=cfg.eps, rope_base=cfg.rope_base,
        gate_on=cfg.gate_on, store=store,
    )
