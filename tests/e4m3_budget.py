"""A-priori allowances for the 8-bit and NVFP4 GEMM parity checks (host logic, no GPU).

An 8-bit GEMM casts an activation operand from a stored bf16 value v with one
power-of-two scale 2^k per group (a token row, or the whole tensor), k fixed by the
group's largest magnitude. The cast is discontinuous: a device value v' that differs
from the oracle's v by a little can land on another e4m3 code, and near a scale
boundary the whole group can change scale. These functions bound that change from the
oracle's values and a stated deviation budget alone (no device value enters a bound);
the GPU tests then assert that the device's operands and every downstream result stay
inside those bounds.
"""
from __future__ import annotations

import numpy as np

from oracle import gemm8 as g8

F64 = np.float64
Z = 6.0  # standard deviations of a sum of sign-symmetric terms covered by ``carry``


def bf16_ulp(v) -> np.ndarray:
    """Spacing of bf16 values at |v|: 2^(e-7) for |v| in [2^e, 2^(e+1)); 2^-133 (the
    smallest subnormal step) at 0."""
    a = np.abs(np.asarray(v, F64))
    _, e = np.frexp(a)  # a = m 2^e, 0.5 <= m < 1: binade exponent e - 1
    return np.where(a > 0, np.ldexp(1.0, e - 8), np.ldexp(1.0, -133))


def cast_change_bound(v, delta, per_row: bool):
    """The oracle's dequantised operand cast(v) and a bound on how far the cast of any
    v' with |v' - v| <= delta (elementwise) can land from it.

    The group's largest magnitude of v' lies in [lo, hi] = [max(|v| - delta),
    max(|v| + delta)], so its scale exponent is any k between k(hi) and k(lo) (k falls
    as the magnitude grows). For each such k the cast is monotone in v', so the largest
    distance over the interval [v - delta, v + delta] is reached at one of its ends.
    Returns (cast(v) as q * 2^-k, bound), both shaped like v; the bound is 0 where no
    admissible v' changes the cast."""
    v = np.asarray(v, F64)
    delta = np.broadcast_to(np.asarray(delta, F64), v.shape)
    q, d = g8.quantize(v, per_row)
    ref = q * d
    a = np.abs(v)
    if per_row:
        lo = np.max(np.maximum(a - delta, 0.0), axis=-1, keepdims=True)
        hi = np.max(a + delta, axis=-1, keepdims=True)
    else:
        lo = np.max(np.maximum(a - delta, 0.0), initial=0.0)
        hi = np.max(a + delta, initial=0.0)
    if v.size and np.any(lo <= 0):
        raise ValueError("a scaling group could be all zeros within its budget")
    k_lo, k_hi = g8.scale_exponent(hi), g8.scale_exponent(lo)
    bound = np.zeros_like(v)
    for k in range(int(np.min(k_lo)) if v.size else 0, (int(np.max(k_hi)) + 1) if v.size else 0):
        live = (k >= k_lo) & (k <= k_hi)
        if not np.any(live):
            continue
        for s in (v - delta, v + delta):
            dev = np.abs(np.ldexp(g8.round_to_e4m3(np.ldexp(s, k)), -k) - ref)
            bound = np.where(live, np.maximum(bound, dev), bound)
    return ref, bound


def carry(d_op, W) -> np.ndarray:
    """Spread that operand changes of at most d_op [R, K] carry through a projection
    with weights W [N, K]: Z * sqrt(d_op^2 (W^2)^T). The weights are sign-symmetric, so
    the carried terms d_j W_cj have independent random signs; for a single changed
    value the bound is Z times that value's whole effect."""
    return Z * np.sqrt((np.asarray(d_op, F64) ** 2) @ (np.asarray(W, F64) ** 2).T)


def norm_carry(h, gamma, dh, eps: float) -> np.ndarray:
    """Bound on the change of gamma * h / sqrt(mean(h^2) + eps) (row-wise) when h moves
    by at most dh elementwise: to first order
    |gamma_j| rstd (dh_j + |h_j| rstd ||dh||_2 / sqrt(d)), with 5% added for the
    second-order terms (dh is far below |h| here)."""
    h = np.asarray(h, F64)
    rstd = 1.0 / np.sqrt(np.mean(h * h, axis=-1, keepdims=True) + eps)
    nd = np.sqrt(np.sum(np.asarray(dh, F64) ** 2, axis=-1, keepdims=True) / h.shape[-1])
    return 1.05 * np.abs(gamma) * rstd * (dh + np.abs(h) * rstd * nd)


def attention_spread(q, k, v) -> np.ndarray:
    """sqrt(sum_k p_jk^2 v_kc^2) for every query row j and channel c of every head, with
    p the softmax probabilities of q k^T / sqrt(hd) (GQA: query head h reads key/value
    head h // (n_q / n_kv)). q [n_q, L, hd], k and v [n_kv, L, hd] -> [L, n_q * hd].

    When every probability carries an independent relative rounding error of at most
    r, the attention output's error has this spread times r (random signs); a device
    that rounds P to bf16 before the P V product has r = 2^-9."""
    q, k, v = (np.asarray(x, F64) for x in (q, k, v))
    n_q, L, hd = q.shape
    G = n_q // k.shape[0]
    out = np.empty((L, n_q * hd))
    for h in range(n_q):
        kv = h // G
        s = q[h] @ k[kv].T / np.sqrt(hd)
        s -= s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p /= p.sum(axis=1, keepdims=True)
        out[:, h * hd:(h + 1) * hd] = np.sqrt((p * p) @ (v[kv] ** 2))
    return out


# ------------------------------------------------------------------ NVFP4 casts
def _e4m3_grid() -> np.ndarray:
    """Every non-negative E4M3 value, ascending (0, the subnormals, the normals up to 448)."""
    vals = [m * 2.0 ** -9 for m in range(8)]
    vals += [(1 + m / 8.0) * 2.0 ** (e - 7) for e in range(1, 16) for m in range(8) if not (e == 15 and m == 7)]
    return np.array(sorted(set(vals)))


E4M3_GRID = _e4m3_grid()


def magnitude_range(v, delta):
    """(max(|v| - delta, 0), max(|v| + delta)) over the whole array: the range of the
    largest magnitude of any v' with |v' - v| <= delta."""
    v = np.asarray(v, F64)
    delta = np.broadcast_to(np.asarray(delta, F64), v.shape)
    lo_t = hi_t = 0.0
    flat_v, flat_d = v.reshape(-1), delta.reshape(-1)
    for i in range(0, flat_v.size, 1 << 20):
        a = np.abs(flat_v[i:i + (1 << 20)])
        dd = flat_d[i:i + (1 << 20)]
        lo_t = max(lo_t, float(np.max(np.maximum(a - dd, 0.0), initial=0.0)))
        hi_t = max(hi_t, float(np.max(a + dd, initial=0.0)))
    return lo_t, hi_t


def nvfp4_change_bound(v, delta, max_exact=2, tensor_range=None, s_t=None):
    """The oracle's NVFP4 cast of v [R, K] (``oracle.nvfp4``) and a bound on how far the cast
    of any v' with |v' - v| <= delta (elementwise) can land from it.

    The tensor's largest magnitude of v' lies in [max(|v| - delta), max(|v| + delta)], so
    its tensor scale is any power of two between the ends' scales; each block's largest
    magnitude lies in its own such interval, so for a given tensor scale its E4M3 block
    scale is any grid value between the ends' casts. For every such pair the element cast
    is monotone in v', so the ends of [v - delta, v + delta] give the largest distance.

    A block whose admissible block scales span more than ``max_exact`` + 1 grid values gets
    a closed-form bound instead of the enumeration (which would cost one pass over the
    whole tensor per grid value): for a scale product den in [den_lo, den_hi] the cast of s
    lies within den_hi of s while |s| <= 6 den (half the widest E2M1 spacing, 2, times den),
    within |s| - 6 den_lo of it beyond, and is 0 where den can be 0; s itself lies within
    |v - ref| + delta of the oracle's cast.

    For rows sampled from a larger tensor, ``s_t`` is the oracle's tensor scale of the
    whole tensor (the reference cast uses it) and ``tensor_range`` = (lo, hi) the range of
    the whole tensor's largest magnitude (``magnitude_range`` over all of its rows)."""
    from oracle import nvfp4 as f4

    v = np.asarray(v, F64)
    R, K = v.shape
    delta = np.broadcast_to(np.asarray(delta, F64), v.shape)
    if s_t is None:
        ref = f4.dequantized(v)
    else:
        q_, sb_, _ = f4.quantize(v, s_t=s_t)
        ref = q_ * np.repeat(sb_, 16, axis=-1) * s_t
    rows = max(1, (1 << 20) // max(K, 1))  # rows per pass (keeps numpy's temporaries in cache)
    lo_t, hi_t = magnitude_range(v, delta) if tensor_range is None else (float(t) for t in tensor_range)
    st_lo, st_hi = f4.tensor_scale(np.array([[lo_t]])), f4.tensor_scale(np.array([[hi_t]]))
    ts_cands = [st_lo]
    while ts_cands[-1] < st_hi:
        ts_cands.append(ts_cands[-1] * 2.0)
    nb = K // 16
    bound = np.zeros((R, K))
    for r0 in range(0, R, rows):  # rows are independent once the tensor scales are fixed
        vr, dr = v[r0:r0 + rows], delta[r0:r0 + rows]
        n = vr.shape[0]
        ab = np.abs(vr).reshape(n, nb, 16)
        db = dr.reshape(n, nb, 16)
        lo_b = np.max(np.maximum(ab - db, 0.0), axis=-1)
        hi_b = np.max(ab + db, axis=-1)
        ends = [(vr - dr).reshape(n, nb, 16), (vr + dr).reshape(n, nb, 16)]
        ref_b = ref[r0:r0 + rows].reshape(n, nb, 16)
        bd = np.zeros((n, nb, 16))
        wide = np.zeros((n, nb), dtype=bool)
        den_lo = np.full((n, nb), np.inf)
        den_hi = np.zeros((n, nb))
        for st in ts_cands:
            i_lo = np.searchsorted(E4M3_GRID, g8.round_to_e4m3(lo_b / (6.0 * st)))
            i_hi = np.searchsorted(E4M3_GRID, g8.round_to_e4m3(hi_b / (6.0 * st)))
            wide |= (i_hi - i_lo) > max_exact
            den_lo = np.minimum(den_lo, E4M3_GRID[i_lo] * st)
            den_hi = np.maximum(den_hi, E4M3_GRID[i_hi] * st)
            n_c = i_hi - i_lo
            for k in range(min(int(np.max(n_c, initial=0)), max_exact) + 1):
                sel = None if k == 0 else n_c >= k  # grid value k above the lowest, where admissible
                sb = E4M3_GRID[i_lo + k if sel is None else i_lo[sel] + k][..., None]
                den = sb * st
                for s in ends:
                    s_k = s if sel is None else s[sel]
                    q = np.where(den > 0, f4.round_to_e2m1(s_k / np.where(den > 0, den, 1.0)), 0.0) * den
                    if sel is None:
                        bd = np.maximum(bd, np.abs(q - ref_b))
                    else:
                        bd[sel] = np.maximum(bd[sel], np.abs(q - ref_b[sel]))
        if np.any(wide):
            sabs = ab[wide] + db[wide]  # largest |s| per element of the wide blocks
            dl, dh = den_lo[wide][:, None], den_hi[wide][:, None]
            cast_err = np.maximum(dh, sabs - 6.0 * dl)
            cast_err = np.where(dl > 0, cast_err, np.maximum(cast_err, sabs))
            bd[wide] = cast_err + np.abs(vr.reshape(n, nb, 16)[wide] - ref_b[wide]) + db[wide]
        bound[r0:r0 + rows] = bd.reshape(n, K)
    return ref, bound
