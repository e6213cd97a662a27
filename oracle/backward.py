"""fp64 CPU oracle of the block backward: analytic gradients of the single-stream block.

TEST INFRASTRUCTURE ONLY (same rules as the rest of this package: the library never
imports it, and it shares no code with the CUDA path).

The Krea 2 Technical Report trains the block ("训练" / Training); the training step
needs the gradients of the block forward of ``block.block_forward`` with respect to its
input, its weights and its modulation. They are written here by the chain rule, step
by step in the forward's own notation and in reverse order, with numpy matmuls as the
only library primitive. The forward values they need are recomputed first
(``forward_saved``), exactly as ``block.block_forward`` defines them.

Pinned in ``tests/test_oracle_backward.py`` against torch autograd through a textbook
block written with torch routines, and against central finite differences.
"""
from __future__ import annotations

import math
from typing import Dict, Optional

import numpy as np

from .block import (
    F64,
    apply_rope_2d,
    modulation,
    rope_angles,
    sigmoid,
    silu,
    storage_rounding,
    token_positions,
)

MOD_NAMES = ("shift_a", "scale_a", "gate_a", "shift_m", "scale_m", "gate_m")


def _rstd(x: np.ndarray, eps: float) -> np.ndarray:
    """1 / sqrt(mean(x^2) + eps) over the last axis, keeping it."""
    return 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)


def rms_backward(x: np.ndarray, r: np.ndarray, dy: np.ndarray) -> np.ndarray:
    """Gradient through y = x * r, r = (mean(x^2) + eps)^(-1/2) over the last axis (size D):
    dx = r dy - r^3 x mean(dy * x)."""
    return r * dy - (r ** 3) * x * np.mean(dy * x, axis=-1, keepdims=True)


def rope_backward(dy: np.ndarray, angles: np.ndarray) -> np.ndarray:
    """Gradient through apply_rope_2d: the transposed rotation, i.e. the rotation by the
    negative angle, (a, b) -> (a cos + b sin, -a sin + b cos)."""
    a = dy[..., 0::2]
    b = dy[..., 1::2]
    cos, sin = np.cos(angles), np.sin(angles)
    out = np.empty_like(dy)
    out[..., 0::2] = a * cos + b * sin
    out[..., 1::2] = -a * sin + b * cos
    return out


def silu_grad(a: np.ndarray) -> np.ndarray:
    """d silu(a) / da = sigma(a) (1 + a (1 - sigma(a)))."""
    s = sigmoid(a)
    return s * (1.0 + a * (1.0 - s))


def forward_saved(X: np.ndarray, mod: Dict[str, np.ndarray], w: Dict[str, np.ndarray], *, L_txt: int,
                  img_hw, n_q: int, n_kv: int, hd: int, eps: float, rope_base: float, gate_on: bool,
                  rnd=None) -> Dict[str, np.ndarray]:
    """The block forward for one batch element X [L, d] (text rows first) with every value
    the backward needs. ``mod`` holds this element's six modulation vectors [d]. ``rnd``
    (optional) maps an intermediate's name to the rounding applied where an
    implementation stores it, as ``block.block_forward``'s ``store``."""
    rnd = rnd or {}
    R = lambda n, v: rnd[n](v) if n in rnd else v  # noqa: E731
    L, d = X.shape
    G = n_q // n_kv
    H, W_ = int(img_hw[0]), int(img_hw[1])
    ang = rope_angles(token_positions(L_txt, H, W_), hd, rope_base)
    s = {"X": X, "ang": ang}
    s["r1"] = _rstd(X, eps)
    s["n1"] = X * s["r1"]
    s["xn"] = R("xn", s["n1"] * (1.0 + w["norm1_w"]) * (1.0 + mod["scale_a"]) + mod["shift_a"])
    P = s["xn"] @ np.asarray(w["w_qkvg"], F64).T
    qr, kr = n_q * hd, n_kv * hd
    heads = lambda m, n: m.reshape(L, n, hd).transpose(1, 0, 2)  # noqa: E731
    s["q_raw"] = heads(P[:, :qr], n_q)
    s["k_raw"] = heads(P[:, qr:qr + kr], n_kv)
    s["v"] = R("v", heads(P[:, qr + kr:qr + 2 * kr], n_kv))
    s["rq"] = _rstd(s["q_raw"], eps)
    s["rk"] = _rstd(s["k_raw"], eps)
    s["qn"] = s["q_raw"] * s["rq"] * (1.0 + w["q_norm_w"])
    s["kn"] = s["k_raw"] * s["rk"] * (1.0 + w["k_norm_w"])
    s["q"] = R("q", apply_rope_2d(s["qn"], ang))
    s["k"] = R("k", apply_rope_2d(s["kn"], ang))
    scale = 1.0 / math.sqrt(hd)
    A = np.empty((n_q, L, L))
    o = np.empty((n_q, L, hd))
    for h in range(n_q):
        S = s["q"][h] @ s["k"][h // G].T * scale
        S = S - S.max(axis=1, keepdims=True)
        E = np.exp(S)
        A[h] = E / E.sum(axis=1, keepdims=True)
        o[h] = A[h] @ s["v"][h // G]
    s["A"] = A
    s["o"] = o.transpose(1, 0, 2).reshape(L, qr)
    if gate_on:
        s["g"] = R("g", sigmoid(P[:, qr + 2 * kr:2 * qr + 2 * kr]))  # the gate value, as stored
        s["og"] = R("o_g", s["o"] * s["g"])
    else:
        s["og"] = R("o_g", s["o"])
    s["fa"] = s["og"] @ np.asarray(w["w_o"], F64).T
    s["h1"] = R("h1", X + mod["gate_a"] * s["fa"])
    s["r2"] = _rstd(s["h1"], eps)
    s["n2"] = s["h1"] * s["r2"]
    s["hn"] = R("hn", s["n2"] * (1.0 + w["norm2_w"]) * (1.0 + mod["scale_m"]) + mod["shift_m"])
    s["a"] = s["hn"] @ np.asarray(w["w_gate"], F64).T
    s["u"] = s["hn"] @ np.asarray(w["w_up"], F64).T
    s["hmid"] = R("hmid", silu(s["a"]) * s["u"])
    s["fm"] = s["hmid"] @ np.asarray(w["w_down"], F64).T
    s["out"] = R("out", s["h1"] + mod["gate_m"] * s["fm"])
    return s


def element_backward(s: Dict[str, np.ndarray], dout: np.ndarray, mod: Dict[str, np.ndarray],
                     w: Dict[str, np.ndarray], *, n_q: int, n_kv: int, hd: int, gate_on: bool):
    """Gradients of one batch element's forward (``forward_saved`` values ``s``) for the
    upstream gradient dout [L, d]. Returns (dX [L, d], weight gradients of this element,
    modulation gradients {name: [d]})."""
    L, d = dout.shape
    G = n_q // n_kv
    qr, kr = n_q * hd, n_kv * hd
    f64 = lambda a: np.asarray(a, F64)  # noqa: E731
    gw, gm = {}, {}
    # MLP residual: out = h1 + gate_m * fm,  fm = hmid W_down^T
    gm["gate_m"] = np.sum(dout * s["fm"], axis=0)
    d_fm = dout * mod["gate_m"]
    gw["w_down"] = d_fm.T @ s["hmid"]
    d_hmid = d_fm @ f64(w["w_down"])
    # SwiGLU: hmid = silu(a) * u
    d_a = d_hmid * s["u"] * silu_grad(s["a"])
    d_u = d_hmid * silu(s["a"])
    gw["w_gate"] = d_a.T @ s["hn"]
    gw["w_up"] = d_u.T @ s["hn"]
    d_hn = d_a @ f64(w["w_gate"]) + d_u @ f64(w["w_up"])
    # norm2 + modulation: hn = n2 (1 + w2)(1 + scale_m) + shift_m,  n2 = h1 * r2
    gm["shift_m"] = np.sum(d_hn, axis=0)
    gm["scale_m"] = np.sum(d_hn * s["n2"], axis=0) * (1.0 + w["norm2_w"])
    gw["norm2_w"] = np.sum(d_hn * s["n2"], axis=0) * (1.0 + mod["scale_m"])
    d_n2 = d_hn * (1.0 + w["norm2_w"]) * (1.0 + mod["scale_m"])
    d_h1 = dout + rms_backward(s["h1"], s["r2"], d_n2)
    # attention residual: h1 = X + gate_a * fa,  fa = og W_o^T
    gm["gate_a"] = np.sum(d_h1 * s["fa"], axis=0)
    d_fa = d_h1 * mod["gate_a"]
    gw["w_o"] = d_fa.T @ s["og"]
    d_og = d_fa @ f64(w["w_o"])
    # output gate: og = o * sg, sg = sigmoid(x W_g^T); d/dx sigmoid = sg (1 - sg)
    if gate_on:
        sg = s["g"]
        d_o = d_og * sg
        d_g = d_og * s["o"] * sg * (1.0 - sg)
    else:
        d_o = d_og
        d_g = None
    # attention, per query head h reading KV head h // G
    d_o = d_o.reshape(L, n_q, hd).transpose(1, 0, 2)
    scale = 1.0 / math.sqrt(hd)
    d_q = np.zeros_like(s["q"])
    d_k = np.zeros_like(s["k"])
    d_v = np.zeros_like(s["v"])
    for h in range(n_q):
        kv = h // G
        A = s["A"][h]
        d_v[kv] += A.T @ d_o[h]
        dA = d_o[h] @ s["v"][kv].T
        dS = A * (dA - np.sum(dA * A, axis=1, keepdims=True))
        d_q[h] = dS @ s["k"][kv] * scale
        d_k[kv] += dS.T @ s["q"][h] * scale
    # RoPE, then the per-head QK-RMSNorm with gain (1 + w)
    d_qn = rope_backward(d_q, s["ang"])
    d_kn = rope_backward(d_k, s["ang"])
    gw["q_norm_w"] = np.sum(d_qn * s["q_raw"] * s["rq"], axis=(0, 1))
    gw["k_norm_w"] = np.sum(d_kn * s["k_raw"] * s["rk"], axis=(0, 1))
    d_q_raw = rms_backward(s["q_raw"], s["rq"], d_qn * (1.0 + w["q_norm_w"]))
    d_k_raw = rms_backward(s["k_raw"], s["rk"], d_kn * (1.0 + w["k_norm_w"]))
    flat = lambda m: m.transpose(1, 0, 2).reshape(L, -1)  # noqa: E731
    parts = [flat(d_q_raw), flat(d_k_raw), flat(d_v)] + ([d_g] if gate_on else [])
    d_P = np.concatenate(parts, axis=1)
    gw["w_qkvg"] = d_P.T @ s["xn"]
    d_xn = d_P @ f64(w["w_qkvg"])
    # norm1 + modulation: xn = n1 (1 + w1)(1 + scale_a) + shift_a,  n1 = X * r1
    gm["shift_a"] = np.sum(d_xn, axis=0)
    gm["scale_a"] = np.sum(d_xn * s["n1"], axis=0) * (1.0 + w["norm1_w"])
    gw["norm1_w"] = np.sum(d_xn * s["n1"], axis=0) * (1.0 + mod["scale_a"])
    d_n1 = d_xn * (1.0 + w["norm1_w"]) * (1.0 + mod["scale_a"])
    d_X = d_h1 + rms_backward(s["X"], s["r1"], d_n1)
    return d_X, gw, gm


def block_backward(x_txt, x_img, img_hw, mod_shared, w, dout, *, n_q: int, n_kv: int, hd: int,
                   eps: float = 1e-6, rope_base: float = 10000.0, gate_on: bool = True, store=None):
    """Gradients of ``block.block_forward`` (all rows) for the upstream gradient dout
    [B, L, d] (joint order, text rows first).

    Returns a dict: d_x_txt [B, Nt, d], d_x_img [B, H*W, d], d_mod_shared [B, 6, d],
    d_mod_bias [6, d], and d_<weight> for w_qkvg, w_o, w_gate, w_up, w_down, norm1_w,
    norm2_w, q_norm_w, k_norm_w (summed over the batch). ``store`` rounds the forward's
    intermediates as ``block.block_forward`` does (the gradients stay float64)."""
    x_txt = np.asarray(x_txt, F64)
    x_img = np.asarray(x_img, F64)
    dout = np.asarray(dout, F64)
    B, Nt, d = x_txt.shape
    mod = modulation(mod_shared, w["mod_bias"])
    names = ("xn", "q", "k", "v", "g", "o_g", "h1", "hn", "hmid", "out")
    smap = store if isinstance(store, dict) else {n: store for n in names}
    rnd = {n: storage_rounding(smap.get(n)) for n in names}
    res = {"d_" + k: 0.0 for k in ("w_qkvg", "w_o", "w_gate", "w_up", "w_down", "norm1_w", "norm2_w",
                                   "q_norm_w", "k_norm_w")}
    d_txt, d_img, d_ms = [], [], []
    for b in range(B):
        X = np.concatenate([x_txt[b], x_img[b]], axis=0)
        mb = {k: mod[k][b] for k in MOD_NAMES}
        s = forward_saved(X, mb, w, L_txt=Nt, img_hw=img_hw, n_q=n_q, n_kv=n_kv, hd=hd, eps=eps,
                          rope_base=rope_base, gate_on=gate_on, rnd=rnd)
        dX, gw, gm = element_backward(s, dout[b], mb, w, n_q=n_q, n_kv=n_kv, hd=hd, gate_on=gate_on)
        d_txt.append(dX[:Nt])
        d_img.append(dX[Nt:])
        d_ms.append(np.stack([gm[k] for k in MOD_NAMES]))
        for k, v in gw.items():
            res["d_" + k] = res["d_" + k] + v
    res["d_x_txt"] = np.stack(d_txt)
    res["d_x_img"] = np.stack(d_img)
    res["d_mod_shared"] = np.stack(d_ms)
    res["d_mod_bias"] = res["d_mod_shared"].sum(axis=0)  # mod = mod_shared[b] + mod_bias
    return res


def run_case_backward(case, dout, *, mod_shared: Optional[np.ndarray] = None, store=None):
    """Gradients of the block forward for a seeded case and upstream gradient dout."""
    from . import mod_shared_for

    cfg = case.cfg
    ms = mod_shared_for(case) if mod_shared is None else mod_shared
    return block_backward(case.x_txt, case.x_img, (cfg.img_h, cfg.img_w), ms, case.w, dout, n_q=cfg.n_q,
                          n_kv=cfg.n_kv, hd=cfg.hd, eps=cfg.eps, rope_base=cfg.rope_base, gate_on=cfg.gate_on,
                          store=store)
