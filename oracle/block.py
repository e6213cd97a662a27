"""fp64 CPU oracle of the Krea 2 single-stream DiT block forward.

TEST INFRASTRUCTURE ONLY. This module is the plain, slow, obviously correct
definition that the CUDA kernels are checked against. Only the tests, the smoke
check and the benchmark's CPU-baseline leg may import it; the library never
does, and it shares no code with the CUDA path.

Every function follows one passage of the Krea 2 Technical Report (the Chinese
translation titled "Krea 2 技术报告", section "架构" / Architecture, and its
reference list), restated here in the report's terms:

* Transformer block: SwiGLU MLP with a 4x expansion; GQA attention with a
  sigmoid output gate after "Gated Attention for LLMs" (ref. 47).
* Modality streams: a single-stream block, weights shared by text and image
  tokens over the joint sequence.
* Timestep conditioning: a shared sinusoidal timestep embedding feeding
  shift/scale/gate modulation, with a per-block tunable bias replacing the
  per-block modulation MLP.
* Positional encoding: axial RoPE; text tokens use RoPE index 0.
* Normalisation: zero-centred RMSNorm as pre-norm and as QK-norm.

Where the report leaves a step open the reading taken is stated at the step (and
listed, with the reason, in the design notes). All arithmetic is float64; matrix
products use numpy's matmul as a library primitive, with no blocking or fusion.
"""
from __future__ import annotations

import math
from typing import Dict, Optional, Sequence

import numpy as np

__all__ = [
    "timestep_embedding",
    "timestep_mlp",
    "modulation",
    "rms_norm",
    "zero_centred_rms_norm",
    "rope_angles",
    "apply_rope_2d",
    "token_positions",
    "gqa_attention",
    "swiglu",
    "block_forward",
    "round_to_bf16",
]

F64 = np.float64
TEMB_DIM = 256  # sinusoid width (DiT / FLUX convention; the report says only "sinusoidal")
TEMB_T_SCALE = 1000.0  # t in [0,1] is scaled to [0,1000] before the sinusoid
TEMB_MAX_PERIOD = 10000.0


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 value (8 significant bits), ties to
    even, directly from float64 (no intermediate float32 rounding)."""
    x = np.asarray(x, F64)
    m, e = np.frexp(x)  # x = m * 2^e, 0.5 <= |m| < 1
    return np.ldexp(np.rint(m * 256.0), e - 8)


def storage_rounding(store: Optional[str]):
    """Identity (exact oracle) or the rounding applied where the CUDA path stores an
    intermediate in its storage dtype ("bf16" or "fp32")."""
    if store is None:
        return lambda a: a
    if store == "bf16":
        return round_to_bf16
    if store == "fp32":
        return lambda a: np.asarray(a, F64).astype(np.float32).astype(F64)
    raise ValueError(store)


def sigmoid(x: np.ndarray) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-x))


def silu(x: np.ndarray) -> np.ndarray:
    return x * sigmoid(x)


# ---------------------------------------------------------------------------
# Timestep conditioning ("架构 › 时间步条件化" / Timestep conditioning)
# ---------------------------------------------------------------------------
def timestep_embedding(t: np.ndarray, dim: int = TEMB_DIM) -> np.ndarray:
    """Sinusoidal timestep embedding, [B] -> [B, dim].

    The report uses sinusoidal embeddings for the timestep. Reading taken (the
    DiT convention, Peebles & Xie, ref. 11): half = dim/2 frequencies
    w_i = 10000^(-i/half), argument 1000*t*w_i, laid out as [cos | sin].
    """
    t = np.asarray(t, dtype=F64)
    half = dim // 2
    i = np.arange(half, dtype=F64)
    freqs = TEMB_MAX_PERIOD ** (-i / half)
    arg = (TEMB_T_SCALE * t)[:, None] * freqs[None, :]
    return np.concatenate([np.cos(arg), np.sin(arg)], axis=1)


def timestep_mlp(e: np.ndarray, w1, b1, w2, b2) -> np.ndarray:
    """Shared timestep MLP: Linear(256->d) -> SiLU -> Linear(d->6d), returned as
    mod_shared [B, 6, d]. Shared by every block of the network (the report
    removes the per-block modulation MLP and keeps a shared embedding)."""
    hmid = silu(e @ np.asarray(w1, F64).T + np.asarray(b1, F64))
    m = hmid @ np.asarray(w2, F64).T + np.asarray(b2, F64)
    d = np.asarray(w1).shape[0]
    return m.reshape(e.shape[0], 6, d)


def modulation(mod_shared: np.ndarray, mod_bias: np.ndarray) -> Dict[str, np.ndarray]:
    """Per-block modulation = shared timestep modulation + this block's tunable
    bias. Chunk order (reading taken, the DiT adaLN order): shift, scale, gate
    for attention, then shift, scale, gate for the MLP. Each entry is [B, d]."""
    m = np.asarray(mod_shared, F64) + np.asarray(mod_bias, F64)[None]
    names = ("shift_a", "scale_a", "gate_a", "shift_m", "scale_m", "gate_m")
    return {n: m[:, i, :] for i, n in enumerate(names)}


# ---------------------------------------------------------------------------
# Normalisation ("架构 › 归一化" / Normalisation; RMSNorm ref. 51, Gemma ref. 79)
# ---------------------------------------------------------------------------
def rms_norm(v: np.ndarray, eps: float) -> np.ndarray:
    """v / sqrt(mean(v^2) + eps) over the last axis (Zhang & Sennrich)."""
    v = np.asarray(v, F64)
    return v / np.sqrt(np.mean(v * v, axis=-1, keepdims=True) + eps)


def zero_centred_rms_norm(v: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """Zero-centred RMSNorm: the learnable gain is stored as an offset w around
    zero and applied as (1 + w), so weight decay pulls the gain toward 1
    (reading taken: the Gemma convention the report cites). No mean is
    subtracted: that would be LayerNorm, the baseline the report replaced."""
    return rms_norm(v, eps) * (1.0 + np.asarray(w, F64))


# ---------------------------------------------------------------------------
# Positional encoding ("架构 › 位置编码" / Positional encoding; N-d RoPE ref. 49)
# ---------------------------------------------------------------------------
def token_positions(n_txt: int, img_h: int, img_w: int) -> np.ndarray:
    """(row, col) RoPE position of every token of the joint sequence, text first.
    Text tokens take index 0 on every axis; image token n = r*W + c (row-major)
    takes (r, c)."""
    L = n_txt + img_h * img_w
    pos = np.zeros((L, 2), dtype=np.int64)
    if img_h * img_w:
        r, c = np.meshgrid(np.arange(img_h), np.arange(img_w), indexing="ij")
        pos[n_txt:, 0] = r.reshape(-1)
        pos[n_txt:, 1] = c.reshape(-1)
    return pos


def rope_angles(pos: np.ndarray, hd: int, base: float) -> np.ndarray:
    """Rotation angle of every channel pair, [L, hd/2].

    Axial 2D RoPE (reading taken: a still image has frame index 0, so the frame
    axis of the report's 3D axial RoPE is the identity and is dropped). The head
    dimension is split in halves: [0, hd/2) rotates with the row position and
    [hd/2, hd) with the column position. Inside a half of size D = hd/2, the
    pair (2j, 2j+1), j < D/2, turns by pos * base^(-2j/D).
    """
    D = hd // 2
    j = np.arange(D // 2, dtype=F64)
    inv_freq = base ** (-2.0 * j / D)
    ang_r = pos[:, 0:1].astype(F64) * inv_freq[None, :]
    ang_c = pos[:, 1:2].astype(F64) * inv_freq[None, :]
    return np.concatenate([ang_r, ang_c], axis=1)


def apply_rope_2d(x: np.ndarray, angles: np.ndarray) -> np.ndarray:
    """Rotate consecutive channel pairs (2p, 2p+1) of x [..., L, hd] by angles
    [L, hd/2]: (a, b) -> (a cos - b sin, a sin + b cos)."""
    a = x[..., 0::2]
    b = x[..., 1::2]
    cos, sin = np.cos(angles), np.sin(angles)
    out = np.empty_like(x)
    out[..., 0::2] = a * cos - b * sin
    out[..., 1::2] = a * sin + b * cos
    return out


# ---------------------------------------------------------------------------
# Attention ("架构 › Transformer块": GQA ref. 45, gated attention ref. 47)
# ---------------------------------------------------------------------------
def gqa_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray) -> np.ndarray:
    """Bidirectional softmax attention with grouped K/V heads.

    q [n_q, Lq, hd], k and v [n_kv, L, hd]. Query head h reads K/V head
    floor(h / G), G = n_q / n_kv (reading taken: contiguous groups). No mask: the
    pass is pure prefill (the report notes diffusion needs no KV cache).
    Returns o [n_q, Lq, hd].
    """
    n_q, _, hd = q.shape
    n_kv = k.shape[0]
    G = n_q // n_kv
    o = np.empty_like(q)
    for h in range(n_q):
        kv = h // G
        s = q[h] @ k[kv].T / math.sqrt(hd)
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p /= p.sum(axis=1, keepdims=True)
        o[h] = p @ v[kv]
    return o


def swiglu(hn: np.ndarray, w_gate, w_up) -> np.ndarray:
    """SwiGLU hidden activation silu(hn W_gate^T) * (hn W_up^T) (Shazeer, ref. 44)."""
    return silu(hn @ np.asarray(w_gate, F64).T) * (hn @ np.asarray(w_up, F64).T)


# ---------------------------------------------------------------------------
# The block
# ---------------------------------------------------------------------------
def block_forward(
    x_txt: np.ndarray,
    x_img: np.ndarray,
    img_hw: Sequence[int],
    mod_shared: np.ndarray,
    w: Dict[str, np.ndarray],
    *,
    n_q: int,
    n_kv: int,
    hd: int,
    eps: float = 1e-6,
    rope_base: float = 10000.0,
    gate_on: bool = True,
    rope_on: bool = True,
    rows: Optional[Sequence[np.ndarray]] = None,
    store=None,
) -> Dict[str, list]:
    """One single-stream block forward over the joint [text; image] sequence.

    x_txt [B, Nt, d], x_img [B, H*W, d], mod_shared [B, 6, d]. ``w`` holds
    w_qkvg (rows q | k | v | g), w_o, w_gate, w_up, w_down, norm1_w, norm2_w,
    q_norm_w, k_norm_w, mod_bias.

    ``rows`` (optional, one index array per batch element) restricts the output
    to those joint-sequence rows. Every step except the keys/values is row-local,
    so K and V are still formed for all L rows and the sampled rows are exact.

    ``store``: None is the exact definition. A dtype name ("bf16" or "fp32"), or a dict
    from intermediate name (xn, q, k, v, g, o_g, h1, hn, hmid, out) to dtype name, rounds
    those intermediates round-to-nearest-even at the point where an implementation
    stores them (names missing from the dict stay exact); the arithmetic between
    stores stays float64.

    Returns a dict of per-batch lists: ``rows`` and, for those rows, q and k
    (after QK-norm and RoPE, [n_q|n_kv, R, hd]), v, g (the gate sigmoid(xn W_g^T),
    [R, n_q*hd]), o_g ([R, n_q*hd], the gated attention output), h1, hn, hmid (SwiGLU
    hidden [R, F]) and out [R, d].
    """
    x_txt = np.asarray(x_txt, F64)
    x_img = np.asarray(x_img, F64)
    B, Nt, d = x_txt.shape
    H, W = int(img_hw[0]), int(img_hw[1])
    L = Nt + H * W
    mod = modulation(mod_shared, w["mod_bias"])
    wq_rows = n_q * hd
    wk_rows = n_kv * hd
    w_qkvg = np.asarray(w["w_qkvg"], F64)
    Wq = w_qkvg[:wq_rows]
    Wk = w_qkvg[wq_rows: wq_rows + wk_rows]
    Wv = w_qkvg[wq_rows + wk_rows: wq_rows + 2 * wk_rows]
    Wg = w_qkvg[wq_rows + 2 * wk_rows: 2 * wq_rows + 2 * wk_rows] if gate_on else None
    W_o = np.asarray(w["w_o"], F64)

    names = ("xn", "q", "k", "v", "g", "o_g", "h1", "hn", "hmid", "out")
    smap = store if isinstance(store, dict) else {n: store for n in names}
    rnd = {n: storage_rounding(smap.get(n)) for n in names}
    pos = token_positions(Nt, H, W)
    ang = rope_angles(pos, hd, rope_base)

    res = {k: [] for k in ("rows", "q", "k", "v", "g", "o_g", "h1", "hn", "hmid", "out")}
    for b in range(B):
        # joint sequence, text rows first ("架构 › 模态流": single-stream block)
        X = np.concatenate([x_txt[b], x_img[b]], axis=0)
        R = np.arange(L) if rows is None else np.asarray(rows[b], dtype=np.int64)

        # pre-norm + modulation: x_norm * (1 + scale) + shift
        xn = rnd["xn"](zero_centred_rms_norm(X, w["norm1_w"], eps) * (1.0 + mod["scale_a"][b]) + mod["shift_a"][b])

        def heads(m, n):  # [L', n*hd] -> [n, L', hd]
            return m.reshape(m.shape[0], n, hd).transpose(1, 0, 2)

        # K and V for every row; Q and G for the sampled rows only
        k = heads(xn @ Wk.T, n_kv)
        v = rnd["v"](heads(xn @ Wv.T, n_kv))
        q = heads(xn[R] @ Wq.T, n_q)
        # per-head QK-RMSNorm over head_dim, zero-centred gain
        q = zero_centred_rms_norm(q, w["q_norm_w"], eps)
        k = zero_centred_rms_norm(k, w["k_norm_w"], eps)
        if rope_on:
            q = apply_rope_2d(q, ang[R])
            k = apply_rope_2d(k, ang)
        q, k = rnd["q"](q), rnd["k"](k)

        o = gqa_attention(q, k, v)  # [n_q, R, hd]
        o = o.transpose(1, 0, 2).reshape(len(R), n_q * hd)
        if gate_on:
            # head-specific elementwise sigmoid gate on the SDPA output; g is the gate
            # value itself, rounded where an implementation stores it
            g = rnd["g"](sigmoid(xn[R] @ Wg.T))
            o_g = o * g
        else:
            g = np.zeros_like(o)
            o_g = o
        o_g = rnd["o_g"](o_g)

        # gated residual ("架构 › 残差设计": standard residual)
        h1 = rnd["h1"](X[R] + mod["gate_a"][b] * (o_g @ W_o.T))
        hn = rnd["hn"](zero_centred_rms_norm(h1, w["norm2_w"], eps) * (1.0 + mod["scale_m"][b]) + mod["shift_m"][b])
        hmid = rnd["hmid"](swiglu(hn, w["w_gate"], w["w_up"]))
        out = rnd["out"](h1 + mod["gate_m"][b] * (hmid @ np.asarray(w["w_down"], F64).T))

        res["rows"].append(R)
        res["q"].append(q)
        res["k"].append(k[:, R])
        res["v"].append(v[:, R])
        res["g"].append(g)
        res["o_g"].append(o_g)
        res["h1"].append(h1)
        res["hn"].append(hn)
        res["hmid"].append(hmid)
        res["out"].append(out)
    return res


def stack_forward(
    x_txt: np.ndarray,
    x_img: np.ndarray,
    img_hw: Sequence[int],
    mod_shared: np.ndarray,
    ws: Sequence[Dict[str, np.ndarray]],
    *,
    store=None,
    **kw,
) -> np.ndarray:
    """A stack of single-stream blocks: block i (weights ``ws[i]``, its own mod_bias on
    the shared timestep modulation) maps the joint sequence to the next one ("架构 › 模态流" /
    Modality streams: text and image tokens pass through every block as one sequence).
    Returns the last block's output [B, L, d] (text rows first). ``store`` and the other
    keywords are block_forward's; with ``store`` set, each block's output is rounded where
    an implementation stores it, so the next block reads the rounded value."""
    x_txt = np.asarray(x_txt, F64)
    x_img = np.asarray(x_img, F64)
    Nt = x_txt.shape[1]
    X = np.concatenate([x_txt, x_img], axis=1)
    for w in ws:
        out = block_forward(X[:, :Nt], X[:, Nt:], img_hw, mod_shared, w, store=store, **kw)["out"]
        X = np.stack(out, axis=0)
    return X
