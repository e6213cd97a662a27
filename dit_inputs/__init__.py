"""Seeded synthetic inputs for the Krea 2 single-stream DiT block.

This module is shared by the CPU oracle's tests and by the GPU harness. It holds
shapes, seeds and random draws only: none of the block's arithmetic lives here.

Workload shapes follow the Krea 2 Technical Report, "Training › Pretraining"
(256px -> 512px -> 1024px stages) and "Future work" (native 2K); the widths, head
counts and FFN size are fixed by the build's configuration table below, since the
report does not print them.

Recipe (every config): draws come from one ``torch.Generator`` seeded with the
config's seed, in float64, in this fixed order:

    t ~ U[0, 1)                                  [B]
    temb.w1 [d, 256], temb.b1 [d], temb.w2 [6d, d], temb.b2 [6d]   ~ N(0, 0.02)
    w_qkvg [(2 n_q + 2 n_kv) hd, d] (rows q|k|v|g; no g rows when the gate is
        off), w_o [d, n_q hd],
    w_gate [F, d], w_up [F, d], w_down [d, F]                      ~ N(0, 0.02)
    norm1_w [d], norm2_w [d], q_norm_w [hd], k_norm_w [hd],
    mod_bias [6, d]                                                ~ N(0, 0.02)
    x_txt [B, Nt, d], x_img [B, H*W, d]                            ~ N(0, 1)

Optional scale factors let a case stress one part (``qk_gain`` adds a constant to
the QK-norm gain offsets, making the attention logits peaky).

Block weights and token activations are then rounded to the storage dtype
(bf16 or fp32); gains, modulation bias, timestep MLP weights and t are rounded to
fp32. Both the oracle and the device receive the same rounded values, so input
quantisation is never counted as error.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional

import numpy as np
import torch

__all__ = ["Config", "CONFIGS", "Case", "make_case", "sample_rows", "config_flops"]


@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    B: int
    img_h: int
    img_w: int
    n_txt: int
    d: int
    n_q: int
    n_kv: int
    hd: int
    F: int
    dtype: str  # "bf16" or "fp32"
    seed: int
    gate_on: bool = True
    eps: float = 1e-6
    rope_base: float = 10000.0

    @property
    def n_img(self) -> int:
        return self.img_h * self.img_w

    @property
    def L(self) -> int:
        return self.n_txt + self.n_img

    @property
    def T(self) -> int:
        return self.B * self.L

    def replace(self, **kw) -> "Config":
        return dataclasses.replace(self, **kw)


def _cfg(name, B, h, w, nt, d, nq, nkv, hd, F, dtype, seed, gate_on=True):
    return Config(name, B, h, w, nt, d, nq, nkv, hd, F, dtype, seed, gate_on)


# The five workloads of the block's specification, plus small bf16 cases that the
# oracle finishes in seconds and that still span several GEMM / attention tiles
# with ragged tails.
CONFIGS: Dict[str, Config] = {
    "tiny": _cfg("tiny", 1, 8, 8, 16, 256, 4, 2, 64, 704, "fp32", 0),
    "256px": _cfg("256px", 32, 16, 16, 256, 3072, 24, 8, 128, 8192, "bf16", 1),
    "512px": _cfg("512px", 8, 32, 32, 256, 3072, 24, 8, 128, 8192, "bf16", 2),
    "1024px": _cfg("1024px", 2, 64, 64, 512, 3072, 24, 8, 128, 8192, "bf16", 3),
}
for _nkv in (24, 8, 4, 1):
    for _g in (True, False):
        _n = f"2k_kv{_nkv}_{'gate' if _g else 'nogate'}"
        CONFIGS[_n] = _cfg(_n, 1, 128, 128, 512, 3072, 24, _nkv, 128, 8192, "bf16", 4, _g)

# Small bf16 parity cases (not benchmark workloads).
CONFIGS["small_a"] = _cfg("small_a", 2, 8, 12, 20, 512, 4, 2, 128, 1408, "bf16", 10)
CONFIGS["small_b"] = _cfg("small_b", 1, 16, 20, 37, 384, 4, 1, 128, 1088, "bf16", 11)
CONFIGS["small_c"] = _cfg("small_c", 3, 12, 16, 64, 768, 6, 6, 128, 2048, "bf16", 12)
CONFIGS["small_imgonly"] = _cfg("small_imgonly", 2, 10, 13, 0, 512, 4, 2, 128, 1408, "bf16", 13)
CONFIGS["small_txtonly"] = _cfg("small_txtonly", 2, 0, 0, 45, 512, 4, 2, 128, 1408, "bf16", 14)
# Odd number of query tiles per KV group (G = 3, 3 tiles): one-tile attention units, and
# 160 units (more than one per SM), so a persistent CTA meets both kinds in one sequence.
CONFIGS["units_odd"] = _cfg("units_odd", 32, 16, 16, 44, 384, 3, 1, 128, 1024, "bf16", 17)
# Many attention units per persistent CTA (64 x 2 KV groups x 5 units = 640 on 152 SMs),
# a one-tile unit closing every KV group and a ragged last query / key tile (L = 300).
CONFIGS["units_many"] = _cfg("units_many", 64, 16, 16, 44, 256, 6, 2, 128, 512, "bf16", 18)
# Many units per CTA with one K/V tile each (L = 100 <= 128), three query tiles per KV
# group (a one-tile unit in every group), gate off (empty staging slots in the ring).
CONFIGS["units_short_nogate"] = _cfg("units_short_nogate", 96, 8, 8, 36, 256, 6, 2, 128, 512, "bf16", 19,
                                     gate_on=False)
CONFIGS["tiny_ragged32"] = _cfg("tiny_ragged32", 2, 5, 7, 9, 192, 3, 1, 64, 320, "fp32", 15)
CONFIGS["small_fp32_hd128"] = _cfg("small_fp32_hd128", 1, 9, 11, 13, 256, 2, 1, 128, 704, "fp32", 16)


@dataclasses.dataclass
class Case:
    """One seeded input set. Every float array is float64 holding exactly the
    rounded values the device receives."""

    cfg: Config
    t: np.ndarray  # [B]
    temb: Dict[str, np.ndarray]  # w1, b1, w2, b2
    w: Dict[str, np.ndarray]  # w_qkvg, w_o, w_gate, w_up, w_down, norm1_w, norm2_w, q_norm_w, k_norm_w, mod_bias
    x_txt: np.ndarray  # [B, Nt, d]
    x_img: np.ndarray  # [B, H*W, d]
    # torch tensors in storage dtype, on the CPU (the harness copies them to the device)
    dev: Dict[str, torch.Tensor]


def _round(a: torch.Tensor, dtype: str) -> torch.Tensor:
    if dtype == "bf16":
        return a.to(torch.bfloat16)
    if dtype == "fp32":
        return a.to(torch.float32)
    raise ValueError(dtype)


def make_case(cfg: Config, *, qk_gain: float = 0.0, x_scale: float = 1.0,
              w_std: float = 0.02) -> Case:
    """Draw one input set for ``cfg`` (recipe in the module docstring)."""
    g = torch.Generator().manual_seed(cfg.seed)
    B, d, hd, F = cfg.B, cfg.d, cfg.hd, cfg.F
    f64 = torch.float64

    def nrm(*shape, std=w_std):
        return torch.randn(*shape, generator=g, dtype=f64) * std

    t = torch.rand(B, generator=g, dtype=f64)
    temb = {"w1": nrm(d, 256), "b1": nrm(d), "w2": nrm(6 * d, d), "b2": nrm(6 * d)}
    # without the output gate the fused projection has no W_g rows
    n_qkvg = ((2 if cfg.gate_on else 1) * cfg.n_q + 2 * cfg.n_kv) * hd
    w = {
        "w_qkvg": nrm(n_qkvg, d),
        "w_o": nrm(d, cfg.n_q * hd),
        "w_gate": nrm(F, d),
        "w_up": nrm(F, d),
        "w_down": nrm(d, F),
    }
    small = {
        "norm1_w": nrm(d), "norm2_w": nrm(d),
        "q_norm_w": nrm(hd) + qk_gain, "k_norm_w": nrm(hd) + qk_gain,
        "mod_bias": nrm(6, d),
    }
    x_txt = torch.randn(B, cfg.n_txt, d, generator=g, dtype=f64) * x_scale
    x_img = torch.randn(B, cfg.n_img, d, generator=g, dtype=f64) * x_scale

    dev: Dict[str, torch.Tensor] = {}
    dev["t"] = t.to(torch.float32)
    for k, v in temb.items():
        dev["temb." + k] = v.to(torch.float32)
    for k, v in w.items():
        dev[k] = _round(v, cfg.dtype)
    for k, v in small.items():
        dev[k] = v.to(torch.float32)
    dev["x_txt"] = _round(x_txt, cfg.dtype)
    dev["x_img"] = _round(x_img, cfg.dtype)

    def back(x: torch.Tensor) -> np.ndarray:
        return x.to(f64).numpy()

    return Case(
        cfg=cfg,
        t=back(dev["t"]),
        temb={k: back(dev["temb." + k]) for k in temb},
        w={**{k: back(dev[k]) for k in w}, **{k: back(dev[k]) for k in small}},
        x_txt=back(dev["x_txt"]),
        x_img=back(dev["x_img"]),
        dev=dev,
    )


def make_stack(cfg: Config, n_blocks: int, **kw) -> List[Case]:
    """Inputs for a stack of ``n_blocks`` blocks: entry 0 is make_case(cfg) (its timestep,
    timestep-MLP weights and token inputs drive the stack); entry i > 0 draws block i's
    weights the same way from seed ``cfg.seed + 7919 * i`` (only its weights are used)."""
    return [make_case(cfg if i == 0 else cfg.replace(seed=cfg.seed + 7919 * i), **kw) for i in range(n_blocks)]


def make_dout(cfg: Config, seed: int = 4321):
    """Upstream gradient [B, L, d] for a backward: standard normal, rounded to the storage
    dtype. Returns (float64 array of the rounded values, torch CPU tensor in the dtype)."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(cfg.B, cfg.L, cfg.d, generator=g, dtype=torch.float64)
    dev = _round(x, cfg.dtype)
    return dev.to(torch.float64).numpy(), dev


def sample_rows(cfg: Config, n_per_batch: int, seed: int = 1234) -> List[np.ndarray]:
    """Stratified row sample per batch element (joint-sequence indices, text rows
    first): first/last text rows, the four image corners, image-edge rows, then
    uniform picks to reach ``n_per_batch``. Sorted, unique."""
    rng = np.random.default_rng(seed)
    out = []
    Nt, H, W, L = cfg.n_txt, cfg.img_h, cfg.img_w, cfg.L
    for _ in range(cfg.B):
        s = set()
        if Nt:
            s.update({0, Nt - 1, Nt // 2})
        if H * W:
            for r, c in [(0, 0), (0, W - 1), (H - 1, 0), (H - 1, W - 1), (H // 2, W // 2)]:
                s.add(Nt + r * W + c)
            for _k in range(8):
                s.add(Nt + int(rng.integers(0, W)))  # top edge
                s.add(Nt + (H - 1) * W + int(rng.integers(0, W)))  # bottom edge
                s.add(Nt + int(rng.integers(0, H)) * W)  # left edge
                s.add(Nt + int(rng.integers(0, H)) * W + W - 1)  # right edge
        want = min(n_per_batch, L)
        while len(s) < want:
            s.add(int(rng.integers(0, L)))
        out.append(np.array(sorted(s), dtype=np.int64))
    return out


def config_flops(cfg: Config) -> float:
    """Algorithmic FLOPs of one block forward (multiply-add = 2 FLOPs): the four
    projections, the two attention contractions, and nothing for elementwise work."""
    T, d, hd, F = cfg.T, cfg.d, cfg.hd, cfg.F
    qkvg_rows = (2 * cfg.n_q + 2 * cfg.n_kv) * hd if cfg.gate_on else (cfg.n_q + 2 * cfg.n_kv) * hd
    lin = 2.0 * T * d * qkvg_rows + 2.0 * T * cfg.n_q * hd * d + 2.0 * T * d * 2 * F + 2.0 * T * F * d
    attn = 4.0 * cfg.B * cfg.L * cfg.L * cfg.n_q * hd
    return lin + attn


def config_backward_flops(cfg: Config) -> float:
    """Algorithmic FLOPs of one block backward: a data and a weight gradient product per
    projection (2x the forward's), and the attention's dV, dP, dQ, dK products plus the
    score product it recomputes (2.5x the forward's two contractions)."""
    attn = 4.0 * cfg.B * cfg.L * cfg.L * cfg.n_q * cfg.hd
    return 2.0 * (config_flops(cfg) - attn) + 2.5 * attn
