"""Helpers shared by the GPU tests: run a seeded case through the C ABI and compare it
with the fp64 oracle on the same rounded inputs."""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence

import numpy as np
import torch

import dit_inputs as di
import oracle
from diffusion_transformer_block_gb300.runner import DitBlock

# unit roundoff of the storage dtype: a stored value carries up to this relative error
UNIT_ROUNDOFF = {"bf16": 2.0 ** -8, "fp32": 2.0 ** -24}
# the block's parity criterion: max-abs error <= TOL * RMS(reference)
TOL = {"bf16": 2e-2, "fp32": 1e-4}


def make_block(cfg: di.Config, max_batch: Optional[int] = None, max_seq: Optional[int] = None) -> DitBlock:
    return DitBlock(max_batch=max_batch or max(cfg.B, 1), max_seq=max_seq or max(cfg.L, 1), d=cfg.d, n_q=cfg.n_q,
                    n_kv=cfg.n_kv, hd=cfg.hd, F=cfg.F, img_h_max=max(cfg.img_h, 1), img_w_max=max(cfg.img_w, 1),
                    gate_on=cfg.gate_on, mode=cfg.dtype, eps=cfg.eps, rope_base=cfg.rope_base)


def upload(blk: DitBlock, case: di.Case):
    dev = blk.device
    blk.set_weights({k: case.dev[k] for k in ("w_qkvg", "w_o", "w_gate", "w_up", "w_down", "norm1_w", "norm2_w",
                                              "q_norm_w", "k_norm_w", "mod_bias")})
    blk.set_temb_weights({k: case.dev["temb." + k] for k in ("w1", "b1", "w2", "b2")})
    t = case.dev["t"].to(dev)
    x_img = case.dev["x_img"].to(dev).contiguous()
    x_txt = case.dev["x_txt"].to(dev).contiguous()
    return t, x_img, x_txt


def run_gpu(case: di.Case, rows: Optional[Sequence[np.ndarray]] = None, blk: Optional[DitBlock] = None,
            mod_shared: Optional[torch.Tensor] = None) -> Dict[str, List[np.ndarray]]:
    """Timestep embed + block forward on the GPU; returns per-batch float64 arrays of the
    requested rows (all rows when ``rows`` is None), keyed like the oracle's result."""
    cfg = case.cfg
    own = blk is None
    blk = blk or make_block(cfg)
    try:
        t, x_img, x_txt = upload(blk, case)
        ms = blk.timestep_embed(t) if mod_shared is None else mod_shared
        out = blk.forward(x_img, x_txt, cfg.B, cfg.img_h, cfg.img_w, cfg.n_txt, ms)
        torch.cuda.synchronize()
        B, L, T, hd = cfg.B, cfg.L, cfg.T, cfg.hd
        ws = {
            "q": blk.workspace("Q", (B, cfg.n_q, L, hd)),
            "k": blk.workspace("K", (B, cfg.n_kv, L, hd)),
            "vt": blk.workspace("VT", (B, cfg.n_kv, hd, (L + 63) // 64 * 64)),
            "g": blk.workspace("G", (B, L, cfg.n_q * hd)),
            "o_g": blk.workspace("OG", (B, L, cfg.n_q * hd)),
            "h1": blk.workspace("H1", (B, L, cfg.d)),
            "hn": blk.workspace("HN", (B, L, cfg.d)),
            "hmid": blk.workspace("HMID", (B, L, cfg.F)),
        }
        res: Dict[str, List[np.ndarray]] = {k: [] for k in ("rows", "q", "k", "v", "g", "o_g", "h1", "hn", "hmid",
                                                            "out")}
        res["mod_shared"] = ms.double().cpu().numpy()
        for b in range(B):
            R = np.arange(L) if rows is None else np.asarray(rows[b])
            Rt = torch.from_numpy(R).to(blk.device)
            f = lambda x: x.double().cpu().numpy()  # noqa: E731
            res["rows"].append(R)
            res["q"].append(f(ws["q"][b][:, Rt]))
            res["k"].append(f(ws["k"][b][:, Rt]))
            res["v"].append(f(ws["vt"][b][:, :, Rt].transpose(1, 2)))
            res["g"].append(f(ws["g"][b][Rt]))
            res["o_g"].append(f(ws["o_g"][b][Rt]))
            res["h1"].append(f(ws["h1"][b][Rt]))
            res["hn"].append(f(ws["hn"][b][Rt]))
            res["hmid"].append(f(ws["hmid"][b][Rt]))
            res["out"].append(f(out[b][Rt]))
        return res
    finally:
        if own:
            blk.close()


def _cat(xs: List[np.ndarray]) -> np.ndarray:
    return np.concatenate([x.reshape(-1) for x in xs]) if xs else np.zeros(0)


def rel_max_err(gpu: List[np.ndarray], ref: List[np.ndarray]) -> float:
    """max |gpu - ref| / RMS(ref) over all listed arrays."""
    g, r = _cat(gpu), _cat(ref)
    if r.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(r * r)))
    return float(np.max(np.abs(g - r)) / max(rms, 1e-300))


def branch_excess(gpu_a, gpu_b, ref_a, ref_b, tol: float, u: float) -> float:
    """Branch check for delta = a - b (a, b stored in the storage dtype):
    returns max_i |d_gpu - d_ref|_i / (tol * RMS(d_ref) + u * (|a_ref| + |b_ref|)_i); <= 1 passes.
    The second term is the rounding of the two stored operands, which no kernel can beat."""
    ga, gb, ra, rb = _cat(gpu_a), _cat(gpu_b), _cat(ref_a), _cat(ref_b)
    dg, dr = ga - gb, ra - rb
    if dr.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(dr * dr)))
    bound = tol * rms + u * (np.abs(ra) + np.abs(rb))
    return float(np.max(np.abs(dg - dr) / np.maximum(bound, 1e-300)))


def joint_rows(case: di.Case, rows: Optional[Sequence[np.ndarray]]) -> List[np.ndarray]:
    X = np.concatenate([case.x_txt, case.x_img], axis=1)
    return [X[b] if rows is None else X[b][np.asarray(rows[b])] for b in range(case.cfg.B)]


def parity_report(case: di.Case, gpu: Dict, ref: Dict) -> Dict[str, float]:
    cfg = case.cfg
    tol, u = TOL[cfg.dtype], UNIT_ROUNDOFF[cfg.dtype]
    X = joint_rows(case, gpu["rows"])
    rep = {k: rel_max_err(gpu[k], ref[k]) for k in ("out", "h1", "q", "k", "v", "o_g", "hn", "hmid")}
    if cfg.gate_on:
        rep["g"] = rel_max_err(gpu["g"], ref["g"])
    rep["attn_branch"] = branch_excess(gpu["h1"], X, ref["h1"], X, tol, u)
    rep["mlp_branch"] = branch_excess(gpu["out"], gpu["h1"], ref["out"], ref["h1"], tol, u)
    return rep


def assert_parity(case: di.Case, gpu: Dict, ref: Dict, intermediates_tol: Optional[float] = None) -> Dict[str, float]:
    rep = parity_report(case, gpu, ref)
    tol = TOL[case.cfg.dtype]
    itol = intermediates_tol or tol
    bad = {k: v for k, v in rep.items() if (v > 1.0 if k.endswith("branch") else v > (tol if k == "out" else itol))}
    assert not bad, f"{case.cfg.name}: parity failures {bad}; full report {rep}"
    return rep
