"""Helpers shared by the GPU tests: run a seeded case through the C ABI and compare it
with the fp64 oracle on the same rounded inputs."""
from __future__ import annotations

import json
import os
from typing import Dict, List, Optional, Sequence

import numpy as np
import torch

import dit_inputs as di
import oracle
from diffusion_transformer_block_gb300.runner import DitBlock

# unit roundoff of a storage dtype: a stored value carries up to this relative error
UNIT_ROUNDOFF = {"bf16": 2.0 ** -8, "fp32": 2.0 ** -24}
# the block's parity criterion: max-abs error <= TOL * RMS(reference)
TOL = {"bf16": 2e-2, "fp32": 1e-4}
NAMES = ("xn", "q", "k", "v", "g", "o_g", "h1", "hn", "hmid", "out")


def path_storage(dtype: str) -> Dict[str, str]:
    """Where the CUDA path rounds: every kept intermediate in the storage dtype, except
    the residual stream h1, which is fp32 in both modes."""
    return {n: ("fp32" if n == "h1" else dtype) for n in NAMES}


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


def excess(gpu: List[np.ndarray], ref: List[np.ndarray], tol: float, ulp: float) -> float:
    """max_i |gpu - ref|_i / (tol * RMS(ref) + ulp * |ref|_i); <= 1 passes. ``ulp`` is one
    unit in the last place of the storage dtype relative to the value (2^-7 for bf16): a
    stored value whose pre-rounding value sits next to a rounding boundary may land one
    ulp away from the reference's rounding."""
    g, r = _cat(gpu), _cat(ref)
    if r.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(r * r)))
    return float(np.max(np.abs(g - r) / np.maximum(tol * rms + ulp * np.abs(r), 1e-300)))


def branch_excess(gpu_a, gpu_b, ref_a, ref_b, tol: float, ulp: float, prop=None) -> float:
    """Branch check for delta = a - b (a, b stored values): max_i |d_gpu - d_ref|_i /
    (tol * RMS(d_ref) + ulp * (|a_ref| + |b_ref|)_i + prop_i); <= 1 passes.
    ``prop`` = the spread that one-ulp differences in the branch's stored input cause
    after its projection (see propagated_ulp)."""
    ga, gb, ra, rb = _cat(gpu_a), _cat(gpu_b), _cat(ref_a), _cat(ref_b)
    dg, dr = ga - gb, ra - rb
    if dr.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(dr * dr)))
    bound = tol * rms + ulp * (np.abs(ra) + np.abs(rb)) + (0.0 if prop is None else _cat(prop))
    return float(np.max(np.abs(dg - dr) / np.maximum(bound, 1e-300)))


def propagated_ulp(inp: List[np.ndarray], W: np.ndarray, gate: np.ndarray, ulp: float) -> List[np.ndarray]:
    """3 sigma of gate * (e W^T) when every element e_j of the stored input independently
    sits one ulp (ulp * |inp_j|) above or below the reference's rounding: an input may
    round the other way when its pre-rounding value lies next to a rounding boundary."""
    W2 = np.asarray(W, np.float64) ** 2
    return [3.0 * np.abs(gate[b]) * np.sqrt(((ulp * x) ** 2) @ W2.T) for b, x in enumerate(inp)]


def joint_rows(case: di.Case, rows: Optional[Sequence[np.ndarray]]) -> List[np.ndarray]:
    X = np.concatenate([case.x_txt, case.x_img], axis=1)
    return [X[b] if rows is None else X[b][np.asarray(rows[b])] for b in range(case.cfg.B)]


STORED = ("q", "k", "v", "o_g", "h1", "hn", "hmid", "out")


def parity_report(case: di.Case, gpu: Dict, ref: Dict, ref_st: Dict) -> Dict[str, float]:
    """``ref`` = exact oracle, ``ref_st`` = oracle with the path's storage rounding.

    out_maxabs_rms : the literal criterion max|out - ref| / RMS(ref), reported.
    out_exact      : the block's criterion with the output's own rounding to its storage
                     dtype excused: max_i |out - ref|_i / (TOL RMS(ref) + u |ref|_i),
                     u = unit roundoff (<= 1 passes). Every rounding upstream of the
                     output counts as error.
    other entries  : excess ratios against ``ref_st`` (<= 1 passes), allowing one ulp of
                     each stored value."""
    cfg = case.cfg
    tol, u = TOL[cfg.dtype], UNIT_ROUNDOFF[cfg.dtype]
    st = path_storage(cfg.dtype)
    ulp = {n: 2 * UNIT_ROUNDOFF[st[n]] for n in NAMES}
    X = joint_rows(case, gpu["rows"])
    rep = {"out_maxabs_rms": rel_max_err(gpu["out"], ref["out"]),
           "out_exact": excess(gpu["out"], ref["out"], tol, u)}
    keys = STORED + (("g",) if cfg.gate_on else ())
    rep.update({k: excess(gpu[k], ref_st[k], tol, ulp[k]) for k in keys})
    mod = oracle.modulation(ref_st["mod_shared"], case.w["mod_bias"])
    prop_a = propagated_ulp(ref_st["o_g"], case.w["w_o"], mod["gate_a"], ulp["o_g"])
    prop_m = propagated_ulp(ref_st["hmid"], case.w["w_down"], mod["gate_m"], ulp["hmid"])
    rep["attn_branch"] = branch_excess(gpu["h1"], X, ref_st["h1"], X, tol, ulp["h1"], prop_a)
    rep["mlp_branch"] = branch_excess(gpu["out"], gpu["h1"], ref_st["out"], ref_st["h1"], tol, ulp["out"], prop_m)
    return rep


def output_split(case: di.Case, gpu: Dict, ref: Dict) -> Dict[str, object]:
    """Splits the block output's error against the exact oracle into the output's own
    rounding and the error of the value it rounds.

    pre = h1 + gate_m * (hmid W_down^T), in fp64 from the GPU's stored h1 (fp32) and hmid:
    the value the down-projection epilogue rounds to the output (up to its fp32
    accumulation, ~1e-6 relative). So |out - pre| is the output's rounding and
    |pre - ref| the error of everything upstream of it, which splits further into the
    residual h1 (|h1 - h1_ref|) and the MLP branch. Returned per workload: the largest
    of each over all compared elements (x RMS(ref)), and the element with the largest
    literal error, with its position, |ref| / RMS and the three parts there."""
    mod = oracle.modulation(np.asarray(gpu["mod_shared"], np.float64), case.w["mod_bias"])
    W = np.asarray(case.w["w_down"], np.float64)
    pre = [gpu["h1"][b] + mod["gate_m"][b] * (gpu["hmid"][b] @ W.T) for b in range(case.cfg.B)]
    out_g, ref_o, pre_c = _cat(gpu["out"]), _cat(ref["out"]), _cat(pre)
    h1_g, h1_r = _cat(gpu["h1"]), _cat(ref["h1"])
    if ref_o.size == 0:
        return {}
    rms = float(np.sqrt(np.mean(ref_o * ref_o)))
    err = np.abs(out_g - ref_o)
    i = int(np.argmax(err))
    d = case.cfg.d
    sizes = [x.size for x in gpu["out"]]
    b = int(np.searchsorted(np.cumsum(sizes), i, side="right"))
    j = i - int(sum(sizes[:b]))
    row, col = int(gpu["rows"][b][j // d]), j % d
    return {
        "maxabs_rms": float(err.max() / rms),
        "rounding_max_rms": float(np.abs(out_g - pre_c).max() / rms),
        "upstream_max_rms": float(np.abs(pre_c - ref_o).max() / rms),
        "h1_max_rms": float(np.abs(h1_g - h1_r).max() / rms),
        "worst": {"batch": b, "row": row, "col": col, "ref_rms": float(abs(ref_o[i]) / rms),
                  "err_rms": float(err[i] / rms), "rounding_rms": float(abs(out_g[i] - pre_c[i]) / rms),
                  "upstream_rms": float(abs(pre_c[i] - ref_o[i]) / rms),
                  "h1_rms": float(abs(h1_g[i] - h1_r[i]) / rms),
                  "mlp_branch_rms": float(abs((pre_c[i] - h1_g[i]) - (ref_o[i] - h1_r[i])) / rms)},
    }


def record(entry: Dict[str, object]) -> None:
    """Appends one JSON line to the file named by KREA_PARITY_RECORD (if set), so a test
    run keeps its parity figures."""
    path = os.environ.get("KREA_PARITY_RECORD")
    if path:
        with open(path, "a") as fh:
            fh.write(json.dumps(entry) + "\n")


def oracle_pair(case: di.Case, rows=None, mod_shared: Optional[np.ndarray] = None):
    ms = oracle.mod_shared_for(case) if mod_shared is None else mod_shared
    ref = oracle.run_case(case, rows=rows, mod_shared=ms)
    ref_st = oracle.run_case(case, rows=rows, mod_shared=ms, store=path_storage(case.cfg.dtype))
    ref_st["mod_shared"] = ms
    return ref, ref_st


def check_parity(case: di.Case, gpu: Dict, rows=None, mod_shared: Optional[np.ndarray] = None) -> Dict[str, float]:
    ref, ref_st = oracle_pair(case, rows, mod_shared)
    rep = parity_report(case, gpu, ref, ref_st)
    split = output_split(case, gpu, ref)
    tol = TOL[case.cfg.dtype]
    # the literal criterion (max-abs error <= tol x RMS), and the error of the value the
    # output rounds (everything upstream of the output's own rounding) within half of it
    rep["out_literal"] = rep["out_maxabs_rms"] / tol
    rep["out_upstream"] = split.get("upstream_max_rms", 0.0) / (0.5 * tol)
    if os.environ.get("KREA_PARITY_RECORD"):
        record({"case": case.cfg.name, "dtype": case.cfg.dtype, "B": case.cfg.B, "L": case.cfg.L,
                "rows": int(sum(len(r) for r in gpu["rows"])), "report": rep, "output_split": split})
    bad = {k: v for k, v in rep.items() if k != "out_maxabs_rms" and v > 1.0}
    assert not bad, f"{case.cfg.name}: parity failures {bad}; full report {rep}"
    return rep
