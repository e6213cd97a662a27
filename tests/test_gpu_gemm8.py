"""8-bit GEMM modes (e4m3 operands, tensor-wise or row-wise power-of-two scales) against
the fp64 8-bit oracle (``oracle.gemm8``).

What is compared:
* weight codes and factors from krea_dit_weights8_quantize: bit for bit (both sides cast
  the same bf16 values);
* the activation operands (codes times factors): XN8 and HN8 equal the oracle's except
  for one-step flips of at most a 1e-3 fraction of the values (where the bf16 value they
  were cast from sits one ulp away); OG8 and HMID8 within their source's allowance plus
  one e4m3 step;
* every stored intermediate (q, k, v, g, o_g, h1, hmid, out) against the oracle with the
  path's storage rounding, allowing one ulp of the stored value, as in the bf16 mode, and
  downstream of each e4m3 cast also the spread that the observed differences of the cast
  operand carry through the GEMM (see report8);
* the output's distance from the exact 8-bit oracle is reported, not asserted (see
  report8).
"""
from typing import Dict

import numpy as np
import pytest
import torch

import dit_inputs as di
import oracle
from gpu_helpers import TOL, UNIT_ROUNDOFF, excess, make_block, path_storage, rel_max_err, upload
from oracle import gemm8 as g8

pytestmark = pytest.mark.gpu

MATS = ("w_qkvg", "w_o", "w_gate", "w_up", "w_down")
E4M3_STEP = 2.0 ** -3  # spacing of e4m3 values relative to the binade


def decode_e4m3(codes: torch.Tensor) -> np.ndarray:
    return codes.view(torch.float8_e4m3fn).to(torch.float64).cpu().numpy()


def make_block8(cfg, scaling):
    return make_block(cfg.replace(dtype="fp8_" + scaling))


def run_gpu8(case, scaling, ms_scale=1.0):
    cfg = case.cfg
    blk = make_block8(cfg, scaling)
    try:
        t, x_img, x_txt = upload(blk, case)
        ms = blk.timestep_embed(t) * ms_scale
        out = blk.forward(x_img, x_txt, cfg.B, cfg.img_h, cfg.img_w, cfg.n_txt, ms)
        torch.cuda.synchronize()
        B, L, T, hd, d, F = cfg.B, cfg.L, cfg.T, cfg.hd, cfg.d, cfg.F
        nq = cfg.n_q * hd
        rows = T if scaling == "row" else 1
        ws = {
            "q": blk.workspace("Q", (B, cfg.n_q, L, hd)),
            "k": blk.workspace("K", (B, cfg.n_kv, L, hd)),
            "vt": blk.workspace("VT", (B, cfg.n_kv, hd, (L + 63) // 64 * 64)),
            "g": blk.workspace("G", (B, L, nq)),
            "o_g": blk.workspace("OG", (B, L, nq)),
            "h1": blk.workspace("H1", (B, L, d)),
            "hmid": blk.workspace("HMID", (B, L, F)),
        }
        ops = {}
        for name, K in (("xn8", d), ("og8", nq), ("hn8", d), ("hmid8", F)):
            codes = decode_e4m3(blk.workspace(name.upper(), (T, K)))
            dq = blk.workspace("DQ_" + name[:-1].upper(), (rows,)).double().cpu().numpy()
            ops[name] = (codes, dq)
        w8 = {k: (decode_e4m3(blk.w8[k]), blk.w8["dq_" + k[2:]].double().cpu().numpy()) for k in MATS}
        f = lambda x: x.double().cpu().numpy()  # noqa: E731
        res: Dict = {k: [] for k in ("q", "k", "v", "g", "o_g", "h1", "hmid", "out")}
        for b in range(B):
            res["q"].append(f(ws["q"][b]))
            res["k"].append(f(ws["k"][b]))
            res["v"].append(f(ws["vt"][b][:, :, :L].transpose(1, 2)))
            res["g"].append(f(ws["g"][b]))
            res["o_g"].append(f(ws["o_g"][b]))
            res["h1"].append(f(ws["h1"][b]))
            res["hmid"].append(f(ws["hmid"][b]))
            res["out"].append(f(out[b]))
        res["mod_shared"] = ms.double().cpu().numpy()
        res["ops"] = ops
        res["w8"] = w8
        return res
    finally:
        blk.close()


def operand_values(gpu, name, per_row):
    codes, dq = gpu["ops"][name]
    return codes * (dq[:, None] if per_row else dq[0])


def operand_mismatch(got, ref, dq, per_row):
    """Fraction of operand values that differ from the oracle's, and the worst
    difference in e4m3 steps (relative to the larger magnitude's binade)."""
    diff = np.abs(got - ref)
    bad = diff > 0
    if not bad.any():
        return 0.0, 0.0
    mag = np.maximum(np.abs(got), np.abs(ref))[bad]
    binade = np.ldexp(1.0, np.frexp(mag)[1] - 1)
    sub = (np.broadcast_to(dq[:, None], got.shape) if per_row else np.full_like(got, dq[0]))[bad] * 2.0 ** -9
    steps = diff[bad] / np.maximum(binade * E4M3_STEP, sub)
    return float(bad.mean()), float(steps.max())


def ratio(got, ref, bound):
    """max_i |got - ref|_i / bound_i (<= 1 passes)."""
    return float(np.max(np.abs(got - ref) / np.maximum(bound, 1e-300))) if ref.size else 0.0


Z = 6.0  # standard deviations of a sum of sign-symmetric terms covered by the carry allowance


def carry(d_op, W):
    """Spread that operand differences d_op [R, K] carry through a projection with weights
    W [N, K]: Z * sqrt(d_op^2 (W^2)^T). The weights are sign-symmetric, so the carried
    terms d_j W_cj have independent random signs; for a single differing value the bound
    is Z times that value's whole effect."""
    return Z * np.sqrt((d_op ** 2) @ (np.asarray(W) ** 2).T)


def report8(case, gpu, scaling) -> Dict[str, float]:
    """Parity report of one 8-bit forward.

    The e4m3 cast is discontinuous: where a bf16 value the path casts sits one ulp away
    from the oracle's (after an attention approximation, or a differently rounded
    residual), its e4m3 code can land one step (1/8 of the value) away, and the GEMM that
    reads it carries that difference on. So every stage downstream of a cast is checked
    against the oracle (with the path's storage rounding) with its own tolerance
    (TOL * RMS + one ulp of the stored value) plus the spread that the observed
    differences of its e4m3 input operand carry through the GEMM (``carry``; for SwiGLU
    silu(a) u moves by at most 1.1 |u| e_a + |silu(a)| e_u + 1.1 e_a e_u, |silu'| <= 1.1).
    The oracle side never uses a GPU value: only the allowance does. The operands
    themselves are checked too: xn8 (cast from the caller's input) up to one-step flips of
    at most a 1e-3 fraction of the values, og8 and hn8 within TOL * RMS + (ulp + one e4m3
    step) |ref|, hmid8 within hmid's allowance plus one step. The output's distance from
    the exact 8-bit oracle (no storage rounding) is reported, not asserted: that
    definition casts different (unrounded) values and so differs by the same kind of
    flips."""
    cfg = case.cfg
    per_row = scaling == "row"
    ms = gpu["mod_shared"]
    store = path_storage("bf16")
    ref_st = g8.run_case8(case, scaling, mod_shared=ms, store=store)
    ref = g8.run_case8(case, scaling, mod_shared=ms)
    tol, u = TOL["bf16"], UNIT_ROUNDOFF["bf16"]
    ulp = {n: 2 * UNIT_ROUNDOFF[store[n]] for n in store}
    cat = lambda xs: np.concatenate(xs, axis=0)  # noqa: E731
    rms = lambda x: float(np.sqrt(np.mean(x ** 2))) if x.size else 0.0  # noqa: E731
    rep = {"out_maxabs_rms_exact8": rel_max_err(gpu["out"], ref["out"]),
           "out_exact_excess": excess(gpu["out"], ref["out"], tol, u)}
    for k in ("q", "k", "v", "o_g") + (("g",) if cfg.gate_on else ()):
        rep[k] = excess(gpu[k], ref_st[k], tol, ulp[k])

    ops = {n: operand_values(gpu, n, per_row) for n in ("xn8", "og8", "hn8", "hmid8")}
    ops_r = {n: cat(ref_st[n]) for n in ops}
    d_op = {n: np.abs(ops[n] - ops_r[n]) for n in ops}
    Wd = {k: g8.dequantized(case.w[k], per_row) for k in ("w_o", "w_gate", "w_up", "w_down")}
    mod = oracle.modulation(ms, case.w["mod_bias"])
    L = cfg.L
    gate_a = np.repeat(mod["gate_a"], L, axis=0)
    gate_m = np.repeat(mod["gate_m"], L, axis=0)
    X = cat([np.concatenate([case.x_txt[b], case.x_img[b]], axis=0) for b in range(cfg.B)])

    # attention residual: h1 and its branch h1 - X
    h1_g, h1_r = cat(gpu["h1"]), cat(ref_st["h1"])
    carry_a = np.abs(gate_a) * carry(d_op["og8"], Wd["w_o"])
    rep["h1"] = ratio(h1_g, h1_r, tol * rms(h1_r) + ulp["h1"] * np.abs(h1_r) + carry_a)
    br_r = h1_r - X
    rep["attn_branch"] = ratio(h1_g - X, br_r, tol * rms(br_r) + ulp["h1"] * (np.abs(h1_r) + np.abs(X)) + carry_a)
    # SwiGLU output
    hn_r = ops_r["hn8"]
    a_r, u_r = hn_r @ Wd["w_gate"].T, hn_r @ Wd["w_up"].T
    e_a, e_u = carry(d_op["hn8"], Wd["w_gate"]), carry(d_op["hn8"], Wd["w_up"])
    carry_h = 1.1 * np.abs(u_r) * e_a + np.abs(g8.silu(a_r)) * e_u + 1.1 * e_a * e_u
    hm_r = cat(ref_st["hmid"])
    bound_h = tol * rms(hm_r) + ulp["hmid"] * np.abs(hm_r) + carry_h
    rep["hmid"] = ratio(cat(gpu["hmid"]), hm_r, bound_h)
    # MLP residual: out and its branch out - h1 (h1's own difference passes straight through)
    out_g, out_r = cat(gpu["out"]), cat(ref_st["out"])
    carry_m = np.abs(gate_m) * carry(d_op["hmid8"], Wd["w_down"]) + np.abs(h1_g - h1_r)
    rep["out"] = ratio(out_g, out_r, tol * rms(out_r) + ulp["out"] * np.abs(out_r) + carry_m)
    bm_r = out_r - h1_r
    rep["mlp_branch"] = ratio(out_g - h1_g, bm_r,
                              tol * rms(bm_r) + ulp["out"] * (np.abs(out_r) + np.abs(h1_r)) + carry_m)
    # operands
    frac, steps = operand_mismatch(ops["xn8"], ops_r["xn8"], gpu["ops"]["xn8"][1], per_row)
    rep["xn8_mismatch_frac"] = frac
    rep["xn8_max_steps"] = steps
    for n, src in (("og8", "o_g"), ("hn8", "hn")):
        r = ops_r[n]
        rep[n] = ratio(ops[n], r, tol * rms(r) + (ulp[src] + E4M3_STEP) * np.abs(r))
    r = ops_r["hmid8"]
    rep["hmid8"] = ratio(ops["hmid8"], r, bound_h + E4M3_STEP * np.abs(r))
    return rep


INFO = ("_rms_exact8", "_exact_excess")


def check8(case, scaling, ms_scale=1.0):
    gpu = run_gpu8(case, scaling, ms_scale)
    rep = report8(case, gpu, scaling)
    bad = {k: v for k, v in rep.items()
           if (k.endswith("_mismatch_frac") and v > 1e-3) or (k.endswith("_max_steps") and v > 1.0 + 1e-9)
           or (not k.endswith(("_mismatch_frac", "_max_steps") + INFO) and v > 1.0)}
    assert not bad, f"{case.cfg.name} {scaling}: parity failures {bad}; full report {rep}"
    return gpu, rep


SMALL = ["small_a", "small_b", "small_c", "small_imgonly", "small_txtonly"]


@pytest.mark.parametrize("scaling", ["tensor", "row"])
@pytest.mark.parametrize("name", SMALL)
def test_gemm8_small_parity(name, scaling):
    check8(di.make_case(di.CONFIGS[name]), scaling)


@pytest.mark.parametrize("scaling", ["tensor", "row"])
def test_gemm8_without_output_gate(scaling):
    check8(di.make_case(di.CONFIGS["small_a"].replace(gate_on=False)), scaling)


@pytest.mark.parametrize("scaling", ["tensor", "row"])
def test_gemm8_branch_dominant(scaling):
    """Small inputs and doubled modulation: the branches dominate the output."""
    case = di.make_case(di.CONFIGS["small_c"], x_scale=0.05)
    gpu, _ = check8(case, scaling, ms_scale=2.0)
    X = np.concatenate([case.x_txt, case.x_img], axis=1)
    assert rel_max_err([X], [np.stack(gpu["out"])]) > 0.5  # the branches dominate


@pytest.mark.parametrize("scaling", ["tensor", "row"])
def test_weights8_codes_are_exact(scaling):
    cfg = di.CONFIGS["small_b"]
    case = di.make_case(cfg)
    gpu = run_gpu8(case, scaling)
    for k in MATS:
        codes, dq = gpu["w8"][k]
        q, d = g8.quantize(case.w[k], scaling == "row")
        np.testing.assert_array_equal(codes, q, err_msg=k)
        np.testing.assert_array_equal(dq, np.ravel(d), err_msg=k)


def test_8bit_handle_rejects_the_bf16_entry_points():
    from diffusion_transformer_block_gb300 import KREA_DIT_ERR_INVALID_ARG, KreaDitError, krea_dit_block_forward

    cfg = di.CONFIGS["small_a"]
    case = di.make_case(cfg)
    blk = make_block8(cfg, "row")
    try:
        t, x_img, x_txt = upload(blk, case)
        ms = blk.timestep_embed(t)
        out = torch.empty(cfg.B, cfg.L, cfg.d, device=blk.device, dtype=torch.bfloat16)
        with pytest.raises(KreaDitError) as e:
            krea_dit_block_forward(blk.handle, x_img, x_txt, cfg.B, cfg.img_h, cfg.img_w, cfg.n_txt, ms, blk._wstruct,
                                   out, torch.cuda.current_stream())
        assert e.value.status == KREA_DIT_ERR_INVALID_ARG
    finally:
        blk.close()


@pytest.mark.slow
@pytest.mark.parametrize("name,scaling", [("256px", "tensor"), ("512px", "row")])
def test_gemm8_full_size(name, scaling):
    """The pages' pairings: tensor-wise scaling at 256px, row-wise at 512px, full batch."""
    _, rep = check8(di.make_case(di.CONFIGS[name]), scaling)
    print(f"{name} {scaling}: " + ", ".join(f"{k} {v:.4g}" for k, v in rep.items()))
