"""8-bit GEMM modes (e4m3 operands, tensor-wise or row-wise power-of-two scales) against
the fp64 8-bit oracle (``oracle.gemm8``).

Every allowance below is computed from the oracle's values and fixed constants; device
values appear only on the measured side of a comparison. What is compared:
* weight codes and factors from krea_dit_weights8_quantize: bit for bit (both sides cast
  the same bf16 values);
* the four activation operands (codes times factors): each within the a-priori bound of
  tests/e4m3_budget.py, given a stated budget for how far the device's pre-cast bf16
  value may sit from the oracle's (zero change allowed where no admissible value could
  move the cast);
* every stored intermediate against the oracle with the path's storage rounding, as in
  the bf16 mode, and downstream of each cast also the spread that the operand bound
  carries through the GEMM;
* the output against the exact 8-bit oracle (no storage rounding), within the storage-
  rounded bound plus the oracle's own distance between the two definitions.
"""
from typing import Dict

import numpy as np
import pytest
import torch

import dit_inputs as di
import oracle
from e4m3_budget import attention_spread, bf16_ulp, carry, cast_change_bound, norm_carry
from gpu_helpers import TOL, UNIT_ROUNDOFF, excess, make_block, path_storage, record, rel_max_err, upload
from oracle import gemm8 as g8

pytestmark = pytest.mark.gpu

MATS = ("w_qkvg", "w_o", "w_gate", "w_up", "w_down")


def decode_e4m3(codes: torch.Tensor) -> np.ndarray:
    return codes.view(torch.float8_e4m3fn).to(torch.float64).cpu().numpy()


def make_block8(cfg, scaling):
    return make_block(cfg.replace(dtype="fp8_" + scaling))


def run_gpu8(case, scaling, ms_scale=1.0):
    """One 8-bit forward. Its modulation input is the oracle's timestep embedding (times
    ms_scale, rounded to fp32), so that both sides start from the same values."""
    cfg = case.cfg
    blk = make_block8(cfg, scaling)
    try:
        upload(blk, case)
        ms_in = (oracle.mod_shared_for(case) * ms_scale).astype(np.float32)
        ms = torch.from_numpy(ms_in).to(blk.device)
        x_img = case.dev["x_img"].to(blk.device).contiguous()
        x_txt = case.dev["x_txt"].to(blk.device).contiguous()
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
        res["mod_shared"] = ms_in.astype(np.float64)  # the input both sides used (not a device result)
        res["ops"] = ops
        res["w8"] = w8
        return res
    finally:
        blk.close()


def operand_values(gpu, name, per_row):
    codes, dq = gpu["ops"][name]
    return codes * (dq[:, None] if per_row else dq[0])


def ratio(got, ref, bound):
    """max_i |got - ref|_i / bound_i (<= 1 passes; where the bound is 0 only equality passes)."""
    if not ref.size:
        return 0.0
    diff = np.abs(got - ref)
    return float(np.max(np.where(diff > 0, diff / np.maximum(bound, 1e-300), 0.0)))


def worst(got, ref, bound, **extra):
    """Where ``ratio`` is largest: flat index, values there and the named extra arrays."""
    diff = np.abs(got - ref)
    r = np.where(diff > 0, diff / np.maximum(bound, 1e-300), 0.0)
    i = int(np.argmax(r)) if r.size else 0
    out = {"index": i, "ratio": float(r.flat[i]) if r.size else 0.0, "got": float(got.flat[i]) if r.size else 0.0,
           "ref": float(ref.flat[i]) if r.size else 0.0, "bound": float(bound.flat[i]) if r.size else 0.0}
    for k, v in extra.items():
        out[k] = float(np.asarray(v).flat[i]) if np.asarray(v).size > 1 else float(v)
    return out


# Budgets for how far the device's pre-cast bf16 value of each operand may sit from the
# oracle's (stored value against stored value). xn (norm1 of the caller's input) and hmid
# (silu(a) u of fp32 products) are fp32 computations rounded to bf16: one ulp. o_g is
# rounded once more than that, and its gate value g may sit one ulp away: two ulps, plus
# the attention's own rounding: the device rounds every probability to bf16 (relative
# error <= 2^-9) before the P V product, which moves o by about 2^-9 * sqrt(sum p^2 v^2)
# per standard deviation (random signs; ``attention_spread``), times |g|. Z_ATT = 10
# standard deviations: over the ~5e7 elements of a full-size call the largest of that
# many normal deviates reaches about 5.8, and the model leaves out smaller terms (q, k
# or g one ulp away from the oracle's rounding, which moves the logits; the order of the
# fp32 sums), which took single elements of the 256px and 512px calls to 1.2-1.4 times a
# six-deviation allowance. hn and hmid also move with
# whatever the operand casts upstream of them carried (the attention output's flips reach
# h1 and through the norm hn; the flips of hn reach hmid through the SwiGLU product rule).
# These budgets are assumptions, and the test checks them: a device operand that left
# its budget would land outside the cast bound and fail the operand check.
M_ULP = {"xn": 1.0, "o_g": 2.0, "hn": 1.0, "hmid": 1.0}
P_ROUND = 2.0 ** -9
Z_ATT = 10.0


def report8(case, gpu, scaling) -> Dict[str, float]:
    """Parity report of one 8-bit forward; every entry is a ratio to an oracle-side
    bound (<= 1 passes), except the ``_info`` entries.

    Operand bounds come from ``cast_change_bound`` under the budgets above. Downstream
    of each cast, the allowance adds the spread its operand bound carries through the
    GEMM (``carry``; through SwiGLU by the product rule with |silu'| <= 1.1). The
    output is checked against the oracle with the path's storage rounding and against
    the exact 8-bit oracle (no storage rounding), the latter within the former's bound
    plus the oracle's own distance between the two definitions."""
    cfg = case.cfg
    per_row = scaling == "row"
    ms = gpu["mod_shared"]
    store = path_storage("bf16")
    ref_st = g8.run_case8(case, scaling, mod_shared=ms, store=store)
    ref = g8.run_case8(case, scaling, mod_shared=ms)
    tol = TOL["bf16"]
    ulp = {n: 2 * UNIT_ROUNDOFF[store[n]] for n in store}
    cat = lambda xs: np.concatenate(xs, axis=0)  # noqa: E731
    rms = lambda x: float(np.sqrt(np.mean(x ** 2))) if x.size else 0.0  # noqa: E731
    rep = {}
    for k in ("q", "k", "v", "o_g") + (("g",) if cfg.gate_on else ()):
        rep[k] = excess(gpu[k], ref_st[k], tol, ulp[k])

    ops = {n: operand_values(gpu, n, per_row) for n in ("xn8", "og8", "hn8", "hmid8")}
    Wd = {k: g8.dequantized(case.w[k], per_row) for k in ("w_o", "w_gate", "w_up", "w_down")}
    mod = oracle.modulation(ms, case.w["mod_bias"])
    L = cfg.L
    gate_a = np.repeat(mod["gate_a"], L, axis=0)
    gate_m = np.repeat(mod["gate_m"], L, axis=0)
    gamma2 = np.repeat((1.0 + case.w["norm2_w"])[None, :] * (1.0 + mod["scale_m"]), L, axis=0)
    X = cat([np.concatenate([case.x_txt[b], case.x_img[b]], axis=0) for b in range(cfg.B)])

    # xn8: the fused projection's operand
    v = cat(ref_st["xn"])
    ref_xn8, bd_xn8 = cast_change_bound(v, M_ULP["xn"] * bf16_ulp(v), per_row)
    rep["xn8"] = ratio(ops["xn8"], ref_xn8, bd_xn8)
    # og8 -> attention residual: h1 and its branch h1 - X
    v = cat(ref_st["o_g"])
    spread = cat([attention_spread(ref_st["q"][b], ref_st["k"][b], ref_st["v"][b]) for b in range(cfg.B)])
    gabs = np.abs(cat(ref_st["g"])) if cfg.gate_on else 1.0
    d_og = M_ULP["o_g"] * bf16_ulp(v) + Z_ATT * P_ROUND * gabs * spread
    del spread
    ref_og8, bd_og8 = cast_change_bound(v, d_og, per_row)
    rep["og8"] = ratio(ops["og8"], ref_og8, bd_og8)
    og_g = cat(gpu["o_g"])
    rep["og8_worst_info"] = worst(ops["og8"], ref_og8, bd_og8, o_g_ref=v, o_g_gpu=og_g, budget=d_og,
                                  o_g_dev_over_budget=np.abs(og_g - v) / np.maximum(d_og, 1e-300),
                                  dq_gpu=gpu["ops"]["og8"][1][0] if not per_row else 0.0,
                                  dq_ref=float(g8.quantize(v, per_row)[1].flat[0]) if not per_row else 0.0)
    rep["o_g_dev_over_budget_info"] = float(np.max(np.abs(og_g - v) / np.maximum(d_og, 1e-300))) if v.size else 0.0
    carry_a = np.abs(gate_a) * carry(bd_og8, Wd["w_o"])
    h1_g, h1_r = cat(gpu["h1"]), cat(ref_st["h1"])
    rep["h1"] = ratio(h1_g, h1_r, tol * rms(h1_r) + ulp["h1"] * np.abs(h1_r) + carry_a)
    br_r = h1_r - X
    rep["attn_branch"] = ratio(h1_g - X, br_r, tol * rms(br_r) + ulp["h1"] * (np.abs(h1_r) + np.abs(X)) + carry_a)
    # hn8: norm2 of h1, which moved by at most carry_a on top of its own rounding
    hn_r = cat(ref_st["hn"])
    d_hn = M_ULP["hn"] * bf16_ulp(hn_r) + norm_carry(h1_r, gamma2, carry_a, cfg.eps)
    ref_hn8, bd_hn8 = cast_change_bound(hn_r, d_hn, per_row)
    rep["hn8"] = ratio(ops["hn8"], ref_hn8, bd_hn8)
    # SwiGLU output hmid, then its cast
    a_r, u_r = ref_hn8 @ Wd["w_gate"].T, ref_hn8 @ Wd["w_up"].T
    e_a, e_u = carry(bd_hn8, Wd["w_gate"]), carry(bd_hn8, Wd["w_up"])
    carry_h = 1.1 * np.abs(u_r) * e_a + np.abs(g8.silu(a_r)) * e_u + 1.1 * e_a * e_u
    del a_r, u_r, e_a, e_u
    hm_r = cat(ref_st["hmid"])
    rep["hmid"] = ratio(cat(gpu["hmid"]), hm_r, tol * rms(hm_r) + ulp["hmid"] * np.abs(hm_r) + carry_h)
    ref_hmid8, bd_hmid8 = cast_change_bound(hm_r, M_ULP["hmid"] * bf16_ulp(hm_r) + carry_h, per_row)
    del carry_h
    rep["hmid8"] = ratio(ops["hmid8"], ref_hmid8, bd_hmid8)
    # MLP residual: out and its branch out - h1 (h1's flips pass straight through to out)
    carry_m = np.abs(gate_m) * carry(bd_hmid8, Wd["w_down"])
    out_g, out_r = cat(gpu["out"]), cat(ref_st["out"])
    bound_out = tol * rms(out_r) + ulp["out"] * np.abs(out_r) + carry_m + carry_a
    rep["out"] = ratio(out_g, out_r, bound_out)
    bm_r = out_r - h1_r
    rep["mlp_branch"] = ratio(out_g - h1_g, bm_r,
                              tol * rms(bm_r) + ulp["out"] * (np.abs(out_r) + np.abs(h1_r)) + carry_m)
    # the exact 8-bit definition (no storage rounding): the oracle's own distance between
    # the two definitions is added to the storage-rounded bound
    out_x = cat(ref["out"])
    bound_x = bound_out + np.abs(out_r - out_x)
    rep["out_exact8"] = ratio(out_g, out_x, bound_x)
    rms_x = max(rms(out_x), 1e-300)
    rep["out_exact8_literal_info"] = rel_max_err([out_g], [out_x])
    rep["out_exact8_literal_bound_info"] = float(np.max(bound_x) / rms_x) if out_x.size else 0.0
    # how much of each operand the bounds allow to move (a-priori fractions)
    for n, bd in (("xn8", bd_xn8), ("og8", bd_og8), ("hn8", bd_hn8), ("hmid8", bd_hmid8)):
        rep[n + "_movable_frac_info"] = float(np.mean(bd > 0)) if bd.size else 0.0
        rep[n + "_moved_frac_info"] = float(np.mean(ops[n] != {"xn8": ref_xn8, "og8": ref_og8, "hn8": ref_hn8,
                                                                "hmid8": ref_hmid8}[n])) if bd.size else 0.0
    return rep


def check8(case, scaling, ms_scale=1.0):
    gpu = run_gpu8(case, scaling, ms_scale)
    rep = report8(case, gpu, scaling)
    record({"case": case.cfg.name, "mode": "fp8_" + scaling, "report": rep})
    bad = {k: v for k, v in rep.items() if not k.endswith("_info") and v > 1.0}
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
    print(f"{name} {scaling}: " + ", ".join(f"{k} {v:.4g}" if isinstance(v, float) else f"{k} {v}"
                                            for k, v in rep.items()))
