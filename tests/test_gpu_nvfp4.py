"""NVFP4 GEMM mode (E2M1 operands, E4M3 scales per 16 elements along K, a power-of-two
scale per tensor) against the fp64 NVFP4 oracle (``oracle.nvfp4``).

Every allowance is computed from the oracle's values and fixed constants; device values
appear only on the measured side of a comparison. What is compared:
* the weight casts of krea_dit_weights4_quantize: codes, block scales and tensor scales
  bit for bit (both sides cast the same bf16 values, deciding every rounding the same way);
* the four activation operands (decoded codes x block scales x tensor scale): each within
  the a-priori bound of ``nvfp4_change_bound`` (tests/e4m3_budget.py) under the same
  budgets for the device's pre-cast bf16 values as the 8-bit test;
* every stored intermediate against the oracle with the path's storage rounding, as in
  the 8-bit test, downstream of each cast also the spread its operand bound carries;
* the output against the exact NVFP4 oracle, within that bound plus the oracle's own
  distance between the storage-rounded and the exact definitions.
"""
from typing import Dict

import numpy as np
import pytest
import torch

import dit_inputs as di
import oracle
from e4m3_budget import attention_spread, bf16_ulp, carry, magnitude_range, norm_carry, nvfp4_change_bound
from gpu_helpers import TOL, UNIT_ROUNDOFF, excess, make_block, path_storage, record, rel_max_err, upload
from oracle import nvfp4 as f4
from oracle.block import (apply_rope_2d, round_to_bf16, rope_angles, sigmoid, silu, token_positions,
                          zero_centred_rms_norm)
from test_gpu_gemm8 import M_ULP, P_ROUND, Z_ATT, ratio

pytestmark = pytest.mark.gpu

MATS = ("w_qkvg", "w_o", "w_gate", "w_up", "w_down")
# E2M1 codes 0..15 (sign | exponent(2) | mantissa(1)) decoded from the bit layout
E2M1 = np.array([(-1.0 if c & 8 else 1.0) * ((0.5 * (c & 1)) if ((c >> 1) & 3) == 0
                                             else 2.0 ** (((c >> 1) & 3) - 1) * (1 + 0.5 * (c & 1))) for c in range(16)])


def decode_codes(codes: torch.Tensor, R: int, K: int) -> np.ndarray:
    """[R, K/2] bytes, element 2i in the low nibble of byte i -> [R, K] values."""
    b = codes.cpu().numpy().astype(np.int64).reshape(R, K // 2)
    out = np.empty((R, K))
    out[:, 0::2] = E2M1[b & 15]
    out[:, 1::2] = E2M1[b >> 4]
    return out


def decode_scales(sf: torch.Tensor, R: int, K: int) -> np.ndarray:
    """Scale atoms -> [R, K/16] E4M3 values (row r, block j of the row)."""
    vals = sf.view(torch.float8_e4m3fn).to(torch.float64).cpu().numpy()
    r = np.arange(R)[:, None]
    b = np.arange(K // 16)[None, :]
    idx = ((r // 128) * (K // 64) + b // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + (b % 4)
    return vals[idx]


def dequant(codes, sf, ts, R, K) -> np.ndarray:
    return decode_codes(codes, R, K) * np.repeat(decode_scales(sf, R, K), 16, axis=1) * float(ts)


def run_gpu4(case) -> Dict:
    """One NVFP4 forward; its modulation input is the oracle's timestep embedding (rounded to
    fp32), so that both sides start from the same values."""
    cfg = case.cfg
    blk = make_block(cfg.replace(dtype="nvfp4"))
    try:
        upload(blk, case)
        ms_in = oracle.mod_shared_for(case).astype(np.float32)
        ms = torch.from_numpy(ms_in).to(blk.device)
        x_img = case.dev["x_img"].to(blk.device).contiguous()
        x_txt = case.dev["x_txt"].to(blk.device).contiguous()
        out = blk.forward(x_img, x_txt, cfg.B, cfg.img_h, cfg.img_w, cfg.n_txt, ms)
        torch.cuda.synchronize()
        B, L, T, hd, d, F = cfg.B, cfg.L, cfg.T, cfg.hd, cfg.d, cfg.F
        nq = cfg.n_q * hd
        f = lambda x: x.double().cpu().numpy()  # noqa: E731
        res: Dict = {"q": [], "k": [], "v": [], "g": [], "o_g": [], "h1": [], "hmid": [], "out": []}
        ws = {"q": blk.workspace("Q", (B, cfg.n_q, L, hd)), "k": blk.workspace("K", (B, cfg.n_kv, L, hd)),
              "vt": blk.workspace("VT", (B, cfg.n_kv, hd, (L + 63) // 64 * 64)), "g": blk.workspace("G", (B, L, nq)),
              "o_g": blk.workspace("OG", (B, L, nq)), "h1": blk.workspace("H1", (B, L, d)),
              "hmid": blk.workspace("HMID", (B, L, F))}
        for b in range(B):
            res["q"].append(f(ws["q"][b]))
            res["k"].append(f(ws["k"][b]))
            res["v"].append(f(ws["vt"][b][:, :, :L].transpose(1, 2)))
            res["g"].append(f(ws["g"][b]))
            res["o_g"].append(f(ws["o_g"][b]))
            res["h1"].append(f(ws["h1"][b]))
            res["hmid"].append(f(ws["hmid"][b]))
            res["out"].append(f(out[b]))
        ops = {}
        for name, K in (("XN4", d), ("OG4", nq), ("HN4", d), ("HMID4", F)):
            codes = blk.workspace(name, (T * K // 2,))
            sf = blk.workspace("SF_" + name, (((T + 127) // 128) * 128 * K // 16,))
            ts = blk.workspace("TS_" + name, (1,)).double().cpu().numpy()[0]
            ops[name.lower()] = dequant(codes, sf, ts, T, K)
        w4 = {}
        for k in MATS:
            rows, cols = case.w[k].shape
            w4[k] = (decode_codes(blk.w4[k], rows, cols), decode_scales(blk.w4["sf_" + k[2:]], rows, cols),
                     float(blk.w4["ts_" + k[2:]][0].item()))
        res.update(mod_shared=ms_in.astype(np.float64), ops=ops, w4=w4)
        return res
    finally:
        blk.close()


def report4(case, gpu) -> Dict[str, float]:
    """Parity report of one NVFP4 forward: ratios to oracle-side bounds (<= 1 passes), except
    the ``_info`` entries. Same structure as the 8-bit report, with the NVFP4 cast bound."""
    cfg = case.cfg
    ms = gpu["mod_shared"]
    store = path_storage("bf16")
    ref_st = f4.run_case4(case, mod_shared=ms, store=store)
    ref = f4.run_case4(case, mod_shared=ms)
    tol = TOL["bf16"]
    ulp = {n: 2 * UNIT_ROUNDOFF[store[n]] for n in store}
    cat = lambda xs: np.concatenate(xs, axis=0)  # noqa: E731
    rms = lambda x: float(np.sqrt(np.mean(x ** 2))) if x.size else 0.0  # noqa: E731
    rep = {}
    for k in ("q", "k", "v", "o_g") + (("g",) if cfg.gate_on else ()):
        rep[k] = excess(gpu[k], ref_st[k], tol, ulp[k])
    ops = gpu["ops"]
    Wd = {k: f4.dequantized(case.w[k]) for k in ("w_o", "w_gate", "w_up", "w_down")}
    mod = oracle.modulation(ms, case.w["mod_bias"])
    L = cfg.L
    gate_a = np.repeat(mod["gate_a"], L, axis=0)
    gate_m = np.repeat(mod["gate_m"], L, axis=0)
    gamma2 = np.repeat((1.0 + case.w["norm2_w"])[None, :] * (1.0 + mod["scale_m"]), L, axis=0)
    X = cat([np.concatenate([case.x_txt[b], case.x_img[b]], axis=0) for b in range(cfg.B)])

    v = cat(ref_st["xn"])
    ref_xn, bd_xn = nvfp4_change_bound(v, M_ULP["xn"] * bf16_ulp(v))
    rep["xn4"] = ratio(ops["xn4"], ref_xn, bd_xn)
    v = cat(ref_st["o_g"])
    spread = cat([attention_spread(ref_st["q"][b], ref_st["k"][b], ref_st["v"][b]) for b in range(cfg.B)])
    gabs = np.abs(cat(ref_st["g"])) if cfg.gate_on else 1.0
    ref_og, bd_og = nvfp4_change_bound(v, M_ULP["o_g"] * bf16_ulp(v) + Z_ATT * P_ROUND * gabs * spread)
    del spread
    rep["og4"] = ratio(ops["og4"], ref_og, bd_og)
    carry_a = np.abs(gate_a) * carry(bd_og, Wd["w_o"])
    h1_g, h1_r = cat(gpu["h1"]), cat(ref_st["h1"])
    rep["h1"] = ratio(h1_g, h1_r, tol * rms(h1_r) + ulp["h1"] * np.abs(h1_r) + carry_a)
    br_r = h1_r - X
    rep["attn_branch"] = ratio(h1_g - X, br_r, tol * rms(br_r) + ulp["h1"] * (np.abs(h1_r) + np.abs(X)) + carry_a)
    hn_r = cat(ref_st["hn"])
    ref_hn, bd_hn = nvfp4_change_bound(hn_r, M_ULP["hn"] * bf16_ulp(hn_r) + norm_carry(h1_r, gamma2, carry_a, cfg.eps))
    rep["hn4"] = ratio(ops["hn4"], ref_hn, bd_hn)
    a_r, u_r = ref_hn @ Wd["w_gate"].T, ref_hn @ Wd["w_up"].T
    e_a, e_u = carry(bd_hn, Wd["w_gate"]), carry(bd_hn, Wd["w_up"])
    carry_h = 1.1 * np.abs(u_r) * e_a + np.abs(silu(a_r)) * e_u + 1.1 * e_a * e_u
    del a_r, u_r, e_a, e_u
    hm_r = cat(ref_st["hmid"])
    rep["hmid"] = ratio(cat(gpu["hmid"]), hm_r, tol * rms(hm_r) + ulp["hmid"] * np.abs(hm_r) + carry_h)
    ref_hm, bd_hm = nvfp4_change_bound(hm_r, M_ULP["hmid"] * bf16_ulp(hm_r) + carry_h)
    del carry_h
    rep["hmid4"] = ratio(ops["hmid4"], ref_hm, bd_hm)
    carry_m = np.abs(gate_m) * carry(bd_hm, Wd["w_down"])
    out_g, out_r = cat(gpu["out"]), cat(ref_st["out"])
    bound_out = tol * rms(out_r) + ulp["out"] * np.abs(out_r) + carry_m + carry_a
    rep["out"] = ratio(out_g, out_r, bound_out)
    bm_r = out_r - h1_r
    rep["mlp_branch"] = ratio(out_g - h1_g, bm_r,
                              tol * rms(bm_r) + ulp["out"] * (np.abs(out_r) + np.abs(h1_r)) + carry_m)
    out_x = cat(ref["out"])
    bound_x = bound_out + np.abs(out_r - out_x)
    rep["out_exact4"] = ratio(out_g, out_x, bound_x)
    rep["out_exact4_literal_info"] = rel_max_err([out_g], [out_x])
    rep["out_exact4_literal_bound_info"] = float(np.max(bound_x) / max(rms(out_x), 1e-300)) if out_x.size else 0.0
    for n, r_, bd in (("xn4", ref_xn, bd_xn), ("og4", ref_og, bd_og), ("hn4", ref_hn, bd_hn),
                      ("hmid4", ref_hm, bd_hm)):
        rep[n + "_movable_frac_info"] = float(np.mean(bd > 0)) if bd.size else 0.0
        rep[n + "_moved_frac_info"] = float(np.mean(ops[n] != r_)) if bd.size else 0.0
    return rep


def check4(case):
    gpu = run_gpu4(case)
    rep = report4(case, gpu)
    record({"case": case.cfg.name, "mode": "nvfp4", "report": rep})
    bad = {k: v for k, v in rep.items() if not k.endswith("_info") and v > 1.0}
    assert not bad, f"{case.cfg.name} nvfp4: parity failures {bad}; full report {rep}"
    return gpu, rep


@pytest.mark.parametrize("name", ["small_a", "small_b", "small_c", "small_imgonly", "small_txtonly"])
def test_nvfp4_small_parity(name):
    check4(di.make_case(di.CONFIGS[name]))


def test_nvfp4_without_output_gate():
    check4(di.make_case(di.CONFIGS["small_a"].replace(gate_on=False)))


def test_nvfp4_weight_casts_are_exact():
    case = di.make_case(di.CONFIGS["small_b"])
    gpu = run_gpu4(case)
    for k in MATS:
        q, sb, st = f4.quantize(case.w[k])
        codes, scales, ts = gpu["w4"][k]
        np.testing.assert_array_equal(codes, q, err_msg=k)
        np.testing.assert_array_equal(scales, sb, err_msg=k)
        assert ts == st, k


def test_nvfp4_handle_rejects_the_other_forwards():
    from diffusion_transformer_block_gb300 import KREA_DIT_ERR_INVALID_ARG, KreaDitError, krea_dit_block_forward

    cfg = di.CONFIGS["small_a"]
    case = di.make_case(cfg)
    blk = make_block(cfg.replace(dtype="nvfp4"))
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


def decode_scales_rows(sf: torch.Tensor, rows: np.ndarray, K: int) -> np.ndarray:
    """Scale atoms -> [len(rows), K/16] E4M3 values of the given global rows."""
    vals = sf.view(torch.float8_e4m3fn).to(torch.float64).cpu().numpy()
    r = np.asarray(rows)[:, None]
    b = np.arange(K // 16)[None, :]
    idx = ((r // 128) * (K // 64) + b // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + (b % 4)
    return vals[idx]


@pytest.mark.slow
def test_nvfp4_full_size_sampled():
    """The 1024px workload at full size, in the configuration the bench times (NVFP4 line),
    checked on sampled rows the oracle computes one by one: the five weight casts bit for bit
    on 256 rows of each matrix; the cast of xn within its a-priori bound and the fused
    projection's q, k, v and g within their bf16 allowance plus what that bound carries
    through the projection (and, for q and k, through the QK norm and the rotation), on 256
    token rows. Every tensor scale is the oracle's, of the whole tensor."""
    cfg = di.CONFIGS["1024px"]
    case = di.make_case(cfg)
    T, L, d, hd, B = cfg.T, cfg.L, cfg.d, cfg.hd, cfg.B
    qr, kr = cfg.n_q * hd, cfg.n_kv * hd
    rng = np.random.default_rng(11)
    rows = np.unique(np.concatenate([[0, cfg.n_txt - 1, cfg.n_txt, L - 1, L, T - 1],
                                     rng.choice(T, min(250, T), replace=False)]))
    blk = make_block(cfg.replace(dtype="nvfp4"))
    try:
        upload(blk, case)
        ms_in = oracle.mod_shared_for(case).astype(np.float32)
        ms = torch.from_numpy(ms_in).to(blk.device)
        blk.forward(case.dev["x_img"].to(blk.device).contiguous(), case.dev["x_txt"].to(blk.device).contiguous(),
                    B, cfg.img_h, cfg.img_w, cfg.n_txt, ms)
        torch.cuda.synchronize()
        rep: Dict[str, float] = {}
        # weight casts: codes, block scales and the tensor scale bit for bit
        for k in MATS:
            W = np.asarray(case.w[k], np.float64)
            R_, C_ = W.shape
            wr = np.unique(np.concatenate([[0, R_ - 1], rng.choice(R_, min(254, R_), replace=False)]))
            st = f4.tensor_scale(W)
            q_ref, sb_ref, _ = f4.quantize(W[wr], s_t=st)
            codes = blk.w4[k].view(R_, C_ // 2)[torch.from_numpy(wr).to(blk.device)]
            assert np.array_equal(decode_codes(codes, len(wr), C_), q_ref), k
            assert np.array_equal(decode_scales_rows(blk.w4["sf_" + k[2:]], wr, C_), sb_ref), k
            assert float(blk.w4["ts_" + k[2:]][0].item()) == st, k
        # the oracle's xn over every row (its tensor scale spans them all), stored as bf16
        mod = oracle.modulation(ms_in.astype(np.float64), case.w["mod_bias"])
        X = np.concatenate([np.concatenate([case.x_txt[b], case.x_img[b]], axis=0) for b in range(B)], axis=0)
        bidx = np.arange(T) // L
        xn = round_to_bf16(zero_centred_rms_norm(X, case.w["norm1_w"], cfg.eps) * (1.0 + mod["scale_a"][bidx])
                           + mod["shift_a"][bidx])
        del X
        delta = M_ULP["xn"] * bf16_ulp(xn)
        ref_x, bd_x = nvfp4_change_bound(xn[rows], delta[rows], tensor_range=magnitude_range(xn, delta),
                                         s_t=f4.tensor_scale(xn))
        del xn, delta
        codes = blk.workspace("XN4", (T * d // 2,)).view(T, d // 2)[torch.from_numpy(rows).to(blk.device)]
        ts = float(blk.workspace("TS_XN4", (1,)).double().cpu().numpy()[0])
        got_x = decode_codes(codes, len(rows), d) * np.repeat(
            decode_scales_rows(blk.workspace("SF_XN4", (((T + 127) // 128) * 128 * d // 16,)), rows, d), 16,
            axis=1) * ts
        rep["xn4"] = ratio(got_x, ref_x, bd_x)
        rep["xn4_moved_frac_info"] = float(np.mean(got_x != ref_x))
        # the fused projection on those rows, from the oracle's cast
        Wd = f4.dequantized(case.w["w_qkvg"])
        proj = ref_x @ Wd.T
        cp = carry(bd_x, Wd)
        del Wd
        tol, ulp = TOL["bf16"], 2 * UNIT_ROUNDOFF["bf16"]
        rms = lambda a: float(np.sqrt(np.mean(a * a)))  # noqa: E731
        b_, l_ = rows // L, rows % L
        ang = rope_angles(token_positions(cfg.n_txt, cfg.img_h, cfg.img_w), hd, cfg.rope_base)[l_]
        f = lambda t: t.double().cpu().numpy()  # noqa: E731
        Qd = f(blk.workspace("Q", (B, cfg.n_q, L, hd)))[b_, :, l_, :]        # [n, n_q, hd]
        Kd = f(blk.workspace("K", (B, cfg.n_kv, L, hd)))[b_, :, l_, :]
        Vd = f(blk.workspace("VT", (B, cfg.n_kv, hd, (L + 63) // 64 * 64)))[b_, :, :, l_]
        for name, lo, n_h, gain, dev in (("q", 0, cfg.n_q, case.w["q_norm_w"], Qd),
                                         ("k", qr, cfg.n_kv, case.w["k_norm_w"], Kd)):
            pre = proj[:, lo:lo + n_h * hd].reshape(-1, n_h, hd)
            ref_h = round_to_bf16(apply_rope_2d(zero_centred_rms_norm(pre, gain, cfg.eps).transpose(1, 0, 2),
                                                ang).transpose(1, 0, 2))
            dn = norm_carry(pre, 1.0 + np.asarray(gain, np.float64), cp[:, lo:lo + n_h * hd].reshape(-1, n_h, hd),
                            cfg.eps)
            drot = np.repeat(dn[..., 0::2] + dn[..., 1::2], 2, axis=-1)  # a rotated pair mixes both inputs
            rep[name] = ratio(dev, ref_h, tol * rms(ref_h) + ulp * np.abs(ref_h) + drot)
        ref_v = round_to_bf16(proj[:, qr + kr:qr + 2 * kr]).reshape(-1, cfg.n_kv, hd)
        rep["v"] = ratio(Vd, ref_v, tol * rms(ref_v) + ulp * np.abs(ref_v)
                         + cp[:, qr + kr:qr + 2 * kr].reshape(-1, cfg.n_kv, hd))
        if cfg.gate_on:
            ref_g = round_to_bf16(sigmoid(proj[:, qr + 2 * kr:2 * qr + 2 * kr]))
            Gd = f(blk.workspace("G", (B, L, qr)))[b_, l_]
            rep["g"] = ratio(Gd, ref_g, tol * rms(ref_g) + ulp * np.abs(ref_g) + 0.25 * cp[:, qr + 2 * kr:])
    finally:
        blk.close()
    record({"case": "1024px", "mode": "nvfp4", "sampled_rows": int(len(rows)), "report": rep})
    print("1024px nvfp4 (sampled): " + ", ".join(f"{k} {v:.4g}" for k, v in rep.items()))
    bad = {k: v for k, v in rep.items() if not k.endswith("_info") and v > 1.0}
    assert not bad, f"1024px nvfp4 sampled: parity failures {bad}; full report {rep}"
