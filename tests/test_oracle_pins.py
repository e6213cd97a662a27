"""Pins of the fp64 oracle to things other than itself (CPU only).

Each test ties one oracle step to a textbook library routine, a closed form, an
invariant the mathematics fixes, or brute force on tiny inputs. The planted-
mistake tests at the end check that plausible slips in the oracle (a dropped
term, a wrong sign, a wrong index, a transposed operand) are caught.
"""
import json
import math
import os

import numpy as np
import torch
import torch.nn.functional as Fn

import dit_inputs as di
import oracle
from oracle import block as ob

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")))
f64 = torch.float64


# ---------------------------------------------------------------- closed forms
def test_golden_rms_norm():
    g = GOLD["rms_norm"]
    np.testing.assert_allclose(oracle.rms_norm(np.array(g["v"]), g["eps"]), g["expect"], rtol=1e-15)
    g = GOLD["zero_centred_gain"]
    np.testing.assert_allclose(
        oracle.zero_centred_rms_norm(np.array(g["v"]), np.array(g["w"]), g["eps"]), g["expect"], rtol=1e-15, atol=1e-300)


def test_golden_timestep_embedding():
    g = GOLD["timestep_embedding"]
    e = oracle.timestep_embedding(np.array([g["t"], 0.0]))
    for idx, val in g["expect_index"].items():
        assert abs(e[0, int(idx)] - val) < 1e-12
    np.testing.assert_array_equal(e[1, :128], 1.0)
    np.testing.assert_array_equal(e[1, 128:], 0.0)


def test_golden_rope():
    g = GOLD["rope_2d"]
    ang = oracle.rope_angles(np.array([g["pos"]]), g["hd"], 10000.0)
    out = oracle.apply_rope_2d(np.array([g["x"]]), ang)
    np.testing.assert_allclose(out[0], g["expect"], rtol=0, atol=1e-15)
    g = GOLD["rope_freq"]
    ang = oracle.rope_angles(np.array([g["pos"]]), g["hd"], 10000.0)
    assert abs(ang[0, g["pair"]] - g["expect_angle"]) < 1e-12
    # the column half is still at position 0
    np.testing.assert_array_equal(ang[0, g["hd"] // 4:], 0.0)


def test_golden_attention_and_swiglu():
    g = GOLD["attention_two_keys"]
    o = oracle.gqa_attention(np.array(g["q"]), np.array(g["k"]), np.array(g["v"]))
    assert abs(o[0, 0, 0] - g["expect"]) < 1e-14
    g = GOLD["swiglu"]
    a, b = np.array(g["a"]), np.array(g["b"])
    out = oracle.swiglu(np.diag(np.ones(2)), np.diag(a), np.diag(b))  # hn = I picks each pair
    np.testing.assert_allclose(np.diag(out), g["expect"], rtol=1e-15)


# ---------------------------------------------------------- library routines
def test_rms_norm_matches_torch():
    rng = np.random.default_rng(0)
    v = rng.standard_normal((7, 96)) * 3.0
    w = rng.standard_normal(96) * 0.1
    ref = Fn.rms_norm(torch.from_numpy(v), (96,), weight=torch.from_numpy(1.0 + w), eps=1e-6).numpy()
    np.testing.assert_allclose(oracle.zero_centred_rms_norm(v, w, 1e-6), ref, rtol=1e-13, atol=1e-13)


def test_rms_norm_scale_invariance():
    rng = np.random.default_rng(1)
    v = rng.standard_normal((5, 64))
    np.testing.assert_allclose(oracle.rms_norm(7.5 * v, 0.0), oracle.rms_norm(v, 0.0), rtol=1e-13)


def test_timestep_mlp_matches_torch():
    rng = np.random.default_rng(2)
    d = 32
    e = rng.standard_normal((3, 256))
    w1, b1 = rng.standard_normal((d, 256)) * 0.02, rng.standard_normal(d) * 0.02
    w2, b2 = rng.standard_normal((6 * d, d)) * 0.02, rng.standard_normal(6 * d) * 0.02
    T = torch.from_numpy
    ref = Fn.linear(Fn.silu(Fn.linear(T(e), T(w1), T(b1))), T(w2), T(b2)).reshape(3, 6, d).numpy()
    np.testing.assert_allclose(oracle.timestep_mlp(e, w1, b1, w2, b2), ref, rtol=1e-12, atol=1e-14)


def test_attention_matches_torch_sdpa_gqa():
    rng = np.random.default_rng(3)
    for n_q, n_kv in [(4, 2), (6, 1), (3, 3), (8, 4)]:
        q = rng.standard_normal((n_q, 19, 64))
        k = rng.standard_normal((n_kv, 23, 64))
        v = rng.standard_normal((n_kv, 23, 64))
        ref = Fn.scaled_dot_product_attention(
            torch.from_numpy(q)[None], torch.from_numpy(k)[None], torch.from_numpy(v)[None], enable_gqa=True)[0]
        np.testing.assert_allclose(oracle.gqa_attention(q, k, v), ref.numpy(), rtol=1e-11, atol=1e-12)


def test_attention_brute_force():
    """Explicit double loop with math.exp and no max-shift on a tiny input."""
    rng = np.random.default_rng(4)
    q = rng.standard_normal((2, 3, 4))
    k = rng.standard_normal((1, 5, 4))
    v = rng.standard_normal((1, 5, 4))
    o = oracle.gqa_attention(q, k, v)
    for h in range(2):
        for i in range(3):
            wts = [math.exp(sum(q[h, i, c] * k[0, j, c] for c in range(4)) / 2.0) for j in range(5)]
            z = sum(wts)
            for c in range(4):
                assert abs(o[h, i, c] - sum(wts[j] * v[0, j, c] for j in range(5)) / z) < 1e-13


def test_attention_rows_sum_to_one():
    rng = np.random.default_rng(5)
    q = rng.standard_normal((4, 11, 32)) * 4
    k = rng.standard_normal((2, 13, 32)) * 4
    ones = np.ones((2, 13, 32))
    np.testing.assert_allclose(oracle.gqa_attention(q, k, ones), 1.0, rtol=0, atol=1e-12)


def test_rope_is_complex_rotation():
    rng = np.random.default_rng(6)
    hd, L = 128, 40
    x = rng.standard_normal((3, L, hd))
    pos = np.stack([rng.integers(0, 64, L), rng.integers(0, 64, L)], 1)
    ang = oracle.rope_angles(pos, hd, 10000.0)
    out = oracle.apply_rope_2d(x, ang)
    z = (x[..., 0::2] + 1j * x[..., 1::2]) * np.exp(1j * ang)
    np.testing.assert_allclose(out[..., 0::2], z.real, atol=1e-13)
    np.testing.assert_allclose(out[..., 1::2], z.imag, atol=1e-13)
    # per-pair norm preserved
    np.testing.assert_allclose(out[..., 0::2] ** 2 + out[..., 1::2] ** 2,
                               x[..., 0::2] ** 2 + x[..., 1::2] ** 2, rtol=1e-12)


def test_rope_relative_property_and_text_identity():
    rng = np.random.default_rng(7)
    hd = 64
    q, k = rng.standard_normal(hd), rng.standard_normal(hd)

    def rot(v, r, c):
        return oracle.apply_rope_2d(v[None], oracle.rope_angles(np.array([[r, c]]), hd, 10000.0))[0]

    a = rot(q, 5, 9) @ rot(k, 2, 3)
    b = rot(q, 5 + 11, 9 + 4) @ rot(k, 2 + 11, 3 + 4)
    assert abs(a - b) < 1e-11
    # text tokens take position (0, 0): identity
    pos = oracle.token_positions(6, 3, 4)
    np.testing.assert_array_equal(pos[:6], 0)
    x = rng.standard_normal((6, hd))
    np.testing.assert_array_equal(oracle.apply_rope_2d(x, oracle.rope_angles(pos[:6], hd, 10000.0)), x)
    # row-major image order
    assert tuple(pos[6 + 1 * 4 + 3]) == (1, 3)
    # position (r, 0) leaves the column half alone, (0, c) the row half
    x = rng.standard_normal(hd)
    np.testing.assert_array_equal(rot(x, 7, 0)[hd // 2:], x[hd // 2:])
    np.testing.assert_array_equal(rot(x, 0, 7)[: hd // 2], x[: hd // 2])


# ------------------------------------------------------------ block invariants
def _small_cfg(**kw):
    base = di.Config("pin", B=2, img_h=3, img_w=4, n_txt=5, d=64, n_q=4, n_kv=2, hd=16, F=96,
                     dtype="fp32", seed=21)
    return base.replace(**kw)


def _joint(case):
    return np.concatenate([case.x_txt, case.x_img], axis=1)


def _rope_torch(x, pos, base):
    """RoPE via torch complex polar form, for the textbook block."""
    hd = x.shape[-1]
    D = hd // 2
    inv = base ** (-2.0 * torch.arange(D // 2, dtype=f64) / D)
    ang = torch.cat([pos[:, :1].to(f64) * inv, pos[:, 1:].to(f64) * inv], dim=1)
    z = torch.view_as_complex(x.reshape(*x.shape[:-1], hd // 2, 2).contiguous())
    return torch.view_as_real(z * torch.polar(torch.ones_like(ang), ang)).reshape(x.shape)


def textbook_dit_block(case, mod, *, gate_on=True):
    """Pre-norm DiT block (Peebles & Xie adaLN form: x + gate * f(norm(x)(1+scale)+shift))
    written with torch library routines only: rms_norm, linear, SDPA with GQA, silu."""
    cfg = case.cfg
    T = lambda a: torch.from_numpy(np.asarray(a, dtype=np.float64))  # noqa: E731
    X = T(_joint(case))
    w = {k: T(v) for k, v in case.w.items()}
    qr, kr = cfg.n_q * cfg.hd, cfg.n_kv * cfg.hd
    Wq, Wk, Wv = w["w_qkvg"][:qr], w["w_qkvg"][qr:qr + kr], w["w_qkvg"][qr + kr:qr + 2 * kr]
    pos = torch.from_numpy(oracle.token_positions(cfg.n_txt, cfg.img_h, cfg.img_w))
    outs = []
    for b in range(cfg.B):
        m = {k: T(v[b]) for k, v in mod.items()}
        x = X[b]
        xn = Fn.rms_norm(x, (cfg.d,), weight=1 + w["norm1_w"], eps=cfg.eps) * (1 + m["scale_a"]) + m["shift_a"]
        q = Fn.linear(xn, Wq).reshape(-1, cfg.n_q, cfg.hd).transpose(0, 1)
        k = Fn.linear(xn, Wk).reshape(-1, cfg.n_kv, cfg.hd).transpose(0, 1)
        v = Fn.linear(xn, Wv).reshape(-1, cfg.n_kv, cfg.hd).transpose(0, 1)
        q = Fn.rms_norm(q, (cfg.hd,), weight=1 + w["q_norm_w"], eps=cfg.eps)
        k = Fn.rms_norm(k, (cfg.hd,), weight=1 + w["k_norm_w"], eps=cfg.eps)
        q, k = _rope_torch(q, pos, cfg.rope_base), _rope_torch(k, pos, cfg.rope_base)
        o = Fn.scaled_dot_product_attention(q[None], k[None], v[None], enable_gqa=True)[0]
        o = o.transpose(0, 1).reshape(-1, qr)
        if gate_on:
            o = o * torch.sigmoid(Fn.linear(xn, w["w_qkvg"][qr + 2 * kr:]))
        h1 = x + m["gate_a"] * Fn.linear(o, w["w_o"])
        hn = Fn.rms_norm(h1, (cfg.d,), weight=1 + w["norm2_w"], eps=cfg.eps) * (1 + m["scale_m"]) + m["shift_m"]
        ff = Fn.linear(Fn.silu(Fn.linear(hn, w["w_gate"])) * Fn.linear(hn, w["w_up"]), w["w_down"])
        outs.append((h1 + m["gate_m"] * ff).numpy())
    return np.stack(outs)


def _mod_from_shared(case, ms):
    return oracle.modulation(ms, case.w["mod_bias"])


def _run(case, ms=None, **kw):
    return np.stack(oracle.run_case(case, mod_shared=ms, **kw)["out"])


def test_block_matches_textbook_dit_block():
    """General modulation: the oracle equals the textbook adaLN pre-norm block."""
    case = di.make_case(_small_cfg())
    ms = oracle.mod_shared_for(case) * 20.0  # make modulation matter
    ref = textbook_dit_block(case, _mod_from_shared(case, ms))
    np.testing.assert_allclose(_run(case, ms), ref, rtol=1e-11, atol=1e-11)


def test_neutral_modulation_is_plain_prenorm_block():
    """shift = scale = 0 and gate = 1 leave a plain pre-norm RMSNorm transformer block."""
    case = di.make_case(_small_cfg())
    B, d = case.cfg.B, case.cfg.d
    ms = np.zeros((B, 6, d))
    ms[:, 2] = 1.0
    ms[:, 5] = 1.0
    ms -= case.w["mod_bias"][None]
    mod = _mod_from_shared(case, ms)
    for kname in ("shift_a", "scale_a", "shift_m", "scale_m"):
        assert np.all(mod[kname] == 0.0)
    ref = textbook_dit_block(case, mod)
    np.testing.assert_allclose(_run(case, ms), ref, rtol=1e-11, atol=1e-11)


def test_zero_modulation_is_identity():
    case = di.make_case(_small_cfg())
    ms = -np.broadcast_to(case.w["mod_bias"], (case.cfg.B, 6, case.cfg.d)).copy()
    np.testing.assert_array_equal(_run(case, ms), _joint(case))


def test_zero_gate_weights_halve_attention_branch():
    cfg = _small_cfg()
    case = di.make_case(cfg)
    ms = oracle.mod_shared_for(case)
    qr, kr = cfg.n_q * cfg.hd, cfg.n_kv * cfg.hd
    case.w["w_qkvg"] = case.w["w_qkvg"].copy()
    case.w["w_qkvg"][qr + 2 * kr:] = 0.0
    X = _joint(case)
    gated = np.stack(oracle.run_case(case, mod_shared=ms)["h1"]) - X
    case_off = di.make_case(cfg.replace(gate_on=False))
    case_off.w = dict(case.w)
    case_off.w["w_qkvg"] = case.w["w_qkvg"][: qr + 2 * kr]
    case_off.x_txt, case_off.x_img = case.x_txt, case.x_img
    ungated = np.stack(oracle.run_case(case_off, mod_shared=ms)["h1"]) - X
    np.testing.assert_allclose(gated, 0.5 * ungated, rtol=1e-12, atol=1e-15)


def test_gqa_with_tiled_kv_equals_mha():
    cfg = _small_cfg(n_q=4, n_kv=2)
    case = di.make_case(cfg)
    ms = oracle.mod_shared_for(case)
    out_gqa = _run(case, ms)
    # MHA: every query head gets its own copy of its group's K/V projection
    hd, G = cfg.hd, cfg.n_q // cfg.n_kv
    qr, kr = cfg.n_q * hd, cfg.n_kv * hd
    W = case.w["w_qkvg"]
    Wk = W[qr:qr + kr].reshape(cfg.n_kv, hd, -1)
    Wv = W[qr + kr:qr + 2 * kr].reshape(cfg.n_kv, hd, -1)
    Wk4 = np.repeat(Wk, G, axis=0).reshape(cfg.n_q * hd, -1)
    Wv4 = np.repeat(Wv, G, axis=0).reshape(cfg.n_q * hd, -1)
    case_mha = di.make_case(cfg.replace(n_kv=cfg.n_q))
    case_mha.w = dict(case.w)
    case_mha.w["w_qkvg"] = np.concatenate([W[:qr], Wk4, Wv4, W[qr + 2 * kr:]], axis=0)
    case_mha.x_txt, case_mha.x_img = case.x_txt, case.x_img
    np.testing.assert_allclose(_run(case_mha, ms), out_gqa, rtol=0, atol=1e-14)


def test_permutation_equivariance_without_rope():
    cfg = _small_cfg(n_txt=0, img_h=1, img_w=17)
    case = di.make_case(cfg)
    ms = oracle.mod_shared_for(case)
    perm = np.random.default_rng(8).permutation(17)
    out = _run(case, ms, rope_on=False)
    case.x_img = case.x_img[:, perm]
    out_p = _run(case, ms, rope_on=False)
    np.testing.assert_allclose(out_p, out[:, perm], rtol=0, atol=1e-13)


def test_text_image_order_does_not_matter():
    """With text at RoPE index 0, putting text after the image gives the same
    per-token outputs (the textbook block takes explicit positions)."""
    case = di.make_case(_small_cfg())
    ms = oracle.mod_shared_for(case)
    out = _run(case, ms)
    cfg = case.cfg
    # swap: feed the image tokens as the "text" slot is impossible (they need positions), so
    # check through the torch block with the joint sequence reversed in order.
    mod = _mod_from_shared(case, ms)
    X = _joint(case)
    Nt = cfg.n_txt
    order = np.r_[np.arange(Nt, cfg.L), np.arange(Nt)]
    pos = oracle.token_positions(Nt, cfg.img_h, cfg.img_w)[order]

    saved = oracle.token_positions
    import oracle.block as blk
    try:
        blk.token_positions = lambda *a: pos
        case2 = di.make_case(cfg.replace(n_txt=0, img_h=1, img_w=cfg.L))
        case2.w = case.w
        case2.x_txt = case.x_txt[:, :0]
        case2.x_img = X[:, order]
        out2 = _run(case2, ms)
    finally:
        blk.token_positions = saved
    np.testing.assert_allclose(out2, out[:, order], rtol=0, atol=1e-13)
    del mod


def test_zero_swiglu_gate_leaves_residual():
    case = di.make_case(_small_cfg())
    case.w["w_gate"] = np.zeros_like(case.w["w_gate"])
    r = oracle.run_case(case)
    np.testing.assert_array_equal(np.stack(r["out"]), np.stack(r["h1"]))


def test_row_sampled_mode_is_exact():
    cfg = _small_cfg(B=2, img_h=6, img_w=5, n_txt=7)
    case = di.make_case(cfg)
    full = oracle.run_case(case)
    rows = di.sample_rows(cfg, 9, seed=3)
    part = oracle.run_case(case, rows=rows)
    for b in range(cfg.B):
        for key in ("out", "h1", "o_g", "hmid"):
            np.testing.assert_allclose(part[key][b], full[key][b][rows[b]], rtol=0, atol=1e-14)
        np.testing.assert_allclose(part["q"][b], full["q"][b][:, rows[b]], rtol=0, atol=1e-14)


def test_seeded_inputs_are_deterministic_and_rounded():
    c1 = di.make_case(di.CONFIGS["small_a"])
    c2 = di.make_case(di.CONFIGS["small_a"])
    np.testing.assert_array_equal(c1.w["w_qkvg"], c2.w["w_qkvg"])
    # bf16 rounding: re-rounding changes nothing
    r = torch.from_numpy(c1.w["w_o"]).to(torch.bfloat16).to(f64).numpy()
    np.testing.assert_array_equal(r, c1.w["w_o"])
    assert c1.w["w_qkvg"].shape == ((2 * 4 + 2 * 2) * 128, 512)


# --------------------------------------------------------- planted mistakes
def _pins_catch(monkeypatch, name, bad):
    """Plant ``bad`` in place of oracle.block.<name> and check that the textbook
    comparison (the broadest pin) now fails."""
    monkeypatch.setattr(ob, name, bad)
    case = di.make_case(_small_cfg())
    ms = oracle.mod_shared_for(case) * 20.0
    ref = textbook_dit_block(case, _mod_from_shared(case, ms))
    got = _run(case, ms)
    assert not np.allclose(got, ref, rtol=1e-9, atol=1e-9), f"planted mistake in {name} went unseen"


def test_planted_rope_sign_is_caught(monkeypatch):
    orig = ob.apply_rope_2d
    _pins_catch(monkeypatch, "apply_rope_2d", lambda x, angles: orig(x, -angles))


def test_planted_gain_without_one_is_caught(monkeypatch):
    _pins_catch(monkeypatch, "zero_centred_rms_norm",
                lambda v, w, eps: ob.rms_norm(v, eps) * np.asarray(w))


def test_planted_gqa_index_is_caught(monkeypatch):
    orig = ob.gqa_attention

    def bad(q, k, v):  # interleaved groups instead of contiguous ones
        n_q, n_kv = q.shape[0], k.shape[0]
        idx = np.arange(n_q) % n_kv
        return orig(q, k[idx], v[idx])
    _pins_catch(monkeypatch, "gqa_attention", bad)


def test_planted_transposed_swiglu_is_caught(monkeypatch):
    _pins_catch(monkeypatch, "swiglu",
                lambda hn, wg, wu: ob.silu(hn @ np.asarray(wu).T) * (hn @ np.asarray(wg).T))


def test_planted_mod_order_is_caught(monkeypatch):
    orig = ob.modulation

    def bad(ms, bias):
        m = orig(ms, bias)
        m["shift_a"], m["scale_a"] = m["scale_a"], m["shift_a"]
        return m
    _pins_catch(monkeypatch, "modulation", bad)


def test_planted_timestep_layout_is_caught():
    """[sin | cos] instead of [cos | sin] breaks the t = 0 closed form."""
    e = oracle.timestep_embedding(np.array([0.0]))
    assert e[0, 0] == 1.0 and e[0, 128] == 0.0
    swapped = np.concatenate([e[:, 128:], e[:, :128]], axis=1)
    assert swapped[0, 0] != 1.0


# ------------------------------------------------------------- storage rounding
def test_round_to_bf16_matches_torch_on_float32_values():
    rng = np.random.default_rng(9)
    x = (rng.standard_normal(100000) * np.exp(rng.uniform(-20, 20, 100000))).astype(np.float32).astype(np.float64)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(oracle.round_to_bf16(x), ref)


def test_round_to_bf16_ties_to_even():
    e = 2.0 ** -8
    cases = {1.0 + e: 1.0, 1.0 + 3 * e: 1.0 + 4 * e, -(1.0 + e): -1.0, 0.0: 0.0, 1.0 + 1.5 * e: 1.0 + 2 * e,
             3.0: 3.0, 1.0 - e / 2: 1.0, 1.0 - e: 1.0 - e}
    for x, want in cases.items():
        assert oracle.round_to_bf16(np.array([x]))[0] == want, x


def test_storage_rounded_oracle_stores_representable_values():
    case = di.make_case(_small_cfg(dtype="bf16"))
    r = oracle.run_case(case, store="bf16")
    for key in ("q", "k", "v", "g", "o_g", "h1", "hn", "hmid", "out"):
        a = np.concatenate([x.reshape(-1) for x in r[key]])
        np.testing.assert_array_equal(oracle.round_to_bf16(a), a)
    exact = oracle.run_case(case)
    err = np.abs(np.stack(r["out"]) - np.stack(exact["out"])).max()
    assert 0 < err < 0.05


# --------------------------------------------------------------- stacks of blocks
def _textbook_stack(cfg, blocks, ms, x_joint, *, text_first=True):
    """Textbook blocks applied in turn; ``text_first=False`` plants a chain that hands the
    next block its image rows as if they were the text rows."""
    import types
    X = x_joint
    Nt = cfg.n_txt
    for c in blocks:
        if text_first:
            xt, xi = X[:, :Nt], X[:, Nt:]
        else:
            xt, xi = X[:, -Nt:], X[:, :-Nt]
        step = types.SimpleNamespace(cfg=cfg, w=c.w, x_txt=xt, x_img=xi)
        X = textbook_dit_block(step, _mod_from_shared(c, ms), gate_on=cfg.gate_on)
    return X


def test_stack_matches_textbook_blocks_in_turn():
    """A stack is the blocks composed in order, each with its own weights and mod_bias on
    the shared modulation, on the joint sequence with text rows first."""
    blocks = di.make_stack(_small_cfg(), 3)
    case = blocks[0]
    ms = oracle.mod_shared_for(case) * 20.0
    got = oracle.run_stack(case, [c.w for c in blocks], mod_shared=ms)
    ref = _textbook_stack(case.cfg, blocks, ms, _joint(case))
    np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-11)
    # the blocks differ, so a chain that reorders or reuses them would not match
    assert np.max(np.abs(got - _textbook_stack(case.cfg, blocks[::-1], ms, _joint(case)))) > 1e-6
    # a chain that swaps the text and image rows between blocks would not match either
    bad = _textbook_stack(case.cfg, blocks, ms, _joint(case), text_first=False)
    assert np.max(np.abs(got - bad)) > 1e-6


def test_stack_skips_a_zero_gate_block_exactly():
    """A block whose gates are zero passes the sequence through unchanged, so inserting it
    anywhere in a stack changes nothing, bit for bit."""
    blocks = di.make_stack(_small_cfg(B=1), 3)
    case = blocks[0]
    ms = oracle.mod_shared_for(case)
    zero = dict(blocks[1].w)
    zero["mod_bias"] = zero["mod_bias"].copy()
    zero["mod_bias"][2] = -ms[0, 2]
    zero["mod_bias"][5] = -ms[0, 5]
    a, c = blocks[0].w, blocks[2].w
    np.testing.assert_array_equal(oracle.run_stack(case, [a, zero, c], mod_shared=ms),
                                  oracle.run_stack(case, [a, c], mod_shared=ms))
    np.testing.assert_array_equal(oracle.run_stack(case, [zero], mod_shared=ms), _joint(case))


def test_stack_of_one_is_the_block_and_storage_rounds_every_output():
    blocks = di.make_stack(_small_cfg(dtype="bf16"), 2)
    case = blocks[0]
    ms = oracle.mod_shared_for(case)
    one = oracle.run_stack(case, [case.w], mod_shared=ms)
    np.testing.assert_array_equal(one, np.stack(oracle.run_case(case, mod_shared=ms)["out"]))
    st = oracle.run_stack(case, [c.w for c in blocks], mod_shared=ms, store="bf16")
    np.testing.assert_array_equal(st, ob.round_to_bf16(st))
