"""Pins of the 8-bit GEMM oracle (CPU only).

The e4m3 rounding is pinned to the format's definition (every finite value built
from its bit fields, ties between neighbours) and to torch's float8_e4m3fn cast; the
scale exponent to its defining inequality; the 8-bit block to a textbook DiT block
written with torch routines whose linears cast their operands through torch's own
float8 type.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as Fn

import dit_inputs as di
import oracle
from oracle import gemm8 as g8

f64 = torch.float64


def e4m3_values():
    """Every finite e4m3 value with its mantissa field, from the bit layout: sign,
    4 exponent bits (bias 7), 3 mantissa bits; exponent field 0 is subnormal; the
    all-ones pattern S.1111.111 is NaN and there are no infinities."""
    out = []
    for s in (0, 1):
        for E in range(16):
            for M in range(8):
                if E == 15 and M == 7:
                    continue
                mag = (M / 8.0) * 2.0 ** -6 if E == 0 else (1.0 + M / 8.0) * 2.0 ** (E - 7)
                out.append(((-1.0) ** s * mag, M))
    return out


def test_every_e4m3_value_is_a_fixed_point():
    vals = np.array([v for v, _ in e4m3_values()])
    np.testing.assert_array_equal(g8.round_to_e4m3(vals), vals)
    pos = np.unique(vals[vals > 0])
    assert len(pos) == 126 and pos.max() == 448.0 and pos.min() == 2.0 ** -9


def test_e4m3_ties_go_to_the_even_mantissa_and_the_rest_to_the_nearest():
    table = sorted({(v, M) for v, M in e4m3_values() if v >= 0})
    for (a, ma), (b, mb) in zip(table, table[1:]):
        mid = 0.5 * (a + b)
        want = a if ma % 2 == 0 else b
        assert g8.round_to_e4m3(mid) == want, (a, b)
        eps = (b - a) * 1e-6
        assert g8.round_to_e4m3(mid - eps) == a and g8.round_to_e4m3(mid + eps) == b
        assert g8.round_to_e4m3(-mid) == -want


def test_e4m3_saturates_at_448():
    for v in (448.0, 449.0, 463.99, 464.0, 479.9, 480.0, 1e6, 3.0e38):
        assert g8.round_to_e4m3(v) == 448.0 and g8.round_to_e4m3(-v) == -448.0


def test_e4m3_matches_torch_float8_cast():
    rng = np.random.default_rng(5)
    mag = 2.0 ** rng.uniform(-12, math.log2(448.0), 200000)
    x = (mag * rng.choice([-1.0, 1.0], mag.size)).astype(np.float32).astype(np.float64)
    ref = torch.from_numpy(x).to(torch.float32).to(torch.float8_e4m3fn).to(f64).numpy()
    np.testing.assert_array_equal(g8.round_to_e4m3(x), ref)


def test_scale_exponent_is_the_largest_k_that_fits():
    rng = np.random.default_rng(6)
    amax = 2.0 ** rng.uniform(-100, 100, 20000)
    amax = np.concatenate([amax, [448.0, 1.0, 0.875, 449.0, 224.0, 2.0 ** -20, 3.0e38]])
    k = g8.scale_exponent(amax)
    assert np.all(np.ldexp(amax, k) <= 448.0)
    assert np.all(np.ldexp(amax, k + 1) > 448.0)
    assert list(g8.scale_exponent(np.array([448.0, 1.0, 0.875, 449.0, 0.0]))) == [0, 8, 9, -1, 0]


def test_quantize_error_and_range():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((64, 96)) * np.exp(rng.uniform(-4, 4, (64, 1)))
    for per_row in (False, True):
        q, d = g8.quantize(x, per_row)
        assert np.all(np.abs(q) <= 448.0)
        scaled = x / d  # exact: d is a power of two
        normal = np.abs(scaled) >= 2.0 ** -6
        err = np.abs(q * d - x)
        assert np.all(err[normal] <= 2.0 ** -4 * np.abs(x[normal]))
        assert np.all(err[~normal] <= 2.0 ** -10 * np.broadcast_to(d, x.shape)[~normal])
        amax = np.abs(scaled).max(axis=-1) if per_row else np.abs(scaled).max()
        assert np.all(amax > 224.0) and np.all(amax <= 448.0)
    # rows 2^20 apart: row-wise groups keep every row to 2^-4 relative error, one
    # tensor-wise group flushes the small row to zero (below half the e4m3 subnormal step)
    y = np.stack([rng.uniform(1.0, 2.0, 32), rng.uniform(1.0, 2.0, 32) * 2.0 ** -20])
    qr, dr = g8.quantize(y, True)
    assert np.all(np.abs(qr * dr - y) <= 2.0 ** -4 * y)
    qt, dt = g8.quantize(y, False)
    assert np.all(qt[1] == 0) and np.all(np.abs(qt[0] * dt - y[0]) <= 2.0 ** -4 * y[0])


# ------------------------------------------------------------ textbook 8-bit block
def _k_by_search(amax: float) -> int:
    """Scale exponent found by stepping: the largest k with amax 2^k <= 448."""
    if amax == 0:
        return 0
    k = 0
    while math.ldexp(amax, k) > 448.0:
        k -= 1
    while math.ldexp(amax, k + 1) <= 448.0:
        k += 1
    return k


def _fp8_torch(x: torch.Tensor, per_row: bool) -> torch.Tensor:
    """Dequantised e4m3 copy of x (bf16-exact values) through torch's float8 type."""
    if per_row:
        ks = [_k_by_search(float(r.abs().max())) for r in x]
        s = torch.tensor([2.0 ** k for k in ks], dtype=f64)[:, None]
    else:
        s = torch.tensor(2.0 ** _k_by_search(float(x.abs().max())), dtype=f64)
    return (x * s).to(torch.float32).to(torch.float8_e4m3fn).to(f64) / s


def _bf(x: torch.Tensor) -> torch.Tensor:
    return x.to(torch.bfloat16).to(f64)


def textbook_block8(case, ms, per_row: bool):
    """Pre-norm adaLN DiT block in torch float64 with every stored tensor rounded to
    bf16 and the four projections' operands cast through float8_e4m3fn."""
    cfg = case.cfg
    T = lambda a: torch.from_numpy(np.asarray(a, dtype=np.float64))  # noqa: E731
    w = {k: T(v) for k, v in case.w.items()}
    mod = {k: T(v) for k, v in oracle.modulation(ms, case.w["mod_bias"]).items()}
    B, L, d = cfg.B, cfg.L, cfg.d
    qr, kr = cfg.n_q * cfg.hd, cfg.n_kv * cfg.hd
    X = torch.cat([T(case.x_txt), T(case.x_img)], dim=1)  # [B, L, d]
    pos = torch.from_numpy(oracle.token_positions(cfg.n_txt, cfg.img_h, cfg.img_w))

    def rope(x):
        hd = x.shape[-1]
        D = hd // 2
        inv = cfg.rope_base ** (-2.0 * torch.arange(D // 2, dtype=f64) / D)
        ang = torch.cat([pos[:, :1].to(f64) * inv, pos[:, 1:].to(f64) * inv], dim=1)
        z = torch.view_as_complex(x.reshape(*x.shape[:-1], hd // 2, 2).contiguous())
        return torch.view_as_real(z * torch.polar(torch.ones_like(ang), ang)).reshape(x.shape)

    def lin8(a, name):  # a [B, L, K]
        a8 = _fp8_torch(a.reshape(B * L, -1), per_row)
        return Fn.linear(a8, _fp8_torch(w[name], per_row)).reshape(B, L, -1)

    def norm_mod(x, gain, shift, scale):
        y = Fn.rms_norm(x, (d,), weight=1 + gain, eps=cfg.eps)
        return _bf(y * (1 + mod[scale][:, None]) + mod[shift][:, None])

    xn = norm_mod(X, w["norm1_w"], "shift_a", "scale_a")
    p = lin8(xn, "w_qkvg")
    q = Fn.rms_norm(p[..., :qr].reshape(B, L, cfg.n_q, cfg.hd).transpose(1, 2), (cfg.hd,),
                    weight=1 + w["q_norm_w"], eps=cfg.eps)
    k = Fn.rms_norm(p[..., qr:qr + kr].reshape(B, L, cfg.n_kv, cfg.hd).transpose(1, 2), (cfg.hd,),
                    weight=1 + w["k_norm_w"], eps=cfg.eps)
    v = _bf(p[..., qr + kr:qr + 2 * kr].reshape(B, L, cfg.n_kv, cfg.hd).transpose(1, 2))
    q, k = _bf(rope(q)), _bf(rope(k))
    o = Fn.scaled_dot_product_attention(q, k, v, enable_gqa=True).transpose(1, 2).reshape(B, L, qr)
    if cfg.gate_on:
        o = o * _bf(torch.sigmoid(p[..., qr + 2 * kr:]))  # the gate is stored as its value
    o = _bf(o)
    h1 = _bf(X + mod["gate_a"][:, None] * lin8(o, "w_o"))
    hn = norm_mod(h1, w["norm2_w"], "shift_m", "scale_m")
    hmid = _bf(Fn.silu(lin8(hn, "w_gate")) * lin8(hn, "w_up"))
    out = _bf(h1 + mod["gate_m"][:, None] * lin8(hmid, "w_down"))
    return {"v": v.numpy(), "o_g": o.numpy(), "h1": h1.numpy(), "hmid": hmid.numpy(), "out": out.numpy()}


@pytest.mark.parametrize("scaling", ["tensor", "row"])
@pytest.mark.parametrize("gate_on", [True, False])
def test_block8_matches_textbook_block_with_float8_linears(scaling, gate_on):
    cfg = di.Config("pin8", B=2, img_h=3, img_w=4, n_txt=5, d=64, n_q=4, n_kv=2, hd=16, F=96, dtype="bf16",
                    seed=31, gate_on=gate_on)
    case = di.make_case(cfg, x_scale=3.0)
    # every third output channel of each projection 2^16 times smaller: far below the
    # largest weight, so tensor-wise groups push its values into the e4m3 subnormals
    # while row-wise groups keep their full precision
    for name in ("w_qkvg", "w_o", "w_gate", "w_up", "w_down"):
        case.w[name] = case.w[name].copy()
        case.w[name][::3] *= 2.0 ** -16
    ms = oracle.mod_shared_for(case) * 10.0
    got = g8.run_case8(case, scaling, mod_shared=ms, store="bf16")
    ref = textbook_block8(case, ms, scaling == "row")
    for name, r in ref.items():
        np.testing.assert_allclose(np.stack(got[name]), r, rtol=0, atol=1e-9 * np.abs(r).max(), err_msg=name)


def test_block8_scalings_differ_and_stay_near_the_bf16_block():
    """Row-wise groups follow each row's range, so the two scalings give different
    results; both stay within the e4m3 error of the unquantised block."""
    cfg = di.Config("pin8", B=2, img_h=3, img_w=4, n_txt=5, d=64, n_q=4, n_kv=2, hd=16, F=96, dtype="bf16", seed=32)
    case = di.make_case(cfg)
    ms = oracle.mod_shared_for(case) * 10.0
    base = np.stack(oracle.run_case(case, mod_shared=ms)["out"])
    t = np.stack(g8.run_case8(case, "tensor", mod_shared=ms)["out"])
    r = np.stack(g8.run_case8(case, "row", mod_shared=ms)["out"])
    assert np.max(np.abs(t - r)) > 0
    branch = np.max(np.abs(base - np.concatenate([case.x_txt, case.x_img], axis=1)))
    for o8 in (t, r):
        assert 0 < np.max(np.abs(o8 - base)) < 0.25 * branch


def test_block8_rejects_unknown_scaling():
    case = di.make_case(di.Config("pin8", B=1, img_h=2, img_w=2, n_txt=1, d=64, n_q=4, n_kv=2, hd=16, F=96,
                                  dtype="bf16", seed=1))
    with pytest.raises(ValueError):
        g8.run_case8(case, "block")


@pytest.mark.parametrize("plant", ["scale_k_plus_one", "truncating_cast", "per_row_as_tensor"])
def test_planted_mistakes_are_caught(monkeypatch, plant):
    se, q = g8.scale_exponent, g8.quantize
    if plant == "scale_k_plus_one":
        monkeypatch.setattr(g8, "scale_exponent", lambda a: se(a) + 1)
    elif plant == "truncating_cast":
        monkeypatch.setattr(g8, "round_to_e4m3", lambda v: np.copysign(
            np.minimum(np.ldexp(np.floor(np.ldexp(np.abs(v), 3 - (np.frexp(np.abs(v))[1] - 1))),
                                (np.frexp(np.abs(v))[1] - 1) - 3), 448.0), v))
    else:
        monkeypatch.setattr(g8, "quantize", lambda x, per_row: q(x, False))
    with pytest.raises(AssertionError):
        test_block8_matches_textbook_block_with_float8_linears("row", True)
