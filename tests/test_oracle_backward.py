"""Pins of the backward oracle (CPU only).

The analytic gradients of ``oracle.backward`` are checked against (1) torch autograd
through a textbook DiT block written with torch routines in float64 (rms_norm, linear,
SDPA with GQA, complex-rotation RoPE, sigmoid, silu), and (2) central finite differences
of the forward oracle ``oracle.block_forward`` along random directions. Planted mistakes
(a dropped term of the RMSNorm gradient, a RoPE rotation of the wrong sense, a SwiGLU
derivative without its product term, attention gradients that drop all but one query
head of each KV group) are shown to fail.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as Fn

import dit_inputs as di
import oracle
from oracle import backward as ob

f64 = torch.float64
WEIGHTS = ("w_qkvg", "w_o", "w_gate", "w_up", "w_down", "norm1_w", "norm2_w", "q_norm_w", "k_norm_w", "mod_bias")


def _cfg(**kw):
    base = di.Config("bwd", B=2, img_h=3, img_w=4, n_txt=5, d=64, n_q=4, n_kv=2, hd=16, F=96, dtype="fp32",
                     seed=41)
    return base.replace(**kw)


def torch_block(cfg, X, ms, w):
    """Textbook adaLN pre-norm block in torch float64: X [B, L, d], ms [B, 6, d]."""
    B, L, d = X.shape
    qr, kr = cfg.n_q * cfg.hd, cfg.n_kv * cfg.hd
    mod = ms + w["mod_bias"][None]
    sh_a, sc_a, g_a, sh_m, sc_m, g_m = (mod[:, i, None, :] for i in range(6))
    pos = torch.from_numpy(oracle.token_positions(cfg.n_txt, cfg.img_h, cfg.img_w))
    D = cfg.hd // 2
    inv = cfg.rope_base ** (-2.0 * torch.arange(D // 2, dtype=f64) / D)
    ang = torch.cat([pos[:, :1].to(f64) * inv, pos[:, 1:].to(f64) * inv], dim=1)
    rot = torch.polar(torch.ones_like(ang), ang)

    def rope(x):
        z = torch.view_as_complex(x.reshape(*x.shape[:-1], cfg.hd // 2, 2).contiguous())
        return torch.view_as_real(z * rot).reshape(x.shape)

    xn = Fn.rms_norm(X, (d,), weight=1 + w["norm1_w"], eps=cfg.eps) * (1 + sc_a) + sh_a
    P = Fn.linear(xn, w["w_qkvg"])
    q = P[..., :qr].reshape(B, L, cfg.n_q, cfg.hd).transpose(1, 2)
    k = P[..., qr:qr + kr].reshape(B, L, cfg.n_kv, cfg.hd).transpose(1, 2)
    v = P[..., qr + kr:qr + 2 * kr].reshape(B, L, cfg.n_kv, cfg.hd).transpose(1, 2)
    q = rope(Fn.rms_norm(q, (cfg.hd,), weight=1 + w["q_norm_w"], eps=cfg.eps))
    k = rope(Fn.rms_norm(k, (cfg.hd,), weight=1 + w["k_norm_w"], eps=cfg.eps))
    o = Fn.scaled_dot_product_attention(q, k, v, enable_gqa=True).transpose(1, 2).reshape(B, L, qr)
    if cfg.gate_on:
        o = o * torch.sigmoid(P[..., qr + 2 * kr:])
    h1 = X + g_a * Fn.linear(o, w["w_o"])
    hn = Fn.rms_norm(h1, (d,), weight=1 + w["norm2_w"], eps=cfg.eps) * (1 + sc_m) + sh_m
    return h1 + g_m * Fn.linear(Fn.silu(Fn.linear(hn, w["w_gate"])) * Fn.linear(hn, w["w_up"]), w["w_down"])


def autograd_grads(case, ms, dout):
    cfg = case.cfg
    T = lambda a: torch.tensor(np.asarray(a, dtype=np.float64), requires_grad=True)  # noqa: E731
    X = T(np.concatenate([case.x_txt, case.x_img], axis=1))
    msT = T(ms)
    w = {k: T(case.w[k]) for k in WEIGHTS}
    out = torch_block(cfg, X, msT, w)
    (out * torch.from_numpy(dout)).sum().backward()
    g = {"d_" + k: w[k].grad.numpy() for k in WEIGHTS}
    Xg = X.grad.numpy()
    g["d_x_txt"], g["d_x_img"] = Xg[:, :cfg.n_txt], Xg[:, cfg.n_txt:]
    g["d_mod_shared"] = msT.grad.numpy()
    return g


def _case(cfg, seed=3):
    case = di.make_case(cfg, qk_gain=0.3)
    ms = oracle.mod_shared_for(case) * 10.0  # make the modulation matter
    dout = np.random.default_rng(seed).standard_normal((cfg.B, cfg.L, cfg.d))
    return case, ms, dout


def _compare(got, ref, rtol=1e-9):
    for k, r in ref.items():
        g = np.asarray(got[k])
        assert g.shape == np.shape(r), k
        if g.size == 0:
            continue
        scale = max(np.max(np.abs(r)), 1e-300)
        np.testing.assert_allclose(g, r, rtol=0, atol=rtol * scale, err_msg=k)


@pytest.mark.parametrize("gate_on", [True, False])
@pytest.mark.parametrize("n_kv", [4, 2, 1])
def test_backward_matches_torch_autograd(gate_on, n_kv):
    cfg = _cfg(gate_on=gate_on, n_kv=n_kv)
    case, ms, dout = _case(cfg)
    got = ob.run_case_backward(case, dout, mod_shared=ms)
    _compare(got, autograd_grads(case, ms, dout))


def test_backward_text_only_and_image_only():
    for kw in (dict(img_h=0, img_w=0, n_txt=9), dict(n_txt=0)):
        cfg = _cfg(**kw)
        case, ms, dout = _case(cfg)
        _compare(ob.run_case_backward(case, dout, mod_shared=ms), autograd_grads(case, ms, dout))


def test_backward_matches_finite_differences():
    """<grad, delta> against (f(p + e delta) - f(p - e delta)) / 2e, f = <out, dout> from the
    forward oracle, for the input, every weight and the modulation."""
    cfg = _cfg(B=1, img_h=2, img_w=3, n_txt=2, d=32, n_q=2, n_kv=1, hd=16, F=48)
    case, ms, dout = _case(cfg)
    g = ob.run_case_backward(case, dout, mod_shared=ms)
    rng = np.random.default_rng(9)

    def f(case_, ms_):
        return float(np.sum(np.stack(oracle.run_case(case_, mod_shared=ms_)["out"]) * dout))

    eps = 1e-6
    targets = ["x_txt", "x_img", "mod_shared"] + list(WEIGHTS)
    for name in targets:
        if name == "mod_shared":
            base = ms
        elif name in ("x_txt", "x_img"):
            base = getattr(case, name)
        else:
            base = case.w[name]
        delta = rng.standard_normal(base.shape)

        def shifted(sign):
            c = di.make_case(cfg, qk_gain=0.3)
            m = ms
            if name == "mod_shared":
                m = ms + sign * eps * delta
            elif name in ("x_txt", "x_img"):
                setattr(c, name, base + sign * eps * delta)
            else:
                c.w[name] = base + sign * eps * delta
            return f(c, m)

        fd = (shifted(1.0) - shifted(-1.0)) / (2 * eps)
        an = float(np.sum(g["d_" + name] * delta))
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, fd, an)


@pytest.mark.parametrize("plant", ["rms_no_second_term", "rope_wrong_sense", "silu_grad_no_product",
                                   "kv_grad_not_summed"])
def test_planted_mistakes_are_caught(monkeypatch, plant):
    if plant == "rms_no_second_term":
        monkeypatch.setattr(ob, "rms_backward", lambda x, r, dy: r * dy)
    elif plant == "rope_wrong_sense":
        monkeypatch.setattr(ob, "rope_backward", lambda dy, ang: oracle.apply_rope_2d(dy, ang))
    elif plant == "silu_grad_no_product":
        monkeypatch.setattr(ob, "silu_grad", lambda a: oracle.block.sigmoid(a))
    else:
        orig = ob.element_backward

        def last_head_only(s, dout, mod, w, *, n_q, n_kv, hd, gate_on):
            # attention gradients from only the last query head of each KV group
            G = n_q // n_kv
            s2 = dict(s)
            A = s["A"].copy()
            for h in range(n_q):
                if h % G != G - 1:
                    A[h] = 0.0
            s2["A"] = A
            return orig(s2, dout, mod, w, n_q=n_q, n_kv=n_kv, hd=hd, gate_on=gate_on)

        monkeypatch.setattr(ob, "element_backward", last_head_only)
    cfg = _cfg()
    case, ms, dout = _case(cfg)
    with pytest.raises(AssertionError):
        _compare(ob.run_case_backward(case, dout, mod_shared=ms), autograd_grads(case, ms, dout))


def test_rms_and_rope_backward_are_the_transposed_jacobians():
    """Closed forms: <J dx, dy> = <dx, J^T dy> for the RMSNorm and the rotation."""
    rng = np.random.default_rng(2)
    x = rng.standard_normal((5, 16))
    r = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + 1e-6)
    dx, dy = rng.standard_normal((2, 5, 16))
    h = 1e-7
    y = lambda z: z / np.sqrt(np.mean(z * z, axis=-1, keepdims=True) + 1e-6)  # noqa: E731
    jdx = (y(x + h * dx) - y(x - h * dx)) / (2 * h)
    assert math.isclose(np.sum(jdx * dy), np.sum(dx * ob.rms_backward(x, r, dy)), rel_tol=1e-6)
    ang = rng.uniform(-3, 3, (5, 8))
    a = oracle.apply_rope_2d(dx, ang)
    assert math.isclose(np.sum(a * dy), np.sum(dx * ob.rope_backward(dy, ang)), rel_tol=1e-12)
