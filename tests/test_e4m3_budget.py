"""CPU pins of the 8-bit parity allowances (tests/e4m3_budget.py): the bound on how far
an e4m3 cast can move must hold for every admissible perturbation (checked by brute
force against the oracle's own cast), be zero where nothing can move, and catch a
change that leaves the budget."""
import numpy as np
import pytest

from e4m3_budget import attention_spread, bf16_ulp, carry, cast_change_bound, norm_carry, nvfp4_change_bound
from oracle import gemm8 as g8
from oracle.block import round_to_bf16


def test_bf16_ulp_matches_the_bf16_grid():
    rng = np.random.default_rng(0)
    v = round_to_bf16(rng.normal(size=1000) * 10.0 ** rng.integers(-6, 6, size=1000))
    u = bf16_ulp(v)
    # v + u is the next bf16 value up (for positive v) and nothing lies strictly between
    up = np.abs(v) + u
    assert np.array_equal(round_to_bf16(up), up)
    assert np.array_equal(round_to_bf16(np.abs(v) + 0.49 * u), np.abs(v))
    assert np.array_equal(bf16_ulp(np.array([1.0, 1.5, 2.0, -3.0])), np.array([2.0 ** -7, 2.0 ** -7, 2.0 ** -6,
                                                                                2.0 ** -6]))


@pytest.mark.parametrize("per_row", [False, True])
def test_cast_bound_holds_for_every_sampled_perturbation(per_row):
    rng = np.random.default_rng(1)
    v = round_to_bf16(rng.normal(size=(16, 96)) * np.exp(rng.normal(size=(16, 1))))
    delta = 2 * bf16_ulp(v) + 1e-3
    ref, bound = cast_change_bound(v, delta, per_row)
    q, d = g8.quantize(v, per_row)
    np.testing.assert_array_equal(ref, q * d)
    for trial in range(200):
        t = rng.uniform(-1.0, 1.0, size=v.shape)
        if trial % 4 == 0:
            t = np.sign(t)  # the ends of every interval
        q2, d2 = g8.quantize(v + t * delta, per_row)
        assert np.all(np.abs(q2 * d2 - ref) <= bound)


def test_cast_bound_is_zero_far_from_boundaries_and_catches_a_larger_move():
    # values on the e4m3 grid (scale 2^0 after quantize: amax = 448 fixes k = 0) move nowhere
    # under a budget smaller than half a step, and cannot be equal under a move of a step
    grid = np.array([[448.0, 1.0, 1.125, 2.0, 3.5, 0.5]])
    ref, bound = cast_change_bound(grid, 0.01, per_row=True)
    np.testing.assert_array_equal(ref, grid)
    assert np.all(bound == 0.0)
    q2, d2 = g8.quantize(grid + np.array([[0, 0.125, 0, 0, 0, 0]]), True)
    assert np.any(np.abs(q2 * d2 - ref) > bound)  # a planted one-step change fails


def test_cast_bound_covers_a_scale_change():
    # the group's largest magnitude sits on the scale boundary 448: any larger value halves
    # the scale, which moves every element of the group to the coarser grid
    v = np.array([[448.0, 1.0 + 2.0 ** -4, 3.0 + 2.0 ** -3]])
    ref, bound = cast_change_bound(v, bf16_ulp(v), per_row=True)
    q2, d2 = g8.quantize(v + bf16_ulp(v), True)
    assert d2[0, 0] == 2 * (ref[0, 0] / g8.quantize(v, True)[0][0, 0])  # the scale changed
    assert np.all(np.abs(q2 * d2 - ref) <= bound)
    assert np.all(bound[0, 1:] > 0)


def test_cast_bound_rejects_a_group_that_could_vanish():
    with pytest.raises(ValueError):
        cast_change_bound(np.array([[1e-3, 0.0]]), 1.0, per_row=True)


def test_carry_and_norm_carry_bound_sampled_changes():
    rng = np.random.default_rng(2)
    W = rng.normal(size=(64, 128)) * 0.02
    d_op = np.abs(rng.normal(size=(8, 128))) * 1e-2
    c = carry(d_op, W)
    for _ in range(100):
        e = d_op * rng.choice([-1.0, 1.0], size=d_op.shape)
        assert np.all(np.abs(e @ W.T) <= c)
    h = rng.normal(size=(8, 128))
    gamma = 1.0 + 0.1 * rng.normal(size=(8, 128))
    dh = np.abs(rng.normal(size=h.shape)) * 1e-3
    nb = norm_carry(h, gamma, dh, 1e-6)
    f = lambda x: gamma * x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + 1e-6)  # noqa: E731
    for _ in range(100):
        e = dh * rng.uniform(-1.0, 1.0, size=h.shape)
        assert np.all(np.abs(f(h + e) - f(h)) <= nb)


def test_attention_spread_brute_force_and_one_hot():
    rng = np.random.default_rng(3)
    n_q, n_kv, L, hd = 4, 2, 7, 8
    q, k, v = rng.normal(size=(n_q, L, hd)), rng.normal(size=(n_kv, L, hd)), rng.normal(size=(n_kv, L, hd))
    got = attention_spread(q, k, v)
    for h in range(n_q):
        for j in range(L):
            s = np.array([q[h, j] @ k[h // 2, t] for t in range(L)]) / np.sqrt(hd)
            p = np.exp(s - s.max())
            p /= p.sum()
            for c in range(hd):
                want = np.sqrt(sum(p[t] ** 2 * v[h // 2, t, c] ** 2 for t in range(L)))
                assert abs(got[j, h * hd + c] - want) <= 1e-12 * max(want, 1.0)
    # a one-hot row (one key far above the rest) has spread |v| of that key
    k1 = np.zeros((1, 3, 4))
    k1[0, 1] = 200.0
    q1 = np.full((1, 3, 4), 1.0)
    v1 = rng.normal(size=(1, 3, 4))
    np.testing.assert_allclose(attention_spread(q1, k1, v1), np.abs(np.broadcast_to(v1[0, 1], (3, 4))), rtol=1e-12)


def test_nvfp4_bound_holds_for_every_sampled_perturbation():
    from oracle import nvfp4 as f4
    rng = np.random.default_rng(4)
    v = round_to_bf16(rng.normal(size=(12, 64)) * np.exp(rng.normal(size=(12, 1))))
    delta = 2 * bf16_ulp(v) + 1e-3
    ref, bound = nvfp4_change_bound(v, delta)
    np.testing.assert_array_equal(ref, f4.dequantized(v))
    for trial in range(200):
        t = rng.uniform(-1.0, 1.0, size=v.shape)
        if trial % 4 == 0:
            t = np.sign(t)
        assert np.all(np.abs(f4.dequantized(v + t * delta) - ref) <= bound + 1e-15)
    # nothing moves under a zero budget, and a change larger than the budget is caught
    _, b0 = nvfp4_change_bound(v, 0.0)
    assert np.all(b0 == 0.0)
    w = v.copy()
    w[3, 5] += 0.7 * np.abs(w[3, 5]) + 0.5
    assert np.any(np.abs(f4.dequantized(w) - ref) > bound)


def test_nvfp4_bound_with_wide_scale_ranges():
    """Budgets comparable to the values give blocks whose block scale can take many grid
    values; there the closed-form part of the bound takes over from the enumeration. It must
    still hold for every sampled perturbation and never undercut the full enumeration."""
    from oracle import nvfp4 as f4
    rng = np.random.default_rng(5)
    for scale in (0.3, 1.0, 3.0):
        v = round_to_bf16(rng.normal(size=(16, 128)) * np.exp(rng.normal(size=(16, 1))))
        delta = 2 * bf16_ulp(v) + scale * np.abs(rng.normal(size=v.shape)) * np.abs(v).mean()
        ref, bound = nvfp4_change_bound(v, delta)
        _, exact = nvfp4_change_bound(v, delta, max_exact=10 ** 6)
        assert np.all(bound >= exact - 1e-12)
        assert np.any(bound > exact + 1e-12)  # the closed form did take over somewhere
        for trial in range(200):
            t = rng.uniform(-1.0, 1.0, size=v.shape)
            if trial % 3 == 0:
                t = np.sign(t)
            assert np.all(np.abs(f4.dequantized(v + t * delta) - ref) <= bound + 1e-12)


def test_nvfp4_bound_on_sampled_rows_matches_the_whole_tensor():
    """With the whole tensor's scale and magnitude range passed in, the cast and the bound of
    sampled rows are those rows of the whole tensor's."""
    from e4m3_budget import magnitude_range
    from oracle import nvfp4 as f4
    rng = np.random.default_rng(6)
    v = round_to_bf16(rng.normal(size=(64, 128)) * np.exp(rng.normal(size=(64, 1))))
    delta = 2 * bf16_ulp(v) + 0.02 * np.abs(v)
    ref, bound = nvfp4_change_bound(v, delta)
    rows = np.array([0, 5, 17, 40, 63])
    ref_s, bound_s = nvfp4_change_bound(v[rows], delta[rows], tensor_range=magnitude_range(v, delta),
                                        s_t=f4.tensor_scale(v))
    np.testing.assert_array_equal(ref_s, ref[rows])
    np.testing.assert_array_equal(bound_s, bound[rows])
