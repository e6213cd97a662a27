"""CPU pins of the NVFP4 oracle (oracle/nvfp4.py): the E2M1 grid and its rounding
against brute force, the two-level scales against their defining inequalities, the
cast's invariances, planted mistakes that the pins must catch, and the block forward's
plumbing of the cast."""
import itertools

import numpy as np
import pytest

import dit_inputs as di
import oracle
from oracle import gemm8 as g8
from oracle import nvfp4 as f4
from oracle.block import round_to_bf16

# the sixteen E2M1 codes (sign | exponent(2) | mantissa(1)), decoded from the bit layout:
# exponent 0 is subnormal (0.5 * mantissa), else 2^(e - 1) * (1 + mantissa / 2)
E2M1_DECODED = np.array([(-1.0 if c & 8 else 1.0) * ((0.5 * (c & 1)) if ((c >> 1) & 3) == 0
                                                     else 2.0 ** (((c >> 1) & 3) - 1) * (1 + 0.5 * (c & 1)))
                         for c in range(16)])


def brute_e2m1(x):
    """Nearest code by exhaustive search; ties to the code with mantissa bit 0."""
    out = []
    for v in np.ravel(x):
        v = min(max(v, -6.0), 6.0)
        d = np.abs(E2M1_DECODED - v)
        best = np.flatnonzero(d == d.min())
        even = [c for c in best if c % 2 == 0]
        c = (even or list(best))[0]
        out.append(E2M1_DECODED[c])
    return np.array(out).reshape(np.shape(x))


def test_grid_is_the_decoded_bit_layout():
    assert sorted(set(np.abs(E2M1_DECODED))) == sorted(f4.E2M1_VALUES.tolist())
    np.testing.assert_array_equal(f4.round_to_e2m1(E2M1_DECODED), E2M1_DECODED)


def test_rounding_matches_brute_force_on_every_bf16_value_in_range():
    # every bf16 value in [-8, 8] (ties included: 0.25, 0.75, ..., 5 are bf16 values)
    mags = np.unique(round_to_bf16(np.concatenate([np.linspace(0, 8, 20001), 2.0 ** -np.arange(0, 40, 0.25)])))
    x = np.concatenate([mags, -mags])
    np.testing.assert_array_equal(f4.round_to_e2m1(x), brute_e2m1(x))


def test_rounding_closed_forms():
    x = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0, 100.0, -0.26, -5.1, 0.0])
    want = np.array([0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, 6.0, 6.0, -0.5, -6.0, 0.0])
    np.testing.assert_array_equal(f4.round_to_e2m1(x), want)


def test_tensor_scale_is_the_smallest_fitting_power_of_two():
    for amax in (1.0, 2688.0, 2689.0, 2688.0 * 2 ** -5, 3.0, 1e-3, 4.75):
        st = f4.tensor_scale(np.array([[amax, -0.5 * amax]]))
        assert st == 2.0 ** np.round(np.log2(st))
        assert amax <= 2688.0 * st and amax > 2688.0 * st / 2
    assert f4.tensor_scale(np.zeros((2, 16))) == 1.0


def test_block_scales_and_codes_satisfy_their_definitions():
    rng = np.random.default_rng(0)
    x = round_to_bf16(rng.normal(size=(8, 64)) * np.exp(rng.normal(size=(8, 1)) * 2))
    q, sb, st = f4.quantize(x)
    blocks = x.reshape(8, 4, 16)
    amax_b = np.abs(blocks).max(-1)
    np.testing.assert_array_equal(sb, g8.round_to_e4m3(amax_b / (6 * st)))
    assert np.all(sb <= 448)
    # each code is the nearest E2M1 value of x / (s_b s_t)
    np.testing.assert_array_equal(q.reshape(8, 4, 16), brute_e2m1(blocks / (sb[..., None] * st)))
    # reconstruction within half a spacing of the scaled grid (or the saturation gap)
    xh = q * np.repeat(sb, 16, axis=-1) * st
    scaled = np.abs(x) / (np.repeat(sb, 16, axis=-1) * st)
    half = np.where(scaled < 2, 0.25, np.where(scaled < 4, 0.5, 1.0))
    err = np.abs(x - xh) / (np.repeat(sb, 16, axis=-1) * st)
    assert np.all(err <= np.maximum(half, scaled - 6.0) + 1e-12)


def test_blocks_are_independent_and_scale_invariant():
    rng = np.random.default_rng(1)
    x = round_to_bf16(rng.normal(size=(4, 64)))
    xh = f4.dequantized(x)
    # a power-of-two multiple of the tensor moves s_t alone: the cast scales exactly
    np.testing.assert_array_equal(f4.dequantized(x * 8.0), xh * 8.0)
    # changing one block (without touching the tensor's amax) leaves every other block's cast
    y = x.copy()
    y[0, 16:32] *= 0.5
    yh = f4.dequantized(y)
    keep = np.ones_like(x, bool)
    keep[0, 16:32] = False
    np.testing.assert_array_equal(yh[keep], xh[keep])


def test_planted_mistakes_are_caught():
    rng = np.random.default_rng(2)
    x = round_to_bf16(rng.normal(size=(4, 64)))
    mags = np.unique(round_to_bf16(np.linspace(0, 6, 2001)))
    # a truncating E2M1 cast
    trunc = np.floor(mags / np.where(mags < 2, 0.5, np.where(mags < 4, 1.0, 2.0))) * np.where(
        mags < 2, 0.5, np.where(mags < 4, 1.0, 2.0))
    assert not np.array_equal(trunc, brute_e2m1(mags))
    # blocks of 32 instead of 16: a block's cast then depends on its neighbour
    def q32(v):
        b = v.reshape(v.shape[0], -1, 32)
        st = f4.tensor_scale(v)
        sb = g8.round_to_e4m3(np.abs(b).max(-1) / (6 * st))
        return (f4.round_to_e2m1(b / (sb[..., None] * st)) * sb[..., None] * st).reshape(v.shape)
    z = x.copy()
    z[0, :32] = round_to_bf16(rng.uniform(-0.1, 0.1, size=32))  # two quiet blocks
    z[1, 0] = 3.0  # the tensor's amax sits elsewhere
    y = z.copy()
    y[0, 16:32] = 1.0  # a louder second block, still below the tensor's amax
    keep = np.ones_like(z, bool)
    keep[0, 16:32] = False
    np.testing.assert_array_equal(f4.dequantized(y)[keep], f4.dequantized(z)[keep])  # 16: untouched
    assert not np.array_equal(q32(y)[keep], q32(z)[keep])  # 32: the first block moves
    # no tensor scale (s_t = 1): large tensors saturate their block scales
    big = x * 1e4
    sb_plain = g8.round_to_e4m3(np.abs(big.reshape(4, 4, 16)).max(-1) / 6)
    assert np.any(sb_plain >= 448) and np.all(f4.quantize(big)[1] < 448)


def test_block_forward4_with_an_exact_cast_is_the_plain_block():
    """The cast plumbing: with the cast replaced by the identity, the quantised block is
    the plain block (so block_forward4 differs from it by the NVFP4 cast alone)."""
    case = di.make_case(di.CONFIGS["small_a"])
    cfg = case.cfg
    ms = oracle.mod_shared_for(case)
    ref = oracle.run_case(case, mod_shared=ms)
    got = g8.block_forward8(case.x_txt, case.x_img, (cfg.img_h, cfg.img_w), ms, case.w, scaling="tensor",
                            n_q=cfg.n_q, n_kv=cfg.n_kv, hd=cfg.hd, eps=cfg.eps, rope_base=cfg.rope_base,
                            gate_on=cfg.gate_on, deq=lambda a: np.asarray(a, np.float64))
    for b in range(cfg.B):
        np.testing.assert_allclose(got["out"][b], ref["out"][b], rtol=0, atol=1e-12)
    r4 = f4.run_case4(case, mod_shared=ms)
    # the NVFP4 block stays near the plain one (4-bit operands: a few percent)
    o4, o = np.stack(r4["out"]), np.stack(ref["out"])
    rel = np.sqrt(np.mean((o4 - o) ** 2) / np.mean((o - np.stack([np.concatenate([case.x_txt[b], case.x_img[b]])
                                                                    for b in range(cfg.B)])) ** 2))
    assert 0 < rel < 0.5


@pytest.mark.parametrize("shape", list(itertools.product((1, 3), (16, 48))))
def test_operands_decode_exactly(shape):
    rng = np.random.default_rng(sum(shape))
    x = round_to_bf16(rng.normal(size=shape) * 3)
    q, sb, st = f4.quantize(x)
    assert set(np.unique(np.abs(q))) <= set(f4.E2M1_VALUES.tolist())
    np.testing.assert_array_equal(g8.round_to_e4m3(sb), sb)
