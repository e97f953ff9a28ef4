"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test checks one oracle function against hand-written fixtures
(tests/golden/), closed forms, exact rational brute force, library routines
that reduce to the same special case, or invariants of the definition.  The
cases are chosen so that a plausible slip (wrong bit order, wrong sign of the
derived bias, fma instead of select, dropped bias term, transposed operand)
fails at least one of them.
"""
import math
import os
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import q1_oracle as O
from bit_affine_quantized_g128_gb300 import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLD, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            yield [c.strip() for c in line.split("|")]


def _f16(h):
    return np.frombuffer(struct.pack("<H", h), dtype=np.float16)[0]


def _bits32(v):
    return struct.unpack("<I", np.float32(v).tobytes())[0]


# ---------------------------------------------------------------- packing
def test_unpack_golden_lsb_first():
    for K, words, idx in _rows("unpack_lsb_first.txt"):
        K = int(K)
        w = np.array([[int(h, 16) for h in words.split()]], dtype=np.uint32)
        want = set(int(i) for i in idx.split())
        got = O.unpack(w, K)[0]
        assert set(np.nonzero(got)[0].tolist()) == want, (words, idx)
        assert got.dtype == np.uint8 and set(np.unique(got)) <= {0, 1}


def test_pack_golden_lsb_first():
    for K, words, idx in _rows("unpack_lsb_first.txt"):
        K = int(K)
        bits = np.zeros((1, K), dtype=np.uint8)
        for i in idx.split():
            bits[0, int(i)] = 1
        want = np.array([[int(h, 16) for h in words.split()]], dtype=np.uint32)
        np.testing.assert_array_equal(O.pack(bits), want)


def test_pack_matches_numpy_packbits_little():
    # LSB-first packing of 32 bits into a little-endian uint32 is what
    # numpy.packbits(bitorder='little') followed by a little-endian uint32 view
    # computes; an independent library routine for the same layout.
    bits = synth.bits(7, 256, seed=11)
    lib = np.packbits(bits, axis=1, bitorder="little").view("<u4")
    np.testing.assert_array_equal(O.pack(bits), lib)


def test_pack_unpack_roundtrip_both_directions():
    w = synth.weight_words(9, 384, seed=5)
    np.testing.assert_array_equal(O.pack(O.unpack(w, 384)), w)
    b = synth.bits(9, 384, seed=6)
    np.testing.assert_array_equal(O.unpack(O.pack(b), 384), b)


# ---------------------------------------------------------------- dequant
def test_dequant_golden_values():
    for sh, bh, q, f32h, bf16h, f16h, _note in _rows("dequant_values.txt"):
        s = np.array([[_f16(int(sh, 16))]], dtype=np.float16)
        b = None if bh == "sym" else np.array([[_f16(int(bh, 16))]], dtype=np.float16)
        K = 128
        word = 0xFFFFFFFF if int(q) else 0
        w = np.full((1, K // 32), word, dtype=np.uint32)
        d = O.dequantize_f32(w, s, b, K)
        assert all(_bits32(v) == int(f32h, 16) for v in d[0]), (sh, bh, q)
        bf = O.dequantize(w, s, b, K, "bf16").view(torch.int16).numpy().astype(np.uint16)
        hf = O.dequantize(w, s, b, K, "f16").view(torch.int16).numpy().astype(np.uint16)
        assert np.all(bf == int(bf16h, 16)), (sh, bh, q, hex(bf[0, 0]))
        assert np.all(hf == int(f16h, 16)), (sh, bh, q, hex(hf[0, 0]))


def test_dequant_bf16_metadata_golden():
    """bf16 scales/biases widen exactly (hand-derived values in the fixture)."""
    n = 0
    for sc_h, b_h, want0, want1, _ in _rows("dequant_bf16_meta.txt"):
        words = np.array([[0xAAAAAAAA, 0, 0, 0]], dtype=np.uint32)  # k = 1, 3, 5, ... set in word 0
        sc = torch.tensor([[int(sc_h, 16)]], dtype=torch.int16).view(torch.bfloat16)
        b = None if b_h == "sym" else torch.tensor([[int(b_h, 16) - (1 << 16) * (int(b_h, 16) >= 1 << 15)]],
                                                   dtype=torch.int16).view(torch.bfloat16)
        if int(sc_h, 16) >= 1 << 15:
            raise AssertionError("fixture scales are positive")
        d = O.dequantize_f32(words, sc, b, 128)
        assert _bits32(d[0, 0]) == int(want0, 16), (sc_h, b_h)
        assert _bits32(d[0, 1]) == int(want1, 16), (sc_h, b_h)
        n += 1
    assert n == 7


def test_bf16_rounding_golden():
    for f32h, bf16h in _rows("bf16_rounding.txt"):
        v = np.frombuffer(struct.pack("<I", int(f32h, 16)), dtype=np.float32)
        got = O.round_to(v, "bf16").view(torch.int16).numpy().astype(np.uint16)[0]
        assert got == int(bf16h, 16), (f32h, hex(got))


def test_dequant_all_zero_bits_is_bias_all_one_is_sum():
    t = synth.q1_tensor(5, 256, seed=21, affine=True)
    s = t.scales.astype(np.float32)
    b = t.biases.astype(np.float32)
    zeros = np.zeros_like(t.words)
    ones = np.full_like(t.words, 0xFFFFFFFF)
    d0 = O.dequantize_f32(zeros, t.scales, t.biases, 256)
    d1 = O.dequantize_f32(ones, t.scales, t.biases, 256)
    for g in range(2):
        np.testing.assert_array_equal(d0[:, g * 128:(g + 1) * 128], np.repeat(b[:, g:g + 1], 128, 1))
        np.testing.assert_array_equal(d1[:, g * 128:(g + 1) * 128],
                                      np.repeat((s[:, g:g + 1] + b[:, g:g + 1]).astype(np.float32), 128, 1))


def test_symmetric_values_are_plus_minus_half_scale_and_both_occur():
    t = synth.q1_tensor(6, 512, seed=31, affine=False)
    d = O.dequantize_f32(t.words, t.scales, None, 512)
    bits = O.unpack(t.words, 512)
    for n in range(6):
        for g in range(4):
            half = np.float32(t.scales[n, g]) / np.float32(2)
            vals = d[n, g * 128:(g + 1) * 128]
            q = bits[n, g * 128:(g + 1) * 128]
            assert set(np.unique(vals).tolist()) == {float(-half), float(half)}
            # bit 1 -> +s/2, bit 0 -> -s/2 (rMLX issue: bit0 -> negative, bit1 -> positive)
            assert np.all(vals[q == 1] == half) and np.all(vals[q == 0] == -half)


def test_symmetric_equals_affine_when_bias_is_exactly_minus_half_scale():
    # scales >= 2^-13 are normal fp16 values whose half is again an fp16 value,
    # so storing the bias -s/2 explicitly is lossless.
    t = synth.q1_tensor(4, 256, seed=41, affine=False)
    s = np.maximum(t.scales, np.float16(2.0 ** -13))
    b = (-(s.astype(np.float32) / 2)).astype(np.float16)
    assert np.all(b.astype(np.float32) == -s.astype(np.float32) / 2)
    da = O.dequantize_f32(t.words, s, b, 256)
    ds = O.dequantize_f32(t.words, s, None, 256)
    np.testing.assert_array_equal(da.view(np.uint32), ds.view(np.uint32))


# ---------------------------------------------------------------- matmul
def _exact_qmm(x_bf16, words, scales, biases, K, group=128):
    """Exact rational brute force: dequant with Python Fractions of the fp32
    values (derived independently of the oracle: bit test per weight, fp32
    add done by numpy scalar), then exact sums."""
    xs = x_bf16.to(torch.float64).numpy()
    M, N = xs.shape[0], words.shape[0]
    out = [[Fraction(0)] * N for _ in range(M)]
    for n in range(N):
        for k in range(K):
            q = (int(words[n, k // 32]) >> (k % 32)) & 1
            s = np.float32(scales[n, k // group])
            b = np.float32(biases[n, k // group]) if biases is not None else np.float32(-0.5) * s
            w = np.float32(s + b) if q else b
            fw = Fraction(float(w))
            for m in range(M):
                out[m][n] += Fraction(float(xs[m, k])) * fw
    return out


@pytest.mark.parametrize("affine", [False, True])
def test_qmm_brute_force_tiny(affine):
    K, N, M = 128, 4, 3
    t = synth.q1_tensor(N, K, seed=51 + affine, affine=affine)
    x = synth.activations(M, K, seed=61)
    want = _exact_qmm(x, t.words, t.scales, t.biases, K)
    got = O.qmm(x, t.words, t.scales, t.biases, K)
    for m in range(M):
        for n in range(N):
            exact = float(want[m][n])
            assert abs(got[m, n] - exact) <= 1e-12 * max(1.0, abs(exact)), (m, n)


def test_qmm_one_hot_selects_a_column():
    K, N = 256, 6
    t = synth.q1_tensor(N, K, seed=71, affine=True)
    wd = O.dequantize_f32(t.words, t.scales, t.biases, K)
    for k in (0, 1, 31, 32, 127, 128, 200, 255):
        x = torch.zeros(1, K, dtype=torch.bfloat16)
        x[0, k] = 1.0
        y = O.qmm(x, t.words, t.scales, t.biases, K)
        np.testing.assert_array_equal(y[0], wd[:, k].astype(np.float64))


@pytest.mark.parametrize("affine", [False, True])
def test_qmm_all_ones_closed_form(affine):
    # x = 1 everywhere: Y[n] = sum_g popcount_g * fl32(s+b) + (128 - popcount_g) * b
    K, N = 384, 5
    t = synth.q1_tensor(N, K, seed=81, affine=affine)
    x = torch.ones(1, K, dtype=torch.bfloat16)
    y = O.qmm(x, t.words, t.scales, t.biases, K)[0]
    for n in range(N):
        tot = Fraction(0)
        for g in range(K // 128):
            pc = sum(bin(int(t.words[n, c])).count("1") for c in range(4 * g, 4 * g + 4))
            s = np.float32(t.scales[n, g])
            b = np.float32(t.biases[n, g]) if affine else np.float32(-0.5) * s
            tot += pc * Fraction(float(np.float32(s + b))) + (128 - pc) * Fraction(float(b))
        assert abs(y[n] - float(tot)) <= 1e-12 * max(1.0, abs(float(tot)))


def test_symmetric_complement_negates():
    K, N, M = 256, 7, 2
    t = synth.q1_tensor(N, K, seed=91, affine=False)
    x = synth.activations(M, K, seed=92)
    y = O.qmm(x, t.words, t.scales, None, K)
    yc = O.qmm(x, ~t.words, t.scales, None, K)
    np.testing.assert_allclose(yc, -y, rtol=0, atol=1e-12)


def test_qmm_linear_in_x():
    K, N = 256, 5
    t = synth.q1_tensor(N, K, seed=101, affine=True)
    a = synth.activations(1, K, seed=102)
    b = synth.activations(1, K, seed=103)
    ya = O.qmm(a, t.words, t.scales, t.biases, K)
    yb = O.qmm(b, t.words, t.scales, t.biases, K)
    yab = O.qmm(a.double() * 2.0 + b.double() * -3.0, t.words, t.scales, t.biases, K)
    np.testing.assert_allclose(yab, 2 * ya - 3 * yb, rtol=1e-12, atol=1e-12)


def test_qmm_rows_subset_matches_full():
    K, N = 256, 9
    t = synth.q1_tensor(N, K, seed=111, affine=True)
    x = synth.activations(2, K, seed=112)
    full = O.qmm(x, t.words, t.scales, t.biases, K)
    rows = np.array([8, 0, 3])
    np.testing.assert_array_equal(O.qmm(x, t.words, t.scales, t.biases, K, rows=rows), full[:, rows])


def test_affine_with_exact_minus_half_bias_close_to_symmetric():
    K, N = 512, 4
    t = synth.q1_tensor(N, K, seed=121, affine=False)
    s = np.maximum(t.scales, np.float16(2.0 ** -13))
    b = (-(s.astype(np.float32) / 2)).astype(np.float16)
    x = synth.activations(3, K, seed=122)
    np.testing.assert_array_equal(O.qmm(x, t.words, s, b, K), O.qmm(x, t.words, s, None, K))


# ---------------------------------------------------------------- group sizes 32 and 64
def test_dequant_group_32_hand_built():
    """K = 128 in four groups of 32: each word takes its own scale."""
    words = np.array([[0xFFFFFFFF, 0x00000000, 0x00000001, 0x80000000]], dtype=np.uint32)
    scales = np.array([[1.0, 2.0, 0.5, 4.0]], dtype=np.float16)
    d = O.dequantize_f32(words, scales, None, 128)[0]
    want = np.concatenate([np.full(32, 0.5), np.full(32, -1.0), [0.25], np.full(31, -0.25),
                           np.full(31, -2.0), [2.0]]).astype(np.float32)
    assert np.array_equal(d, want)


def test_dequant_group_64_affine_hand_built():
    """K = 128 in two groups of 64: {0, 1} then {-1.5, fl32(3 - 1.5) = 1.5}."""
    words = np.array([[0x0000FFFF, 0xFFFF0000, 0x00000000, 0xFFFFFFFF]], dtype=np.uint32)
    scales = np.array([[1.0, 3.0]], dtype=np.float16)
    biases = np.array([[0.0, -1.5]], dtype=np.float16)
    d = O.dequantize_f32(words, scales, biases, 128)[0]
    want = np.concatenate([np.full(16, 1.0), np.full(32, 0.0), np.full(16, 1.0),
                           np.full(32, -1.5), np.full(32, 1.5)]).astype(np.float32)
    assert np.array_equal(d, want)


@pytest.mark.parametrize("group", [32, 64])
@pytest.mark.parametrize("affine", [False, True])
def test_qmm_brute_force_small_groups(group, affine):
    K, N, M = 128, 3, 2
    t = synth.q1_tensor(N, K, seed=71 + group + affine, affine=affine, group=group)
    x = synth.activations(M, K, seed=72)
    want = _exact_qmm(x, t.words, t.scales, t.biases, K, group)
    got = O.qmm(x, t.words, t.scales, t.biases, K)
    for m in range(M):
        for n in range(N):
            assert got[m, n] == pytest.approx(float(want[m][n]), rel=1e-12, abs=1e-12)


def test_group_size_from_metadata_shape():
    assert O.group_size_of(512, np.zeros((2, 16))) == 32
    assert O.group_size_of(512, np.zeros((2, 8))) == 64
    assert O.group_size_of(512, np.zeros((2, 4))) == 128
    with pytest.raises(ValueError):
        O.group_size_of(512, np.zeros((2, 2)))  # 256 per group


# ---------------------------------------------------------------- FFN
def test_silu_closed_form():
    for g in (-20.0, -1.5, 0.0, 0.25, 3.0, 30.0):
        assert O.silu(np.array([g]))[0] == pytest.approx(g / (1 + math.exp(-g)), rel=1e-15, abs=1e-300)
    assert O.silu(np.array([0.0]))[0] == 0.0


def test_ffn_brute_force_tiny():
    D, F, M = 128, 256, 2
    gate = synth.q1_tensor(F, D, seed=131, affine=False)
    up = synth.q1_tensor(F, D, seed=132, affine=True)
    down = synth.q1_tensor(D, F, seed=133, affine=False)
    x = synth.activations(M, D, seed=134)
    g = _exact_qmm(x, gate.words, gate.scales, None, D)
    u = _exact_qmm(x, up.words, up.scales, up.biases, D)
    h = np.array([[float(g[m][f]) / (1 + math.exp(-float(g[m][f]))) * float(u[m][f])
                   for f in range(F)] for m in range(M)])
    # the down projection of h, summed with math.fsum (exactly rounded sums)
    wd = O.dequantize_f32(down.words, down.scales, None, F)  # pinned above
    want = np.array([[math.fsum(h[m, k] * float(wd[n, k]) for k in range(F)) for n in range(D)]
                     for m in range(M)])
    y, h_o = O.ffn(x, (gate.words, gate.scales, None, D), (up.words, up.scales, up.biases, D),
                   (down.words, down.scales, None, F))
    np.testing.assert_allclose(h_o, h, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(y, want, rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------- decode chain
def _selection(rows, K, sel):
    """Affine Q1 tensor whose dequantized row n is the one-hot e_{sel[n]}:
    scale 1, bias 0, bit sel[n] of row n set (packed here by hand)."""
    words = np.zeros((rows, K // 32), dtype=np.uint32)
    for n, k in enumerate(sel):
        words[n, k // 32] |= np.uint32(1) << np.uint32(k % 32)
    scales = np.full((rows, K // 128), np.float16(1.0))
    biases = np.zeros((rows, K // 128), dtype=np.float16)
    return (words, scales, biases, K)


def test_decode_chain_on_selection_matrices():
    """With one-hot weight rows every product is a gather: a = h[pi], g = a[rho],
    u = a[sigma], h' = bf16(SiLU(g) * u)[tau].  Distinct random index maps per
    layer catch a transposed operand, a swapped gate/up or a wrong layer order."""
    D, F, M, L = 128, 256, 2, 2
    rng = np.random.default_rng(77)
    x = synth.activations(M, D, seed=78)
    layers, maps = [], []
    for _ in range(L):
        pi = rng.permutation(D)
        rho, sigma = rng.integers(0, D, F), rng.integers(0, D, F)
        tau = rng.permutation(F)[:D]
        layers.append((_selection(D, D, pi), _selection(F, D, rho), _selection(F, D, sigma),
                       _selection(D, F, tau)))
        maps.append((pi, rho, sigma, tau))
    h = x.to(torch.float64)
    for pi, rho, sigma, tau in maps:
        a = h[:, pi]                       # exact: each output is one input value
        hh = torch.nn.functional.silu(a[:, rho]) * a[:, sigma]
        # one rounding to bf16 (through fp32, as the pinned bf16 rounding does)
        h = hh[:, tau].to(torch.float32).to(torch.bfloat16).to(torch.float64)
    got = O.decode_chain(x, layers)
    assert got.dtype == torch.bfloat16
    assert torch.equal(got.to(torch.float64), h)


# ---------------------------------------------------------------- exact repack from dense
def _group(lo, hi, pattern_seed=0):
    rng = np.random.default_rng(pattern_seed)
    q = rng.integers(0, 2, 128).astype(np.uint8)
    q[0], q[1] = 0, 1
    return np.where(q == 1, np.float32(hi), np.float32(lo)).astype(np.float32), q


def test_pack_group_hand_built_cases():
    # symmetric +-0.75: scale 1.5 (fp16 0x3E00), bit 1 for +0.75
    v, q = _group(-0.75, 0.75)
    bits, sc, b = O.pack_group(v, symmetric=True)
    assert b is None and sc.view(np.uint16) == 0x3E00 and np.array_equal(bits, q)
    # affine {0.25, 1.0}: bias 0.25, scale 0.75 (exact in fp16)
    v, q = _group(0.25, 1.0)
    bits, sc, b = O.pack_group(v, symmetric=False)
    assert float(b) == 0.25 and float(sc) == 0.75 and np.array_equal(bits, q)
    # {-0, +0}: bit 1 for +0; symmetric scale +0 (derived bias -0), affine bias -0
    v, q = _group(-0.0, 0.0)
    bits, sc, b = O.pack_group(v, symmetric=True)
    assert sc.view(np.uint16) == 0x0000 and np.array_equal(bits, q)
    bits, sc, b = O.pack_group(v, symmetric=False)
    assert b.view(np.uint16) == 0x8000 and sc.view(np.uint16) == 0x0000 and np.array_equal(bits, q)
    # one value: symmetric +0.5 -> scale 1.0, all bits 1; -0.5 -> scale 1.0, all bits 0
    bits, sc, b = O.pack_group(np.full(128, 0.5, np.float32), symmetric=True)
    assert float(sc) == 1.0 and bits.all()
    bits, sc, b = O.pack_group(np.full(128, -0.5, np.float32), symmetric=True)
    assert float(sc) == 1.0 and not bits.any()
    # one value, affine: the bias is the value, all bits 0
    bits, sc, b = O.pack_group(np.full(128, 3.0, np.float32), symmetric=False)
    assert float(b) == 3.0 and not bits.any()
    # refusals: three values, NaN, infinity, not +-m in symmetric mode, a bias
    # that is not an fp16 value
    v3 = _group(-0.5, 0.5)[0]
    v3[5] = np.float32(0.25)
    assert O.pack_group(v3, True) is None and O.pack_group(v3, False) is None
    for bad in (np.nan, np.inf, -np.inf):
        vb = _group(-0.5, 0.5)[0]
        vb[7] = np.float32(bad)
        assert O.pack_group(vb, True) is None and O.pack_group(vb, False) is None
    assert O.pack_group(_group(-0.5, 0.75)[0], True) is None
    assert O.pack_group(_group(1.0 + 2.0 ** -20, 2.0)[0], False) is None


def test_pack_group_scale_rule_matches_exhaustive_search():
    """An affine group {lo, hi} (lo an fp16 value) is kept iff some finite fp16
    scale gives fl32(scale + lo) == hi; the chosen scale must be one of them."""
    all16 = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16)
    all16 = np.concatenate([all16, -all16[1:]]).astype(np.float32)
    rng = np.random.default_rng(11)
    kept = refused = 0
    for _ in range(3000):
        lo = np.float32(np.float16(rng.normal() * 10 ** rng.uniform(-6, 4)))
        hi = np.float32(lo + np.float32(abs(rng.normal()) * 10 ** rng.uniform(-8, 3)))
        if hi == lo:
            continue
        v = _group(lo, hi)[0]
        r = O.pack_group(v, symmetric=False)
        exists = np.any((all16 + lo).astype(np.float32).view(np.uint32) == np.float32(hi).view(np.uint32))
        assert (r is not None) == bool(exists), (lo, hi)
        if r is not None:
            assert np.float32(np.float32(r[1]) + np.float32(r[2])) == hi
            kept += 1
        else:
            refused += 1
    assert kept > 300 and refused > 300


@pytest.mark.parametrize("affine", [False, True])
def test_pack_from_dense_round_trip(affine):
    N, K = 24, 384
    t = synth.q1_tensor(N, K, seed=141 + affine, affine=affine)
    dense = O.dequantize_f32(t.words, t.scales, t.biases, K)    # pinned above
    w, sc, b, bad = O.pack_from_dense(dense, symmetric=not affine)
    assert bad == 0
    # every bit comes back (no group of the random tensor is single-valued)
    assert np.array_equal(w, t.words)
    if not affine:
        assert np.array_equal(sc.view(np.uint16), t.scales.view(np.uint16))
    back = O.dequantize_f32(w, sc, b, K)
    assert np.array_equal(back.view(np.uint32), dense.view(np.uint32))
    # a group with a third value is refused and zeroed; the rest are untouched
    dense2 = dense.copy()
    dense2[3, 130] = np.float32(1234.5)
    w2, sc2, b2, bad2 = O.pack_from_dense(dense2, symmetric=not affine)
    assert bad2 == 1 and float(sc2[3, 1]) == 0.0 and not w2[3, 4:8].any()
    assert np.array_equal(np.delete(w2, slice(4, 8), axis=1), np.delete(w, slice(4, 8), axis=1))


# ---------------------------------------------------------------- gather
def test_embed_gather_rows_and_out_of_range():
    V, K = 10, 256
    t = synth.q1_tensor(V, K, seed=141, affine=True)
    ids = np.array([3, 0, 9, 10, -1, 3], dtype=np.int32)
    out, bad = O.embed_gather(ids, t.words, t.scales, t.biases, K, "f32")
    assert bad == 2
    wd = O.dequantize_f32(t.words, t.scales, t.biases, K)
    for i, r in enumerate(ids):
        if 0 <= r < V:
            np.testing.assert_array_equal(out[i].numpy(), wd[r])
        else:
            assert torch.all(out[i] == 0)


# ---------------------------------------------------------------- symmetric check
def test_is_symmetric_exact_and_edge_cases():
    s = np.array([[0.5, 0.25], [1.0, 2.0 ** -13]], dtype=np.float16)
    b = (-(s.astype(np.float32) / 2)).astype(np.float16)
    assert O.is_symmetric(s, b)
    b2 = b.copy()
    b2[1, 1] = np.float16(-2.0 ** -13)  # one group differs -> affine
    assert not O.is_symmetric(s, b2)
    # +0 and -0: s = 0 gives derived bias -0; a stored +0 still counts as equal
    z = np.zeros((1, 1), dtype=np.float16)
    assert O.is_symmetric(z, np.zeros((1, 1), dtype=np.float16))
    nan = np.array([[np.nan]], dtype=np.float16)
    assert not O.is_symmetric(nan, nan)
    # a scale too small for -s/2 to be an fp16 value cannot be stored exactly
    tiny = np.array([[_f16(0x0001)]], dtype=np.float16)
    assert not O.is_symmetric(tiny, (-(tiny.astype(np.float32) / 2)).astype(np.float16))


# ---------------------------------------------------------------- accounting
def test_storage_bytes_bias_is_one_sixty_fourth_byte_per_weight():
    # "Support Bonsai-27B affine Q1", "Measured impact": 412,262,400 bytes of
    # fp16 biases removed; at 2 bytes per 128 weights that is 26.38e9 weights,
    # consistent with a 27B-parameter checkpoint.
    st = O.storage_bytes(17408, 5120, symmetric=False)
    assert st["biases"] * 64 == 17408 * 5120
    assert st["packed"] == 17408 * 5120 // 8
    params = 412_262_400 * 64
    assert 26.0e9 < params < 27.0e9
    sym = O.storage_bytes(17408, 5120, symmetric=True)
    # 1.125 bits per weight symmetric, 1.25 affine
    assert sym["total"] * 8 / (17408 * 5120) == pytest.approx(1.125)
    assert st["total"] * 8 / (17408 * 5120) == pytest.approx(1.25)


# ---------------------------------------------------------------- tolerance helper
@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_half_ulp_covers_one_rounding_and_is_tight(dtype):
    # the output-rounding term of the matmul bar: rounding any value once to
    # the dtype moves it by at most half_ulp, and half_ulp is not loose by
    # more than a factor of two (a value half-way between two neighbours moves
    # by exactly half an ulp)
    from tests.tolerance import half_ulp
    rng = np.random.default_rng(5)
    top = 14 if dtype == "f16" else 20  # within fp16's range
    y = rng.standard_normal(20000) * np.exp2(rng.integers(-20, top, 20000))
    y = np.concatenate([y, [1.0 - 2.0 ** -12, 255.9, -3.0, 1e-6]])
    r = O.round_to(y, dtype).double().numpy()
    err = np.abs(r - y.astype(np.float32).astype(np.float64))
    h = half_ulp(y, dtype)
    assert np.all(err <= h)
    one = O.round_to(np.array([1.0]), dtype).double().numpy()
    assert half_ulp(one, dtype)[0] == {"bf16": 2.0 ** -8, "f16": 2.0 ** -11, "f32": 2.0 ** -24}[dtype]
