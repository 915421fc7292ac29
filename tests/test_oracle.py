"""Pins for the CPU oracle: each test checks it against something other than
itself -- hand-written fixtures, exact rational arithmetic, closed forms,
invariants of the definition, and the IEEE round-to-nearest-even rule."""
import os
import struct
from fractions import Fraction

import numpy as np
import pytest

import oracle
from affine_bit_quantized_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- helpers

def bf16_bits_to_fraction(h: int) -> Fraction:
    f = struct.unpack("<f", struct.pack("<I", (int(h) & 0xFFFF) << 16))[0]
    return Fraction(f)


def fraction_to_bf16_bits(v: Fraction) -> int:
    """Round an exact rational to bf16, nearest with ties to even (Python's
    round() on a Fraction is round-half-even)."""
    if v == 0:
        return 0
    sign = 0x8000 if v < 0 else 0
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    # now 2^e <= a < 2^(e+1)
    e = max(e, -126)
    spacing = Fraction(2) ** (e - 7)
    r = round(a / spacing) * spacing
    if r >= Fraction(2) ** 128:
        return sign | 0x7F80
    bits = struct.unpack("<I", struct.pack("<f", float(r)))[0] >> 16
    assert bf16_bits_to_fraction(bits) == r
    return sign | bits


def codes_from_words_by_hand(word: int, bits: int):
    per = 32 // bits
    return [(word >> (bits * i)) & ((1 << bits) - 1) for i in range(per)]


# ---------------------------------------------------------------- bf16 rounding

def test_bf16_rounding_exhaustive_identity_and_midpoints():
    """Every finite bf16 value maps to itself; each midpoint between
    neighbours goes to the one with the even significand; a hair either side
    of a midpoint goes to the nearer neighbour."""
    pos = np.arange(0, 0x7F80, dtype=np.uint32)       # +0 .. largest finite
    vals = (pos << 16).view(np.float32).astype(np.float64)
    assert np.array_equal(oracle.double_to_bf16(vals), pos.astype(np.uint16))
    assert np.array_equal(oracle.double_to_bf16(-vals), (pos | 0x8000).astype(np.uint16))
    lo, hi = vals[:-1], vals[1:]
    mid = (lo + hi) / 2                                  # exact in double
    got = oracle.double_to_bf16(mid)
    even = np.where(pos[:-1] % 2 == 0, pos[:-1], pos[1:]).astype(np.uint16)
    assert np.array_equal(got, even)
    eps = (hi - lo) * 2.0 ** -20
    assert np.array_equal(oracle.double_to_bf16(mid - eps), pos[:-1].astype(np.uint16))
    assert np.array_equal(oracle.double_to_bf16(mid + eps), pos[1:].astype(np.uint16))


def test_bf16_rounding_special_values():
    big = float(bf16_bits_to_fraction(0x7F7F))
    half_ulp = 2.0 ** (127 - 8)
    assert oracle.double_to_bf16(np.array([big + half_ulp]))[0] == 0x7F80     # ties to even -> inf
    assert oracle.double_to_bf16(np.array([big + half_ulp * 0.99]))[0] == 0x7F7F
    assert oracle.double_to_bf16(np.array([np.inf, -np.inf]))[1] == 0xFF80
    assert oracle.double_to_bf16(np.array([np.nan]))[0] & 0x7FC0 == 0x7FC0
    assert oracle.double_to_bf16(np.array([-0.0]))[0] == 0x8000
    # a double just above a bf16 midpoint that float32 would first round onto
    # the midpoint (the double-rounding trap): 1 + 2^-8 + 2^-40
    v = 1.0 + 2.0 ** -8 + 2.0 ** -40
    assert oracle.double_to_bf16(np.array([v]))[0] == 0x3F81
    assert fraction_to_bf16_bits(Fraction(v)) == 0x3F81


def test_bf16_widening_exact():
    for h in (0x3F80, 0xBF00, 0x0001, 0x7F7F, 0x4318):
        assert oracle.bf16_to_double([h])[0] == float(bf16_bits_to_fraction(h))


# ---------------------------------------------------------------- packing

def _read_nibble_fixture():
    rows = []
    with open(os.path.join(GOLDEN, "nibble_order.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            rows.append((int(parts[0]), int(parts[1], 16), [int(c) for c in parts[2:]]))
    return rows


def test_nibble_order_fixture():
    for bits, word, codes in _read_nibble_fixture():
        per = 32 // bits
        got = oracle.unpack(np.array([[word]], np.uint32), 1, per, bits)[0].tolist()
        assert got == codes, (bits, hex(word))
        assert oracle.pack(np.array([codes], np.uint8), bits)[0, 0] == word


@pytest.mark.parametrize("bits", [4, 8])
def test_pack_unpack_exhaustive_positions(bits):
    per = 32 // bits
    vals = 1 << bits
    # every code value at every position of a word, other positions zero
    codes = np.zeros((vals * per, per), np.uint8)
    for v in range(vals):
        for p in range(per):
            codes[v * per + p, p] = v
    words = oracle.pack(codes, bits)
    for i in range(codes.shape[0]):
        assert codes_from_words_by_hand(int(words[i, 0]), bits) == codes[i].tolist()
    assert np.array_equal(oracle.unpack(words, codes.shape[0], per, bits), codes)


@pytest.mark.parametrize("bits", [4, 8])
def test_pack_unpack_round_trip_random(bits):
    rng = np.random.default_rng(1)
    words = rng.integers(0, 1 << 32, size=(7, 3 * bits), dtype=np.uint32)   # K = 96 codes per row
    K = 3 * 32
    codes = oracle.unpack(words, 7, K, bits)
    assert codes.max() < (1 << bits)
    assert np.array_equal(oracle.pack(codes, bits), words)


# ---------------------------------------------------------------- matmul pins

def _case(M, N, K, seed, bits=4):
    w = synth.make_weights(N, K, seed, bits=bits)
    x = synth.make_x(M, K, seed)
    return x, w


def brute_force(x, w):
    """Exact rational evaluation of the definition; returns (exact, bf16)."""
    M, K = x.shape
    N = w.N
    per = 32 // w.bits
    exact = [[Fraction(0)] * N for _ in range(M)]
    for n in range(N):
        for k in range(K):
            word = int(w.w_packed[n, k // per])
            q = (word >> (w.bits * (k % per))) & ((1 << w.bits) - 1)
            g = k // w.group_size
            wk = bf16_bits_to_fraction(w.scales[n, g]) * q + bf16_bits_to_fraction(w.biases[n, g])
            for m in range(M):
                exact[m][n] += bf16_bits_to_fraction(x[m, k]) * wk
    bits = np.array([[fraction_to_bf16_bits(v) for v in row] for row in exact], np.uint16)
    return exact, bits


@pytest.mark.parametrize("M,N,K,bits,seed", [(1, 4, 64, 4, 3), (2, 3, 128, 4, 4), (2, 2, 64, 8, 5),
                                             (1, 1, 128, 8, 6)])
def test_brute_force_rational(M, N, K, bits, seed):
    x, w = _case(M, N, K, seed, bits)
    exact, ref_bits = brute_force(x, w)
    y_exact, y_bf16 = oracle.matmul(x, w.w_packed, w.scales, w.biases, M, N, K, bits=bits)
    assert np.array_equal(y_bf16, ref_bits)
    for m in range(M):
        for n in range(N):
            assert abs(Fraction(y_exact[m, n]) - exact[m][n]) <= abs(exact[m][n]) * Fraction(1, 2 ** 45)


def test_worked_example_fixture():
    vals = {}
    with open(os.path.join(GOLDEN, "worked_example.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                key, *rest = line.split()
                vals[key] = rest
    M, N, K = (int(vals[k][0]) for k in ("M", "N", "K"))
    words = np.empty((N, K // 8), np.uint32)
    words[0, :] = int(vals["row0_word"][0], 16)
    words[1, :] = int(vals["row1_word"][0], 16)
    scales = np.array([int(v, 16) for v in vals["scales"]], np.uint16).reshape(N, 2)
    biases = np.array([int(v, 16) for v in vals["biases"]], np.uint16).reshape(N, 2)
    xg = [int(v, 16) for v in vals["x_group_values"]]
    x = np.array([[xg[k // 64] for k in range(K)]], np.uint16)
    y_exact, y_bf16 = oracle.matmul(x, words, scales, biases, M, N, K)
    assert y_exact[0].tolist() == [float(v) for v in vals["y_exact"]]
    assert y_bf16[0].tolist() == [int(v, 16) for v in vals["y_bf16"]]


def test_one_hot_x_returns_dequantized_column_and_endpoints():
    """A one-hot x picks one dequantized weight column: q=0 gives the bias,
    q=15 gives 15*scale + bias."""
    N, K = 5, 128
    w = synth.make_weights(N, K, 11)
    codes = oracle.unpack(w.w_packed, N, K)
    codes[:, 3] = 0
    codes[:, 70] = 15
    codes[:, 100] = 9
    wp = oracle.pack(codes)
    s = w.scales.astype(np.uint32)
    for k in (3, 70, 100, 127):
        x = np.zeros((1, K), np.uint16)
        x[0, k] = 0x3F80                                   # 1.0
        y_exact, y_bf16 = oracle.matmul(x, wp, w.scales, w.biases, 1, N, K)
        g = k // 64
        for n in range(N):
            want = bf16_bits_to_fraction(s[n, g]) * int(codes[n, k]) + bf16_bits_to_fraction(w.biases[n, g])
            assert Fraction(y_exact[0, n]) == want
            assert y_bf16[0, n] == fraction_to_bf16_bits(want)
        if k == 3:
            assert np.array_equal(y_bf16[0], w.biases[:, 0])
        if k == 70:
            want15 = [bf16_bits_to_fraction(s[n, 1]) * 15 + bf16_bits_to_fraction(w.biases[n, 1]) for n in range(N)]
            assert y_exact[0].tolist() == [float(v) for v in want15]


def test_one_hot_x_eight_bit_endpoints():
    """8-bit codes: a one-hot x returns q=0 -> bias, q=255 -> 255*scale + bias,
    and a middle code exactly (byte order: lowest byte = lowest k)."""
    N, K = 4, 128
    w = synth.make_weights(N, K, 12, bits=8)
    codes = oracle.unpack(w.w_packed, N, K, 8)
    codes[:, 5] = 0
    codes[:, 66] = 255
    codes[:, 99] = 128
    wp = oracle.pack(codes, 8)
    assert (int(wp[0, 66 // 4]) >> (8 * (66 % 4))) & 0xFF == 255       # byte 2 of word 16
    for k, q in ((5, 0), (66, 255), (99, 128)):
        x = np.zeros((1, K), np.uint16)
        x[0, k] = 0x3F80
        y_exact, y_bf16 = oracle.matmul(x, wp, w.scales, w.biases, 1, N, K, bits=8)
        g = k // 64
        for n in range(N):
            want = bf16_bits_to_fraction(w.scales[n, g]) * q + bf16_bits_to_fraction(w.biases[n, g])
            assert Fraction(y_exact[0, n]) == want
            assert y_bf16[0, n] == fraction_to_bf16_bits(want)


def test_zero_x_gives_zero():
    x = np.zeros((3, 192), np.uint16)
    w = synth.make_weights(9, 192, 12)
    y_exact, y_bf16 = oracle.matmul(x, w.w_packed, w.scales, w.biases, 3, 9, 192)
    assert not y_exact.any() and not y_bf16.any()


def test_constant_codes_closed_form():
    """All-ones x over one group with constant code c: y = 64 * (scale*c + bias)."""
    N, K = 4, 128
    for c in (0, 1, 7, 15):
        codes = np.full((N, K), c, np.uint8)
        wp = oracle.pack(codes)
        w = synth.make_weights(N, K, 13)
        x = np.zeros((1, K), np.uint16)
        x[0, 64:128] = 0x3F80
        y_exact, _ = oracle.matmul(x, wp, w.scales, w.biases, 1, N, K)
        for n in range(N):
            want = 64 * (bf16_bits_to_fraction(w.scales[n, 1]) * c + bf16_bits_to_fraction(w.biases[n, 1]))
            assert Fraction(y_exact[0, n]) == want


def test_group_permutation_invariance():
    """Permuting whole K groups of W (codes, scales, biases) together with x
    leaves y unchanged up to double summation order."""
    M, N, K = 2, 6, 512
    x, w = _case(M, N, K, 14)
    G = K // 64
    perm = np.random.default_rng(2).permutation(G)
    codes = oracle.unpack(w.w_packed, N, K).reshape(N, G, 64)[:, perm].reshape(N, K)
    xp = x.reshape(M, G, 64)[:, perm].reshape(M, K)
    y0, b0 = oracle.matmul(x, w.w_packed, w.scales, w.biases, M, N, K)
    y1, b1 = oracle.matmul(xp, oracle.pack(codes), w.scales[:, perm], w.biases[:, perm], M, N, K)
    assert np.allclose(y0, y1, rtol=1e-13, atol=1e-13)


def test_dequant_matches_definition_on_fixture_rows():
    N, K = 2, 64
    wp = np.array([[0x76543210] * 8, [0xFFFFFFFF] * 8], np.uint32)
    s = np.array([[0x3F00], [0x3E00]], np.uint16)      # 0.5, 0.125
    b = np.array([[0xBF80], [0x0000]], np.uint16)      # -1, 0
    w = oracle.dequant(wp, s, b, N, K)
    assert w[0, :8].tolist() == [0.5 * q - 1.0 for q in range(8)]
    assert np.all(w[1] == 0.125 * 15)


def test_sampled_matches_full():
    M, N, K = 3, 40, 256
    x, w = _case(M, N, K, 15)
    y_exact, y_bf16 = oracle.matmul(x, w.w_packed, w.scales, w.biases, M, N, K, nthreads=3)
    rng = np.random.default_rng(3)
    im, inn = rng.integers(0, M, 50), rng.integers(0, N, 50)
    se, sb = oracle.matmul_sampled(x, w.w_packed, w.scales, w.biases, M, N, K, im, inn)
    assert np.array_equal(se, y_exact[im, inn]) and np.array_equal(sb, y_bf16[im, inn])


def test_thread_count_does_not_change_result():
    M, N, K = 2, 33, 320
    x, w = _case(M, N, K, 16)
    a = oracle.matmul(x, w.w_packed, w.scales, w.biases, M, N, K, nthreads=1)
    b = oracle.matmul(x, w.w_packed, w.scales, w.biases, M, N, K, nthreads=5)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# ---------------------------------------------------------------- quantization

@pytest.mark.parametrize("bits", [4, 8])
def test_quantize_invariants(bits):
    rng = np.random.default_rng(4)
    N, K = 6, 256
    w = rng.normal(0, 0.05, size=(N, K)).astype(np.float32)
    w[2, 64:128] = 0.25                                   # constant group
    wp, s, b = oracle.quantize(w, bits=bits)
    deq = oracle.dequant(wp, s, b, N, K, bits=bits)
    sd = np.repeat(oracle.bf16_to_double(s), 64, axis=1)
    qmax = (1 << bits) - 1
    codes = oracle.unpack(wp, N, K, bits)
    # each group's min maps to code 0 region and its max to the top code region
    for n in range(N):
        for g in range(K // 64):
            seg = w[n, g * 64:(g + 1) * 64].astype(np.float64)
            bias = float(bf16_bits_to_fraction(b[n, g]))
            assert b[n, g] == fraction_to_bf16_bits(Fraction(float(seg.min())))
            if seg.max() == seg.min():
                assert s[n, g] == 0 and not codes[n, g * 64:(g + 1) * 64].any()
                continue
            span = Fraction(float(seg.max())) - Fraction(float(seg.min()))
            assert s[n, g] == fraction_to_bf16_bits(span / qmax)
            # nearest code: the error of every non-clamped element is at most half a step
            q = codes[n, g * 64:(g + 1) * 64].astype(np.float64)
            step = float(bf16_bits_to_fraction(s[n, g]))
            inside = (q > 0) & (q < qmax)
            err = np.abs(seg - (step * q + bias))
            assert np.all(err[inside] <= step / 2 * (1 + 1e-12))
    # the dequantized matrix is within a step of the original everywhere
    assert np.all(np.abs(deq - w) <= sd * 1.01 + 1e-6)


# ---------------------------------------------------------------- expert-indexed (gather) pins

@pytest.mark.parametrize("bits", [4, 8])
def test_gather_brute_force_rational(bits):
    """Every output row of the gather oracle equals the exact rational value of
    its token row times its expert (brute force), rounded once to bf16."""
    T, E, N, K = 3, 3, 3, 64
    ew = synth.ExpertWeights(E, N, K, 70, bits=bits)
    x = synth.make_x(T, K, 71)
    lhs, rhs = synth.make_routing(T, E, 2, 72)
    y_exact, y_bf16 = oracle.gather_matmul(x, ew.w_packed, ew.scales, ew.biases, lhs, rhs, N, K, bits=bits)
    for r in range(lhs.size):
        w = synth.QuantWeights(ew.w_packed[rhs[r]], ew.scales[rhs[r]], ew.biases[rhs[r]], N, K, 64, bits)
        exact, ref_bits = brute_force(x[lhs[r]:lhs[r] + 1], w)
        assert np.array_equal(y_bf16[r], ref_bits[0]), r
        for n in range(N):
            assert abs(Fraction(y_exact[r, n]) - exact[0][n]) <= abs(exact[0][n]) * Fraction(1, 2 ** 45)


def test_gather_rows_follow_their_indices():
    """Output rows depend only on their own (token, expert) pair: reordering the
    index pairs reorders the rows, and a repeated pair repeats its row."""
    T, E, N, K = 5, 4, 6, 128
    ew = synth.ExpertWeights(E, N, K, 80)
    x = synth.make_x(T, K, 81)
    lhs, rhs = synth.make_routing(T, E, 2, 82)
    _, y = oracle.gather_matmul(x, ew.w_packed, ew.scales, ew.biases, lhs, rhs, N, K)
    perm = np.random.default_rng(0).permutation(lhs.size)
    _, yp = oracle.gather_matmul(x, ew.w_packed, ew.scales, ew.biases, lhs[perm], rhs[perm], N, K)
    assert np.array_equal(yp, y[perm])
    lhs2, rhs2 = np.concatenate([lhs, lhs[:1]]), np.concatenate([rhs, rhs[:1]])
    _, y2 = oracle.gather_matmul(x, ew.w_packed, ew.scales, ew.biases, lhs2, rhs2, N, K)
    assert np.array_equal(y2[-1], y[0])


def test_gather_sampled_matches_full():
    T, E, N, K = 6, 3, 40, 256
    ew = synth.ExpertWeights(E, N, K, 90)
    x = synth.make_x(T, K, 91)
    lhs, rhs = synth.make_routing(T, E, 2, 92)
    ye, yb = oracle.gather_matmul(x, ew.w_packed, ew.scales, ew.biases, lhs, rhs, N, K)
    rng = np.random.default_rng(1)
    ir, inn = rng.integers(0, lhs.size, 200), rng.integers(0, N, 200)
    se, sb = oracle.gather_matmul_sampled(x, ew.w_packed, ew.scales, ew.biases, lhs, rhs, N, K, ir, inn)
    assert np.array_equal(sb, yb[ir, inn])
    assert np.array_equal(se, ye[ir, inn])


def test_routing_recipe():
    T, E, k = 1000, 8, 2
    lhs, rhs = synth.make_routing(T, E, k, 5)
    assert lhs.dtype == np.int32 and rhs.dtype == np.int32 and lhs.size == T * k
    assert np.all(np.diff(rhs) >= 0)                              # sorted by expert
    for e in range(E):
        toks = lhs[rhs == e]
        assert np.all(np.diff(toks) > 0)                          # by token within an expert, no repeats
    assert np.array_equal(np.bincount(lhs, minlength=T), np.full(T, k))   # every token k times
    counts = np.bincount(rhs, minlength=E)
    assert counts.min() > 0.8 * T * k / E and counts.max() < 1.2 * T * k / E   # roughly uniform


# ---------------------------------------------------------------- NVFP4 pins

def test_e2m1_values_fixture():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "e2m1_values.txt")) if l.strip() and not l.startswith("#")]
    assert len(rows) == 16
    for code, value in rows:
        got = oracle.e2m1_to_double(int(code, 16))
        want = float(value)
        assert got == want and np.signbit(got) == np.signbit(want), (code, got, want)


def test_e4m3_matches_torch_float8():
    """Every FP8 E4M3 byte decodes as torch's float8_e4m3fn does (an independent
    implementation of the same format), NaN included."""
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_to_double(b) for b in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert oracle.e4m3_to_double(0x38) == 1.0 and oracle.e4m3_to_double(0x7E) == 448.0
    assert oracle.e4m3_to_double(0x01) == 2.0 ** -9 and oracle.e4m3_to_double(0x08) == 2.0 ** -6


def brute_force_nvfp4(x, w):
    """Exact rational value of every output (Fraction), rounded once to bf16."""
    M, K = x.shape
    e2m1 = {c: Fraction(v) for c, v in ((0, 0), (1, Fraction(1, 2)), (2, 1), (3, Fraction(3, 2)), (4, 2), (5, 3),
                                          (6, 4), (7, 6))}
    glob = Fraction(w.global_scale)
    exact = [[Fraction(0)] * w.N for _ in range(M)]
    for n in range(w.N):
        for k in range(K):
            c = (int(w.w_packed[n, k // 8]) >> (4 * (k % 8))) & 15
            mag = e2m1[c & 7]
            sb = int(w.scales[n, k // 16])
            e, m = (sb >> 3) & 15, sb & 7
            s = Fraction(m, 8) * Fraction(2) ** -6 if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
            wk = glob * s * (-mag if c & 8 else mag)
            for mm in range(M):
                exact[mm][n] += bf16_bits_to_fraction(x[mm, k]) * wk
    bits = np.array([[fraction_to_bf16_bits(v) for v in row] for row in exact], np.uint16)
    return exact, bits


@pytest.mark.parametrize("M,N,K,seed", [(1, 4, 32, 1), (2, 3, 64, 2), (1, 2, 128, 3)])
def test_nvfp4_brute_force_rational(M, N, K, seed):
    w = synth.make_nvfp4_weights(N, K, seed)
    x = synth.make_x(M, K, seed)
    exact, ref_bits = brute_force_nvfp4(x, w)
    y_exact, y_bf16 = oracle.nvfp4_matmul(x, w.w_packed, w.scales, w.global_scale, M, N, K)
    assert np.array_equal(y_bf16, ref_bits)
    for m in range(M):
        for n in range(N):
            assert abs(Fraction(y_exact[m, n]) - exact[m][n]) <= abs(exact[m][n]) * Fraction(1, 2 ** 45)


def test_nvfp4_one_hot_column_and_sampled():
    N, K = 20, 64
    w = synth.make_nvfp4_weights(N, K, 9)
    wd = oracle.nvfp4_dequant(w.w_packed, w.scales, w.global_scale, N, K)
    for k in (0, 15, 16, 63):
        x = np.zeros((1, K), np.uint16)
        x[0, k] = 0x3F80                                        # 1.0
        ye, _ = oracle.nvfp4_matmul(x, w.w_packed, w.scales, w.global_scale, 1, N, K)
        for n in range(N):
            c = (int(w.w_packed[n, k // 8]) >> (4 * (k % 8))) & 15
            want = w.global_scale * oracle.e4m3_to_double(int(w.scales[n, k // 16])) * oracle.e2m1_to_double(c)
            assert ye[0, n] == want == wd[n, k]
    x = synth.make_x(3, K, 9)
    ye, yb = oracle.nvfp4_matmul(x, w.w_packed, w.scales, w.global_scale, 3, N, K)
    im, inn = np.array([0, 2, 1, 2]), np.array([0, 19, 7, 3])
    se, sb = oracle.nvfp4_matmul_sampled(x, w.w_packed, w.scales, w.global_scale, 3, N, K, im, inn)
    assert np.array_equal(se, ye[im, inn]) and np.array_equal(sb, yb[im, inn])


def test_nvfp4_recipe():
    w = synth.make_nvfp4_weights(64, 1024, 5)
    codes = (w.w_packed[:, :, None] >> (4 * np.arange(8, dtype=np.uint32))) & 15
    assert set(np.unique(codes)) == set(range(16))                       # every E2M1 encoding drawn
    assert w.scales.min() >= 0x48 and w.scales.max() <= 0x7E             # finite, normal E4M3 scales
    assert w.global_scale == 2.0 ** -13
