"""Pins of the CPU oracle against things other than the oracle itself.

Each check here is independent of the oracle's own formulas: golden values
fixed by the public format definitions or derived by hand from the recipe,
a library routine (torch's float8_e4m3fn casts), brute-force nearest-value
search with an explicit tie rule, exact rational arithmetic
(fractions.Fraction), closed forms and invariants.  Together they are chosen
so that a dropped term, a wrong sign, index or nibble order, a transposed
operand or a wrong rounding rule in the oracle fails at least one of them
(tests/test_oracle_mutants.py plants such mistakes and checks that).
"""
import math
import random
from fractions import Fraction

import numpy as np
import torch

from conftest import read_golden


def _golden_table(name):
    out = {}
    for code, val in read_golden(name):
        out[int(code, 16)] = float(val)
    return out


E2M1 = _golden_table("e2m1_codes.txt")
E4M3_T = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
E4M3_POS = np.array([E4M3_T[b] for b in range(0x7F)])        # finite, >= 0
E2M1_POS = np.array([E2M1[c] for c in range(8)])


def _same(a, b):
    if math.isnan(a) or math.isnan(b):
        return math.isnan(a) and math.isnan(b)
    return a == b and math.copysign(1, a) == math.copysign(1, b)


def _bits_to_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def _bf16_values(bits):
    return _bits_to_bf16(bits).double().numpy()


# -------------------------------------------------------------- brute force

def _nearest_code(a, table):
    """Brute-force nearest of |a| in table[code]; a tie goes to the even code."""
    d = np.abs(table - a)
    best = d.min()
    cands = np.nonzero(d == best)[0]
    even = [c for c in cands if c % 2 == 0]
    return int(even[0] if even else cands[0])


def bf_e4m3(v):
    v = float(np.float32(v))
    sign = 0x80 if math.copysign(1, v) < 0 else 0
    a = abs(v)
    if a >= 448.0:
        return sign | 0x7E
    return sign | _nearest_code(a, E4M3_POS)


def bf_e2m1(v):
    v = float(np.float32(v))
    sign = 8 if math.copysign(1, v) < 0 else 0
    a = abs(v)
    if a > 6.0:
        return sign | 7
    return sign | _nearest_code(a, E2M1_POS)


# ------------------------------------------------------------------ decode

def test_e2m1_golden(orc):
    assert len(E2M1) == 16
    for code, v in E2M1.items():
        assert _same(orc.e2m1_value(code), v), hex(code)


def test_e4m3_golden(orc):
    for b, v in _golden_table("e4m3_codes.txt").items():
        assert _same(orc.e4m3_value(b), v), hex(b)


def test_e4m3_all_codes_match_torch(orc):
    for b in range(256):
        assert _same(orc.e4m3_value(b), float(E4M3_T[b])), hex(b)


def test_e4m3_invariants(orc):
    vals = [orc.e4m3_value(b) for b in range(0x7F)]
    assert all(vals[i] < vals[i + 1] for i in range(len(vals) - 1))
    assert vals[-1] == 448.0 and vals[1] == 2.0 ** -9 and vals[0] == 0.0
    assert math.isnan(orc.e4m3_value(0x7F)) and math.isnan(orc.e4m3_value(0xFF))
    for b in range(0x7F):
        assert _same(orc.e4m3_value(b | 0x80), -vals[b])


def test_bf16_decode_matches_torch(orc):
    rng = np.random.default_rng(5)
    bits = rng.integers(0, 1 << 16, size=3000, dtype=np.uint16)
    ref = _bf16_values(bits)
    for b, r in zip(bits, ref):
        assert _same(orc.bf16_value(int(b)), float(r))


# ------------------------------------------------------------------ encode

def test_e4m3_encode_identity_on_codes(orc):
    for b in list(range(0x7F)) + list(range(0x80, 0xFF)):
        assert orc.e4m3_encode(orc.e4m3_value(b)) == b, hex(b)


def test_e4m3_encode_midpoints_go_to_even(orc):
    for b in range(0x7E):
        lo, hi = E4M3_T[b], E4M3_T[b + 1]
        mid = (lo + hi) / 2
        assert float(np.float32(mid)) == mid
        want = b if b % 2 == 0 else b + 1
        assert orc.e4m3_encode(mid) == want
        assert orc.e4m3_encode(-mid) == want | 0x80
        below = float(np.nextafter(np.float32(mid), np.float32(0)))
        above = float(np.nextafter(np.float32(mid), np.float32(1e9)))
        assert orc.e4m3_encode(below) == b
        assert orc.e4m3_encode(above) == b + 1


def test_e4m3_encode_bruteforce_random(orc):
    rnd = random.Random(11)
    vals = [0.0, -0.0, 448.0, 449.0, 464.0, 480.0, 1e30, -1e30, float("inf"),
            2.0 ** -10, 2.0 ** -9, 1.5 * 2.0 ** -10, 3e-45]
    vals += [rnd.choice([-1, 1]) * 2.0 ** rnd.uniform(-13, 10) for _ in range(20000)]
    for v in vals:
        assert orc.e4m3_encode(v) == bf_e4m3(v), v


def test_e4m3_encode_matches_torch_in_range(orc):
    rng = np.random.default_rng(3)
    v = (rng.standard_normal(20000) * 60).astype(np.float32)
    v = v[np.abs(v) <= 448]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for x, r in zip(v, ref):
        assert orc.e4m3_encode(float(x)) == int(r), x


def test_e2m1_encode_bruteforce(orc):
    rnd = random.Random(12)
    vals = [0.0, -0.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 7.0, 1e9]
    for lo, hi in zip([0, .5, 1, 1.5, 2, 3, 4], [.5, 1, 1.5, 2, 3, 4, 6]):
        m = (lo + hi) / 2
        vals += [m, float(np.nextafter(np.float32(m), np.float32(0))),
                 float(np.nextafter(np.float32(m), np.float32(9)))]
    vals += [rnd.uniform(-8, 8) for _ in range(20000)]
    for v in vals:
        assert orc.e2m1_encode(v) == bf_e2m1(v), v
        assert orc.e2m1_encode(-v) == bf_e2m1(-v), -v


# -------------------------------------------------------- golden examples

def _parse_example(name):
    d = {"w": [], "codes": []}
    for r in read_golden(name):
        if r[0] in ("w", "codes"):
            d[r[0]].append(r[1:])
        else:
            d[r[0]] = r[1:]
    return d


def _nibble(nib, m, k):
    return (int(nib[m, k // 2]) >> (4 * (k % 2))) & 15


def test_nvfp4_golden_example(orc):
    ex = _parse_example("nvfp4_example.txt")
    W = np.array([[float(v) for blk in ex["w"] for v in blk]], np.float32)
    assert W.shape == (1, int(ex["K"][0]))
    nib, sc, gs = orc.nvfp4_quantise(W)
    assert gs == float(ex["gs"][0])
    assert [int(s) for s in sc[0]] == [int(s, 16) for s in ex["scales"]]
    codes = [int(c, 16) for blk in ex["codes"] for c in blk]
    assert [_nibble(nib, 0, k) for k in range(W.shape[1])] == codes
    x = np.full((1, W.shape[1]), 0x3F80, np.uint16)            # BF16 1.0
    y, a = orc.gemv_nvfp4(nib, sc, gs, x)
    assert y[0, 0] == float(ex["y_ones"][0])
    assert a[0, 0] == float(ex["a_ones"][0])


def test_fp8_golden_example(orc):
    ex = _parse_example("fp8_example.txt")
    W = np.array([[float(v) for v in r] for r in ex["w"]], np.float32)
    q, rs = orc.fp8_quantise(W)
    assert rs[0] == float(ex["rs"][0]) and rs[2] == 0.0
    for m, row in enumerate(ex["codes"]):
        assert [int(c) for c in q[m]] == [int(c, 16) for c in row], m


# ------------------------------------------------------ quantiser pinning

def _rand_w(seed, M, K, std=0.02):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn((M, K), generator=g) * std).numpy()


def test_nvfp4_quantiser_decisions_bruteforce(orc):
    W = _rand_w(21, 8, 96)
    W[3, 16:32] = 0.0                                  # a zero block
    W[5, 32:48] *= 1e-5                                # a subnormal-scale block
    nib, sc, gs = orc.nvfp4_quantise(W)
    f32 = np.float32
    assert gs == f32(np.abs(W).max()) / f32(2688.0)
    assert sc[3, 1] == 0 and sc[5, 2] < 8              # zero and subnormal scale
    for m in range(W.shape[0]):
        for b in range(W.shape[1] // 16):
            blk = W[m, 16 * b:16 * b + 16]
            s = (f32(np.abs(blk).max()) / f32(gs)) / f32(6.0)
            assert sc[m, b] == bf_e4m3(s), (m, b)
            d = f32(E4M3_T[sc[m, b]]) * f32(gs)
            for j, w in enumerate(blk):
                want = 0 if d == 0 else bf_e2m1(f32(w) / d)
                assert _nibble(nib, m, 16 * b + j) == want, (m, b, j)


def test_nvfp4_quantiser_invariants(orc):
    W = _rand_w(22, 16, 256)
    nib, sc, gs = orc.nvfp4_quantise(W)
    What = orc.nvfp4_dequant(nib, sc, gs, *W.shape)
    for m in range(W.shape[0]):
        for b in range(W.shape[1] // 16):
            d = E4M3_T[sc[m, b]] * gs
            q = W[m, 16 * b:16 * b + 16] / d
            deq = What[m, 16 * b:16 * b + 16] / d
            # every element within the largest half-gap of the E2M1 grid
            assert np.all(np.abs(q - deq) <= 1.0 + 1e-6)
            # the block maximum lands on the top of the grid (magnitude code 7)
            j = int(np.argmax(np.abs(W[m, 16 * b:16 * b + 16])))
            assert _nibble(nib, m, 16 * b + j) & 7 == 7
    # power-of-two scaling of W scales gs and leaves every code unchanged
    nib2, sc2, gs2 = orc.nvfp4_quantise(W * np.float32(8.0))
    assert gs2 == gs * 8 and np.array_equal(nib, nib2) and np.array_equal(sc, sc2)


def test_nvfp4_requantise_is_idempotent(orc):
    for seed in range(4):
        W = _rand_w(30 + seed, 8, 128)
        nib, sc, gs = orc.nvfp4_quantise(W)
        W2 = orc.nvfp4_dequant(nib, sc, gs, *W.shape).astype(np.float32)
        nib2, sc2, gs2 = orc.nvfp4_quantise(W2)
        assert gs2 == gs and np.array_equal(sc, sc2) and np.array_equal(nib, nib2)


def test_fp8_quantiser_decisions_and_invariants(orc):
    W = _rand_w(23, 6, 64)
    W[2] = 0.0
    q, rs = orc.fp8_quantise(W)
    f32 = np.float32
    for m in range(W.shape[0]):
        assert rs[m] == f32(np.abs(W[m]).max()) / f32(448.0)
        for k in range(W.shape[1]):
            want = 0 if rs[m] == 0 else bf_e4m3(f32(W[m, k]) / rs[m])
            assert q[m, k] == want
        if rs[m] > 0:
            assert (q[m, int(np.argmax(np.abs(W[m])))] & 0x7F) == 0x7E
    W2 = orc.fp8_dequant(q, rs, *W.shape).astype(np.float32)
    q2, rs2 = orc.fp8_quantise(W2)
    assert np.array_equal(rs, rs2) and np.array_equal(q, q2)


# --------------------------------------------------------------- the GEMV

def _x_bits(seed, N, K, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn((N, K), generator=g) * scale).to(torch.bfloat16)
    return x.view(torch.int16).numpy().view(np.uint16)


def _exact(wv, x_bits):
    """Exact rational y[n][m], a[n][m] from Fraction weights wv[m][k]."""
    xv = _bf16_values(x_bits)
    xs = [[Fraction(float(v)) for v in row] for row in xv]
    N, M, K = len(xs), len(wv), len(wv[0])
    y = [[sum(wv[m][k] * xs[n][k] for k in range(K)) for m in range(M)] for n in range(N)]
    a = [[sum(abs(wv[m][k] * xs[n][k]) for k in range(K)) for m in range(M)]
         for n in range(N)]
    return y, a


def test_gemv_nvfp4_bruteforce_4x16(orc):
    for seed in range(3):
        M, K, N = 4, 16, 3
        W = _rand_w(40 + seed, M, K)
        nib, sc, gs = orc.nvfp4_quantise(W)
        x = _x_bits(50 + seed, N, K)
        y, a = orc.gemv_nvfp4(nib, sc, gs, x)
        # weights decoded from the golden tables, exact rationals
        wv = [[Fraction(E2M1[_nibble(nib, m, k)]) * Fraction(float(E4M3_T[sc[m, k // 16]]))
               * Fraction(gs) for k in range(K)] for m in range(M)]
        ye, ae = _exact(wv, x)
        u = 2.0 ** -53
        for n in range(N):
            for m in range(M):
                assert abs(Fraction(y[n, m]) - ye[n][m]) <= (K - 1) * u * ae[n][m]
                assert abs(Fraction(a[n, m]) - ae[n][m]) <= (K - 1) * u * ae[n][m]


def test_gemv_fp8_bruteforce_4x16(orc):
    M, K, N = 4, 16, 2
    W = _rand_w(44, M, K)
    q, rs = orc.fp8_quantise(W)
    x = _x_bits(54, N, K)
    y, a = orc.gemv_fp8(q, rs, x)
    wv = [[Fraction(float(E4M3_T[q[m, k]])) * Fraction(float(rs[m])) for k in range(K)]
          for m in range(M)]
    ye, ae = _exact(wv, x)
    for n in range(N):
        for m in range(M):
            assert abs(Fraction(y[n, m]) - ye[n][m]) <= (K - 1) * 2.0 ** -53 * ae[n][m]
            assert abs(Fraction(a[n, m]) - ae[n][m]) <= (K - 1) * 2.0 ** -53 * ae[n][m]


def test_gemv_rows_columns_and_threads_are_independent(orc):
    W = _rand_w(45, 32, 64)
    nib, sc, gs = orc.nvfp4_quantise(W)
    x = _x_bits(55, 5, 64)
    y, a = orc.gemv_nvfp4(nib, sc, gs, x)
    rows = np.array([31, 0, 7, 7], np.int64)
    ys, as_ = orc.gemv_nvfp4(nib, sc, gs, x[2:4], rows=rows)
    assert np.array_equal(ys, y[2:4][:, rows]) and np.array_equal(as_, a[2:4][:, rows])
    y4, _ = orc.gemv_nvfp4(nib, sc, gs, x, threads=4)
    assert np.array_equal(y4, y)


def test_gemv_linearity_in_x(orc):
    M, K = 16, 128
    W = _rand_w(46, M, K)
    nib, sc, gs = orc.nvfp4_quantise(W)
    x1 = _bits_to_bf16(_x_bits(56, 1, K))
    x2 = _bits_to_bf16(_x_bits(57, 1, K))
    mask = torch.arange(K) % 3 == 0
    x1 = torch.where(mask, x1, torch.zeros_like(x1))
    x2 = torch.where(mask, torch.zeros_like(x2), x2)
    alpha, beta = 4.0, -0.25
    xs = (alpha * x1.float() + beta * x2.float()).to(torch.bfloat16)
    assert torch.equal(xs.float(), alpha * x1.float() + beta * x2.float())

    def bits(t):
        return t.view(torch.int16).numpy().view(np.uint16)

    y1, a1 = orc.gemv_nvfp4(nib, sc, gs, bits(x1))
    y2, a2 = orc.gemv_nvfp4(nib, sc, gs, bits(x2))
    ys, _ = orc.gemv_nvfp4(nib, sc, gs, bits(xs))
    bound = K * 2.0 ** -52 * (abs(alpha) * a1 + abs(beta) * a2)
    assert np.all(np.abs(ys - (alpha * y1 + beta * y2)) <= bound)


def test_gemv_zero_block_contributes_nothing(orc):
    M, K = 8, 64
    W = _rand_w(47, M, K)
    W[:, 16:32] = 0.0
    nib, sc, gs = orc.nvfp4_quantise(W)
    assert np.all(sc[:, 1] == 0) and np.all(nib[:, 8:16] == 0)
    x = _x_bits(58, 2, K)
    x0 = x.copy()
    x0[:, 16:32] = 0
    y, _ = orc.gemv_nvfp4(nib, sc, gs, x)
    y0, _ = orc.gemv_nvfp4(nib, sc, gs, x0)
    assert np.array_equal(y, y0)
    # an all-zero matrix gives gs = 0, zero codes and y = 0
    nibz, scz, gsz = orc.nvfp4_quantise(np.zeros((3, 32), np.float32))
    assert gsz == 0.0 and not nibz.any() and not scz.any()
    yz, az = orc.gemv_nvfp4(nibz, scz, gsz, x[:, :32])
    assert not yz.any() and not az.any()


def test_gemv_all_max_nibble_closed_form(orc):
    M, K, N = 3, 64, 2
    nib = np.full((M, K // 2), 0x77, np.uint8)
    sc = np.full((M, K // 16), 0x7E, np.uint8)
    gs = 0.03125
    x = _x_bits(59, N, K)
    y, a = orc.gemv_nvfp4(nib, sc, gs, x)
    xv = _bf16_values(x)
    for n in range(N):
        want = 2688.0 * gs * math.fsum(xv[n])
        wanta = 2688.0 * gs * math.fsum(np.abs(xv[n]))
        assert np.all(np.abs(y[n] - want) <= K * 2.0 ** -53 * wanta)
        assert np.all(np.abs(a[n] - wanta) <= K * 2.0 ** -53 * wanta)


def test_gemv_textbook_reduction(orc):
    """Scales 1.0 (0x38) and gs = 1: y equals numpy's float64 x @ e2m1(W).T."""
    rng = np.random.default_rng(60)
    M, K, N = 12, 64, 3
    codes = rng.integers(0, 16, size=(M, K))
    nib = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    sc = np.full((M, K // 16), 0x38, np.uint8)
    x = _x_bits(61, N, K)
    y, _ = orc.gemv_nvfp4(nib, sc, 1.0, x)
    wv = np.vectorize(lambda c: E2M1[int(c)])(codes).astype(np.float64)
    assert np.array_equal(y, _bf16_values(x) @ wv.T)


def test_gemv_fp8_textbook_reduction(orc):
    """Row scales 1.0: y equals numpy's float64 x @ e4m3(Q).T."""
    rng = np.random.default_rng(62)
    M, K, N = 10, 48, 2
    q = rng.integers(0, 256, size=(M, K)).astype(np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x01                       # no NaN codes
    rs = np.ones(M, np.float32)
    x = _x_bits(63, N, K, scale=0.25)
    y, _ = orc.gemv_fp8(q, rs, x)
    assert np.array_equal(y, _bf16_values(x) @ E4M3_T[q].T)


def test_check_counts_out_of_tolerance(orc):
    yref = np.array([1.0, -2.0, 100.0, 0.0])
    a = np.array([10.0, 10.0, 1000.0, 0.0])
    ok = torch.tensor(yref, dtype=torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    bad, worst = orc.check(ok, yref, a)
    assert bad == 0 and worst <= 1.0
    off = ok.copy()
    off[2] = torch.tensor([104.5], dtype=torch.bfloat16).view(torch.int16).numpy().view(
        np.uint16)[0]
    bad, worst = orc.check(off, yref, a)          # 4.5 > 4e-3*1000 + 1e-6
    assert bad == 1 and worst > 1.0


def test_quantise_rows_with_given_gs_matches_whole_matrix(orc):
    W = _rand_w(70, 40, 96)
    nib, sc, gs = orc.nvfp4_quantise(W)
    assert orc.amax(W) == np.abs(W).max()
    rows = [0, 17, 39]
    nr, sr = orc.nvfp4_quantise_gs(W[rows], gs)
    assert np.array_equal(nr, nib[rows]) and np.array_equal(sr, sc[rows])


# ------------------------------------------------------- fused neighbours

def test_bf16_round_matches_torch_on_fp32_values(orc):
    """For FP32 inputs one FP64 rounding equals torch's FP32 -> BF16 cast
    (round to nearest even), across normal, subnormal and huge values."""
    rng = np.random.default_rng(11)
    vals = np.concatenate([rng.standard_normal(4000).astype(np.float32),
                           (rng.standard_normal(2000) * 1e-39).astype(np.float32),
                           (rng.standard_normal(2000) * 1e37).astype(np.float32),
                           np.float32([0.0, -0.0, 1.0, -2.5, 3e38, -3.3e38])])
    want = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([orc.bf16_round(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, want)


def test_bf16_round_midpoints_and_edges(orc):
    """Midpoints between neighbouring BF16 values go to the even
    significand; a hair above or below goes to the nearer one; the
    subnormal spacing is 2^-133; past the largest finite value is inf."""
    rng = np.random.default_rng(12)
    for b in rng.integers(0x0001, 0x7F7E, 500):
        lo, hi = orc.bf16_value(int(b)), orc.bf16_value(int(b) + 1)
        mid = (lo + hi) / 2                       # exact in FP64
        even = int(b) if int(b) % 2 == 0 else int(b) + 1
        assert orc.bf16_round(mid) == even
        assert orc.bf16_round(-mid) == even | 0x8000
        assert orc.bf16_round(np.nextafter(mid, 0)) == int(b)
        assert orc.bf16_round(np.nextafter(mid, np.inf)) == int(b) + 1
    assert orc.bf16_round(2.0 ** -133) == 0x0001
    assert orc.bf16_round(2.0 ** -134) == 0x0000        # tie with 0: even
    assert orc.bf16_round(3 * 2.0 ** -134) == 0x0002    # tie between 1 and 2: even
    assert orc.bf16_round(orc.bf16_value(0x7F7F)) == 0x7F7F
    assert orc.bf16_round(2.0 ** 128) == 0x7F80
    assert orc.bf16_round(-0.0) == 0x8000


def test_silu_against_library_sigmoid(orc):
    """SiLU(g) = g * sigmoid(g), with scipy's expit as the sigmoid, and the
    identity SiLU(g) - SiLU(-g) = g."""
    from scipy.special import expit

    for g in np.linspace(-30, 30, 241):
        want = g * expit(g)
        assert abs(orc.silu(g) - want) <= 1e-15 * max(1.0, abs(want))
        assert abs(orc.silu(g) - orc.silu(-g) - g) <= 1e-14 * max(1.0, abs(g))
    assert orc.silu(0.0) == 0.0


def test_swiglu_values_and_bound(orc):
    """h = SiLU(gate) * up (the gate goes through SiLU, not the up), and
    the bound grows with both products' scales and with |h|."""
    from scipy.special import expit

    g = np.array([2.0, 3.0, -1.5, 0.0, 10.0])
    u = np.array([3.0, 2.0, 4.0, 7.0, -0.5])
    zero = np.zeros_like(g)
    h, b = orc.swiglu(g, u, zero, zero)
    assert np.allclose(h, g * expit(g) * u, rtol=1e-15, atol=0)
    assert h[0] != h[1]                                  # not symmetric in gate/up
    assert np.allclose(b, np.abs(h) / 256 + 1.1e-6 * (np.abs(u) + 1e-6)
                       + np.abs(g * expit(g)) * 1e-6 + 1e-6, rtol=1e-12)
    _, b2 = orc.swiglu(g, u, zero + 1.0, zero)
    _, b3 = orc.swiglu(g, u, zero, zero + 1.0)
    assert np.all(b2 > b) and np.all(b3 >= b)


def test_rmsnorm_against_library(orc):
    """RMS normalisation against torch's rms_norm in FP64, rounded once to
    BF16 (the rounding pinned above), at K of a layer and with outliers."""
    rng = np.random.default_rng(13)
    for N, K, scale in ((1, 5120, 1.0), (8, 512, 30.0), (3, 17408, 1e-3)):
        x = torch.from_numpy(rng.standard_normal((N, K)) * scale).to(torch.bfloat16)
        x[:, rng.integers(0, K, 4)] *= 20
        gamma = torch.from_numpy(1 + 0.1 * rng.standard_normal(K)).to(torch.bfloat16)
        ref = torch.nn.functional.rms_norm(x.double(), (K,), gamma.double(), eps=1e-6)
        want = np.array([[orc.bf16_round(v) for v in row] for row in ref.numpy()],
                        dtype=np.uint16)
        xb = x.view(torch.int16).numpy().view(np.uint16)
        gb = gamma.view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(orc.rmsnorm(xb, gb, 1e-6), want)


def test_rmsnorm_closed_forms(orc):
    """A constant row c gives gamma * c / sqrt(c^2 + eps); with eps = 0 a
    power-of-two scale of x leaves the output unchanged."""
    K = 256
    gamma = torch.linspace(0.5, 2.0, K).to(torch.bfloat16)
    gb = gamma.view(torch.int16).numpy().view(np.uint16)
    x = torch.full((1, K), 3.0).to(torch.bfloat16)
    out = orc.rmsnorm(x.view(torch.int16).numpy().view(np.uint16), gb, 1e-6)
    want = [orc.bf16_round(orc.bf16_value(int(gv)) * 3.0 / np.sqrt(9.0 + 1e-6)) for gv in gb]
    assert np.array_equal(out[0], np.array(want, dtype=np.uint16))
    rng = np.random.default_rng(14)
    x = torch.from_numpy(rng.standard_normal((2, K))).to(torch.bfloat16)
    a = orc.rmsnorm(x.view(torch.int16).numpy().view(np.uint16), gb, 0.0)
    b = orc.rmsnorm((x * 8).view(torch.int16).numpy().view(np.uint16), gb, 0.0)
    assert np.array_equal(a, b)


# ---------------------------------------------------------- other formats

def test_e8m0_values(orc):
    """E8M0 is a bare exponent: 2^(e-127), 0xFF NaN (OCP Microscaling)."""
    assert orc.e8m0_value(127) == 1.0
    assert orc.e8m0_value(0) == 2.0 ** -127
    assert orc.e8m0_value(254) == 2.0 ** 127
    assert orc.e8m0_value(130) == 8.0
    assert math.isnan(orc.e8m0_value(255))


def test_mxfp8_quantiser_decisions(orc):
    """Per 32-block: the scale puts the block amax in [256, 512) (shared
    exponent floor(log2 amax) - 8) unless the scale range clamps it; every
    code is the nearest E4M3 value to w / X by brute force over all finite
    codes, ties to the even code, saturating at 448; a zero block gets
    scale 1 and zero codes."""
    rng = np.random.default_rng(21)
    W = (rng.standard_normal((6, 256)) * rng.choice([1e-3, 0.02, 3.0, 1e3], (6, 1))) \
        .astype(np.float32)
    W[1, 32:64] = 0.0
    q, sc = orc.mxfp8_quantise(W)
    finite = [(orc.e4m3_value(c), c) for c in range(256) if not math.isnan(orc.e4m3_value(c))]
    for m in range(6):
        for b in range(8):
            blk = W[m, 32 * b:32 * b + 32]
            e = int(sc[m, b])
            amax = float(np.abs(blk).max())
            if amax == 0:
                assert e == 127 and not q[m, 32 * b:32 * b + 32].any()
                continue
            X = 2.0 ** (e - 127)
            if 10 < e < 134:
                assert 256 <= amax / X < 512
            for j in range(32):
                v = float(np.float32(blk[j]) / np.float32(X))
                best = min(finite, key=lambda t: (abs(t[0] - v), t[1] & 1))
                want = best[1] if abs(v) < 448 else (0x7E | (0x80 if v < 0 else 0))
                if best[0] == 0 and v < 0:
                    want = 0x80
                assert q[m, 32 * b + j] == want, (m, b, j, v)


def test_mxfp8_textbook_reduction(orc):
    """With every scale byte 127 (X = 1) the product is plain FP8: numpy
    x @ e4m3(q).T in float64, exactly; other scale bytes multiply their
    32-block by 2^(e-127)."""
    rng = np.random.default_rng(22)
    M, K, N = 5, 128, 3
    q = rng.integers(0, 256, (M, K)).astype(np.uint8)
    q[(q & 0x7F) == 0x7F] = 0
    sc = np.full((M, K // 32), 127, np.uint8)
    x = torch.from_numpy(rng.standard_normal((N, K))).to(torch.bfloat16)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    y, _ = orc.gemv_mxfp8(q, sc, xb)
    Wd = np.vectorize(orc.e4m3_value)(q)
    assert np.array_equal(y, x.double().numpy() @ Wd.T)
    assert np.array_equal(orc.mxfp8_dequant(q, sc, M, K), Wd)
    pw = rng.integers(-4, 5, (M, K // 32))
    sc = (127 + pw).astype(np.uint8)
    Ws = Wd * np.repeat(2.0 ** pw, 32, axis=1)
    assert np.array_equal(orc.mxfp8_dequant(q, sc, M, K), Ws)
    y, _ = orc.gemv_mxfp8(q, sc, xb)
    assert np.array_equal(y, x.double().numpy() @ Ws.T)


def test_int4g_quantiser_decisions(orc):
    """Per 128-group: the scale is BF16(amax / 7); each code is the integer
    nearest to w / s (ties to even) clamped to -8..7, plus the zero point 8,
    by brute force over the 16 codes; a zero group stores scale 0 and 8s."""
    rng = np.random.default_rng(23)
    W = (rng.standard_normal((4, 512)) * 0.02).astype(np.float32)
    W[2, 128:256] = 0.0
    W[3, 5] = 1.0                     # one large value: most of its group rounds to 0
    nib, sc = orc.int4g_quantise(W)
    codes = np.empty((4, 512), np.int64)
    codes[:, 0::2] = nib & 15
    codes[:, 1::2] = nib >> 4
    for m in range(4):
        for g in range(4):
            blk = W[m, 128 * g:128 * g + 128]
            s = orc.bf16_value(int(sc[m, g]))
            amax = np.float32(np.abs(blk).max())
            assert sc[m, g] == orc.bf16_round(float(amax / np.float32(7.0)))
            for j in range(128):
                if s == 0:
                    assert codes[m, 128 * g + j] == 8
                    continue
                r = float(np.float32(blk[j]) / np.float32(s))
                best = min(range(-8, 8), key=lambda c: (abs(c - r), c & 1))
                assert codes[m, 128 * g + j] == best + 8, (m, g, j, r)


def test_int4g_textbook_reduction(orc):
    """With power-of-two group scales the weights are the integers q - 8
    times each group's scale, and the product is numpy x @ W.T in float64,
    exactly (a scale of 1 everywhere gives the plain integer product)."""
    rng = np.random.default_rng(24)
    M, K, N = 4, 512, 3
    nib = rng.integers(0, 256, (M, K // 2)).astype(np.uint8)
    x = torch.from_numpy(rng.standard_normal((N, K))).to(torch.bfloat16)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    Wi = np.empty((M, K))
    Wi[:, 0::2] = (nib & 15).astype(np.int64) - 8
    Wi[:, 1::2] = (nib >> 4).astype(np.int64) - 8
    sc = np.full((M, K // 128), 0x3F80, np.uint16)          # 1.0
    y, _ = orc.gemv_int4g(nib, sc, xb)
    assert np.array_equal(y, x.double().numpy() @ Wi.T)
    pw = rng.integers(-3, 4, (M, K // 128))
    sc = (0x3F80 + (pw << 7)).astype(np.uint16)             # 2^pw
    Ws = Wi * np.repeat(2.0 ** pw, 128, axis=1)
    assert np.array_equal(orc.int4g_dequant(nib, sc, M, K), Ws)
    y, _ = orc.gemv_int4g(nib, sc, xb)
    assert np.array_equal(y, x.double().numpy() @ Ws.T)
