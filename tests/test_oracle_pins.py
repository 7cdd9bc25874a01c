"""Pins for the CPU oracle: each check compares it with something other than
itself -- numpy's IEEE binary16 conversion, an integer-exact rounding
comparator, closed-form blocks, the pages' printed values, invariants of the
format and exact rational arithmetic on tiny inputs.

Sources (page titles): "MODEL-BASELINE-RESULTS" (fak) ACT 3 item 1 (block
format, d = maxabs/127), ACT 4 "Correctness" (round half away from zero,
0.49999997 -> 0), ACT 5 item 3 (zeros, denormals, exact halves); "Frigg"
README Finding 8 (W8A16 matmul).
"""
import os
from concurrent.futures import ThreadPoolExecutor
from fractions import Fraction

import numpy as np
import pytest

import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_facts.txt")


# ---------------------------------------------------------------------------
# independent helpers (no oracle code)
# ---------------------------------------------------------------------------
def _f32_parts(w: np.ndarray):
    """|w| = W * 2^bw exactly (w finite)."""
    u = np.abs(w.astype(np.float32)).view(np.uint32).astype(np.int64)
    e = (u >> 23) & 0xFF
    m = u & 0x7FFFFF
    W = np.where(e == 0, m, m | 0x800000)
    bw = np.where(e == 0, -149, e - 150)
    return W, bw


def _f16_parts(h: int):
    e = (h >> 10) & 0x1F
    m = h & 0x3FF
    if e == 0:
        return m, -24
    return m | 0x400, e - 25


def exact_codes(w: np.ndarray, s_bits: int) -> np.ndarray:
    """Integer-exact round-half-away(|w|/s), clamped to 127, signed.
    Valid for s/4 <= |w| <= 256*s (returns 0 below s/4 by construction)."""
    S, bs = _f16_parts(int(s_bits))
    if S == 0:
        return np.zeros(w.shape, np.int8)
    W, bw = _f32_parts(w)
    D = bw - bs
    k = np.zeros(w.shape, np.int64)
    pos = D >= 0
    num = np.where(pos, W << np.clip(D, 0, 40), W)
    den = np.where(pos, S, S << np.clip(-D, 0, 40))
    ok = (D >= -40) & (D <= 40)
    k[ok] = (2 * num[ok] + den[ok]) // (2 * den[ok])
    k = np.minimum(k, 127)
    return np.where(w < 0, -k, k).astype(np.int8)


def f16_bits_numpy(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float32).astype(np.float16).view(np.uint16)


def f16_value(h: int) -> float:
    return float(np.array([h], dtype=np.uint16).view(np.float16)[0])


# ---------------------------------------------------------------------------
# binary16 conversion: exhaustive against numpy (IEEE round-to-nearest-even)
# ---------------------------------------------------------------------------
def test_f16_encode_exhaustive(oracle):
    chunk = 1 << 24

    def run(c):
        u = np.arange(c * chunk, (c + 1) * chunk, dtype=np.uint64).astype(np.uint32)
        f = u.view(np.float32)
        with np.errstate(over="ignore", invalid="ignore"):
            ref = f.astype(np.float16).view(np.uint16)
        got = oracle.f32_to_f16(f)
        nan = np.isnan(f)
        bad = (got != ref) & ~nan
        # NaN payloads are not specified; both must be NaN with the sign kept
        badnan = nan & (((got & 0x7C00) != 0x7C00) | ((got & 0x3FF) == 0) | ((got ^ ref) & 0x8000 != 0))
        return int(bad.sum() + badnan.sum())

    with ThreadPoolExecutor(os.cpu_count() or 4) as ex:
        mism = sum(ex.map(run, range(1 << 8)))
    assert mism == 0


def test_f16_decode_exhaustive(oracle):
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = h.view(np.float16).astype(np.float64)
    got = oracle.f16_to_f64(h)
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def test_bf16_decode_exhaustive(oracle):
    import ctypes
    lib = oracle._load()
    h = np.arange(65536, dtype=np.uint32)
    ref = (h << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    got = np.array([lib.q8ref_bf16_to_f64(ctypes.c_uint16(int(v))) for v in h])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


# ---------------------------------------------------------------------------
# the code rule: integer-exact comparator, exhaustive over whole binades
# ---------------------------------------------------------------------------
EXHAUSTIVE_SCALES = [0x3C00, 0x2E67, 0x0400, 0x0003, 0x7BFF, 0x1A5B]


@pytest.mark.parametrize("s_bits", EXHAUSTIVE_SCALES)
def test_code_rule_exhaustive(oracle, s_bits):
    s = f16_value(s_bits)
    lo = np.float32(s / 4).view(np.uint32)
    hi = np.float32(min(256 * s, 3.0e38)).view(np.uint32)
    chunk = 1 << 23
    starts = range(int(lo), int(hi) + 1, chunk)

    def run(a):
        b = min(a + chunk, int(hi) + 1)
        u = np.arange(a, b, dtype=np.uint64).astype(np.uint32)
        w = u.view(np.float32)
        ref = exact_codes(w, s_bits)
        got = oracle.code(w, s_bits)
        gotn = oracle.code(-w, s_bits)
        return int((got != ref).sum() + (gotn != -ref).sum())

    with ThreadPoolExecutor(os.cpu_count() or 4) as ex:
        assert sum(ex.map(run, starts)) == 0


def test_code_rule_below_quarter_scale_is_zero(oracle):
    g = np.random.default_rng(1)
    for s_bits in EXHAUSTIVE_SCALES:
        s = f16_value(s_bits)
        w = (g.uniform(0, 0.25, 100000) * s).astype(np.float32)
        w[:3] = [0.0, np.nextafter(np.float32(s / 2), np.float32(0)), 1e-45]
        assert not oracle.code(w, s_bits).any()
        assert not oracle.code(-w, s_bits).any()
        # the tie s/2 itself goes away from zero
        half = np.float32(s / 2)
        if float(half) == s / 2:
            assert oracle.code(np.array([half]), s_bits)[0] == 1
            assert oracle.code(np.array([-half]), s_bits)[0] == -1


def test_code_zero_scale_gives_zero(oracle):
    w = np.array([0.0, 1.0, -1.0, 1e30], dtype=np.float32)
    assert not oracle.code(w, 0).any()


# ---------------------------------------------------------------------------
# values the pages print
# ---------------------------------------------------------------------------
def _golden():
    rows = []
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if line:
            rows.append(line.split())
    return rows


def test_page_facts(oracle):
    rows = _golden()
    assert len(rows) >= 10
    for r in rows:
        if r[0] == "code":
            w = np.array([np.float32(float(r[1]))])
            assert int(oracle.code(w, int(r[2], 16))[0]) == int(r[3]), r
        elif r[0] == "bytes_per_weight":
            blk, sbytes, bpw = int(r[1]), int(r[2]), float(r[3])
            q, s, _ = oracle.quantize_rows(np.zeros((1, blk), np.float32))
            assert (q.nbytes + s.nbytes) / q.size == bpw == (blk + sbytes) / blk
        elif r[0] == "scale":
            blk = synth.normal_f32((1, 32), 0, "facts") * np.float32(0.01)
            blk[0, 5] = np.float32(float(r[1]))
            q, s, fl = oracle.quantize_rows(blk)
            assert fl == 0 and int(s[0, 0]) == int(r[3], 16), r
            assert abs(int(q[0, 5])) == 127


# ---------------------------------------------------------------------------
# blocks with closed-form codes: exact halves and their neighbours
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("exp,mant", [(0, 0), (-3, 1023), (-14, 0), (-14, 517), (5, 3), (9, 1000)])
@pytest.mark.parametrize("sign", [1.0, -1.0])
def test_exact_half_blocks(oracle, exp, mant, sign):
    s_bits = ((exp + 15) << 10) | mant                   # binary16 bits, by construction
    s = np.float32(np.ldexp(1.0 + mant / 1024.0, exp))
    ks = np.arange(31) % 127
    blk = np.empty((1, 32), np.float32)
    blk[0, 0] = np.float32(127.0 * float(s) * sign)
    alt = np.where(np.arange(31) % 2 == 0, 1.0, -1.0) * sign
    blk[0, 1:] = ((ks + 0.5) * float(s) * alt).astype(np.float32)
    assert np.array_equal(blk[0, 1:].astype(np.float64), (ks + 0.5) * float(s) * alt)
    q, sb, fl = oracle.quantize_rows(blk)
    assert fl == 0 and int(sb[0, 0]) == s_bits
    expect = np.empty(32, np.int64)
    expect[0] = 127 * sign
    expect[1:] = (ks + 1) * alt                           # ties go away from zero
    assert np.array_equal(q[0].astype(np.int64), expect)
    # one ulp toward zero from each tie rounds down, one ulp away stays up
    down = np.nextafter(blk[0, 1:], np.float32(0)).astype(np.float32)
    up = np.nextafter(blk[0, 1:], np.float32(np.inf) * np.sign(blk[0, 1:])).astype(np.float32)
    b2 = blk.copy(); b2[0, 1:] = down
    q2, sb2, _ = oracle.quantize_rows(b2)
    assert int(sb2[0, 0]) == s_bits
    assert np.array_equal(q2[0, 1:].astype(np.int64), ks * alt)
    b3 = blk.copy(); b3[0, 1:] = up
    q3, _, _ = oracle.quantize_rows(b3)
    assert np.array_equal(q3[0, 1:].astype(np.int64), np.minimum(ks + 1, 127) * alt)


# ---------------------------------------------------------------------------
# special blocks
# ---------------------------------------------------------------------------
def test_zero_negzero_denormal_blocks(oracle):
    w = np.zeros((3, 64), np.float32)
    w[1, :32] = np.float32(-0.0)
    w[2, :32] = np.arange(32, dtype=np.float32) * np.float32(2.0 ** -149)
    w[2, 32:] = -np.arange(32, dtype=np.float32) * np.float32(2.0 ** -130)
    q, s, fl = oracle.quantize_rows(w)
    assert fl == 0
    assert not q.any()
    assert not s.any()          # +0 scale bits for all of them


def test_subnormal_scale_block(oracle):
    # amax/127 lands in the binary16 subnormal range: codes use the rounded scale
    # and may need the clamp
    g = np.random.default_rng(7)
    for _ in range(200):
        blk = (g.standard_normal((1, 32)) * g.uniform(1e-7, 5e-5)).astype(np.float32)
        q, s, fl = oracle.quantize_rows(blk)
        assert fl == 0
        amax = np.max(np.abs(blk))
        d32 = np.float32(amax) / np.float32(127.0)
        assert int(s[0, 0]) == int(f16_bits_numpy(d32))
        if s[0, 0]:
            assert np.array_equal(q[0], exact_codes(blk[0], int(s[0, 0])))
        else:
            assert not q.any()


def test_nonfinite_and_overflow_flags(oracle):
    w = synth.normal_f32((2, 128), 0, "flags", 0.02)
    w[0, 3] = np.nan
    w[0, 40] = np.inf
    w[1, 70] = np.float32(127.0 * 65520.0)      # amax/127 = 65520 -> binary16 inf
    w[1, 100] = np.float32(127.0 * 65504.0)     # largest finite scale: fine
    q, s, fl = oracle.quantize_rows(w, with_flags=True)
    assert fl[0, 0] == oracle.FLAG_NONFINITE and fl[0, 1] == oracle.FLAG_NONFINITE
    assert fl[1, 2] == oracle.FLAG_SCALE_OVF
    assert fl[1, 3] == 0 and int(s[1, 3]) == 0x7BFF
    for (r, b) in [(0, 0), (0, 1), (1, 2)]:
        assert int(s[r, b]) == 0 and not q[r, b * 32:(b + 1) * 32].any()
    assert fl[0, 2] == fl[0, 3] == fl[1, 0] == fl[1, 1] == 0


# ---------------------------------------------------------------------------
# invariants on every block of the stress rows and random matrices
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("which", ["stress", "normal"])
def test_quantizer_invariants(oracle, which):
    if which == "stress":
        w = synth.quant_stress_rows()
    else:
        w = synth.weights(64, 1536, 0, "inv")
    q, s, fl = oracle.quantize_rows(w, with_flags=True)
    assert not fl.any()
    rows, K = w.shape
    wb = w.reshape(rows, K // 32, 32).astype(np.float64)
    qb = q.reshape(rows, K // 32, 32).astype(np.int64)
    # scale: independent binary32 division then numpy binary16 rounding
    amax = np.max(np.abs(w.reshape(rows, K // 32, 32)), axis=2)
    d32 = (amax.astype(np.float32) / np.float32(127.0)).astype(np.float32)
    assert np.array_equal(s, f16_bits_numpy(d32))
    sv = s.view(np.float16).astype(np.float64)[:, :, None]
    normal = (s & 0x7C00) != 0
    # max |q| = 127 whenever the scale is a normal binary16
    assert np.all(np.max(np.abs(qb), axis=2)[normal] == 127)
    # sign agrees or the code is zero
    assert np.all((qb == 0) | (np.sign(qb) == np.sign(wb)))
    # quantise -> dequantise error <= d/2 for normal scales; for subnormal
    # scales the clamp can add amax - 127*s
    err = np.abs(wb - sv * qb)
    bound = np.where(normal[:, :, None], sv / 2,
                     np.maximum(sv / 2, amax[:, :, None].astype(np.float64) - 127 * sv))
    assert np.all(err <= bound)
    # codes are the integer-exact rounding against the stored scale
    for r in range(0, rows, 3):
        for b in range(K // 32):
            if s[r, b]:
                assert np.array_equal(q[r, b * 32:(b + 1) * 32],
                                      exact_codes(w[r, b * 32:(b + 1) * 32], int(s[r, b])))
    # idempotence: re-quantising the dequantised blocks gives the same codes
    wd = (sv * qb).reshape(rows, K).astype(np.float32)
    assert np.array_equal(wd.astype(np.float64), (sv * qb).reshape(rows, K))
    q2, s2, _ = oracle.quantize_rows(wd)
    keep = np.repeat(normal, 32, axis=1)
    assert np.array_equal(q2[keep], q[keep])
    assert np.array_equal(s2[normal], s[normal])


# ---------------------------------------------------------------------------
# matmul: exact rationals on tiny inputs, closed forms, the bound
# ---------------------------------------------------------------------------
def _fraction_matmul(q, s, x):
    N, K = q.shape
    M = x.shape[0]
    sv = [[Fraction(f16_value(int(v))) for v in row] for row in s]
    xv = synth.bf16_bits_to_f32(x).astype(np.float64)
    y = [[Fraction(0)] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                if q[n, k]:
                    acc += sv[n][k // 32] * int(q[n, k]) * Fraction(float(xv[m, k]))
            y[m][n] = acc
    return y


@pytest.mark.parametrize("N", [1, 2, 3, 5, 7, 33])
@pytest.mark.parametrize("K", [32, 64, 96])
@pytest.mark.parametrize("M", [1, 3])
def test_matmul_bruteforce_rational(oracle, N, K, M):
    w = synth.weights(N, K, 3, f"bf{N}.{K}")
    q, s, _ = oracle.quantize_rows(w)
    x = synth.activations(M, K, 3, f"bfx{M}.{K}")
    y, B = oracle.matmul(q, s, x)
    ref = _fraction_matmul(q, s, x)
    for m in range(M):
        for n in range(N):
            assert abs(Fraction(y[m, n]) - ref[m][n]) <= Fraction(K * 2.0 ** -52) * Fraction(B[m, n])
            assert B[m, n] >= abs(y[m, n])


def test_matmul_unit_vector(oracle):
    N, K = 40, 128
    q, s, _ = oracle.quantize_rows(synth.weights(N, K, 0, "uv"))
    for k in [0, 31, 32, 77, 127]:
        y, B = oracle.matmul(q, s, synth.unit_vector_x(K, k))
        expect = s[:, k // 32].view(np.float16).astype(np.float64) * q[:, k]
        assert np.array_equal(y[0], expect)
        assert np.array_equal(B[0], np.abs(expect))


def test_matmul_exact_case_integer(oracle):
    N, K, M = 37, 160, 4
    q, s, x = synth.exact_case(N, K, M, 0)
    y, _ = oracle.matmul(q, s, x)
    # integer arithmetic: s = 2^e, e = exp_bits - 15, x small integers
    e = ((s >> 10).astype(np.int64) - 15)
    xi = synth.bf16_bits_to_f32(x).astype(np.int64)
    ref = np.zeros((M, N), np.int64)  # in units of 2^-3
    for kb in range(K // 32):
        part = q[:, kb * 32:(kb + 1) * 32].astype(np.int64) @ xi[:, kb * 32:(kb + 1) * 32].T
        ref += (part * (2 ** (e[:, kb] + 3))[:, None]).T
    assert np.array_equal(y, ref / 8.0)


def test_matmul_rows_subset_and_threads(oracle):
    N, K, M = 300, 256, 2
    q, s, _ = oracle.quantize_rows(synth.weights(N, K, 0, "sub"))
    x = synth.activations(M, K, 0, "subx")
    y1, B1 = oracle.matmul(q, s, x)
    y4, B4 = oracle.matmul(q, s, x, threads=4)
    assert np.array_equal(y1, y4) and np.array_equal(B1, B4)
    rows = np.array([0, 5, 299])
    ys, Bs = oracle.matmul(q, s, x, rows=rows)
    assert np.array_equal(ys, y1[:, rows]) and np.array_equal(Bs, B1[:, rows])


def test_matmul_transposition_sensitivity(oracle):
    # a transposed operand or swapped index would change these values
    N, K, M = 3, 64, 2
    q = np.zeros((N, K), np.int8)
    q[0, 0] = 1; q[1, 33] = 2; q[2, 63] = -3
    s = np.full((N, K // 32), 0x3C00, np.uint16)
    s[1, 1] = 0x4000  # 2.0 for row 1, second block
    xf = np.zeros((M, K), np.float32)
    xf[0, 0] = 1; xf[0, 33] = 5; xf[1, 63] = 7; xf[1, 0] = -1
    y, B = oracle.matmul(q, s, synth.f32_to_bf16_bits(xf))
    assert np.array_equal(y, np.array([[1.0, 20.0, 0.0], [-1.0, 0.0, -21.0]]))


# ---------------------------------------------------------------------------
# GGUF Q8_0 block repack
# ---------------------------------------------------------------------------
GGUF_GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "gguf_q8_0_blocks.txt")


def _gguf_golden():
    blocks = []
    for line in open(GGUF_GOLDEN):
        line = line.split("#")[0].split()
        if not line:
            continue
        assert line[0] == "block" and len(line) == 34
        blocks.append((int(line[1], 16), [int(v) for v in line[2:]]))
    return blocks


def test_gguf_blocks_split_by_hand():
    """Bytes built here by hand (scale little endian, then the codes) split
    into the scales and codes the fixture lists."""
    import oracle
    blocks = _gguf_golden()
    raw = b"".join(d.to_bytes(2, "little") + bytes(c & 0xFF for c in codes) for d, codes in blocks)
    assert len(raw) == 34 * len(blocks)
    q, s = oracle.gguf_to_planar(np.frombuffer(raw, dtype=np.uint8), 1, 32 * len(blocks))
    assert s.tolist() == [[d for d, _ in blocks]]
    assert q.reshape(-1).tolist() == [c for _, codes in blocks for c in codes]
    # and back, byte for byte
    assert oracle.planar_to_gguf(q, s).tobytes() == raw


def test_gguf_round_trip_random_bytes():
    """Any byte string of whole blocks survives split and merge, for several
    row shapes of the same block run (the split does not depend on K)."""
    import oracle
    rng = np.random.default_rng(7)
    raw = rng.integers(0, 256, size=34 * 96, dtype=np.uint8)
    for rows, K in [(1, 3072), (3, 1024), (96, 32), (12, 256)]:
        q, s = oracle.gguf_to_planar(raw, rows, K)
        assert q.shape == (rows, K) and s.shape == (rows, K // 32)
        # block g's scale is bytes 34g, 34g+1 (little endian); its codes the next 32
        g = 37
        assert int(s.reshape(-1)[g]) == int(raw[34 * g]) | (int(raw[34 * g + 1]) << 8)
        assert q.reshape(-1)[32 * g:32 * g + 32].view(np.uint8).tolist() == raw[34 * g + 2:34 * g + 34].tolist()
        assert np.array_equal(oracle.planar_to_gguf(q, s), raw)


# ---------------------------------------------------------------------------
# compatibility code rule: half-away rounding of the binary32 quotient w / d32
# ---------------------------------------------------------------------------
def _fl32_of_fraction(r):
    """Round the rational r to the nearest binary32 value, ties to even, with
    integer arithmetic only (an implementation independent of the oracle)."""
    from fractions import Fraction
    if r == 0:
        return Fraction(0)
    sign = -1 if r < 0 else 1
    r = abs(r)
    a, b = r.numerator, r.denominator
    e = a.bit_length() - b.bit_length()
    if (a < (b << e)) if e >= 0 else ((a << -e) < b):
        e -= 1
    # 2^e <= r < 2^(e+1); quantum 2^(e-23), or 2^-149 below the normal range
    qe = max(e - 23, -149)
    num, den = (a << -qe, b) if qe <= 0 else (a, b << qe)
    m, rem = divmod(num, den)
    if 2 * rem > den or (2 * rem == den and (m & 1)):
        m += 1
    return sign * Fraction(m) * (Fraction(2) ** qe)


def _half_away_code(t):
    from fractions import Fraction
    k = int(abs(t) + Fraction(1, 2))  # floor of a non-negative rational
    k = min(k, 127)
    return -k if t < 0 else k


def test_fl32_quotient_rule_by_exact_arithmetic():
    """code_fl32 against an integer-exact re-derivation: the quotient w / d32
    rounded to binary32 (ties to even), then half away from zero, clamped."""
    import oracle
    from fractions import Fraction
    rng = np.random.default_rng(11)
    for amax in [1.0, 127.0, 0.02, 3.1, 1e-3, 7.75e-3, 250.0, 6.0e-5]:
        d32 = np.float32(np.float32(amax) / np.float32(127.0))
        w = (rng.uniform(-1.0, 1.0, size=4000) * amax).astype(np.float32)
        # plus the weights just around every half-integer multiple of d32
        halves = np.array([(k + 0.5) * float(d32) for k in range(127)], dtype=np.float32)
        w = np.concatenate([w, halves, -halves, np.nextafter(halves, np.float32(0)),
                            np.nextafter(halves, np.float32(np.inf)), np.float32([0.0, -0.0, amax, -amax])])
        got = oracle.code_fl32(w, d32)
        want = [_half_away_code(_fl32_of_fraction(Fraction(float(v)) / Fraction(float(d32)))) for v in w]
        assert got.tolist() == want, amax


def test_fl32_rule_on_page_values():
    """With d32 = 1 the binary32 quotient is the weight itself, so the page's
    rounding facts apply unchanged (0.49999997 -> 0, half away from zero)."""
    import oracle
    for kind, w, sbits, expected in _golden():
        if kind == "code" and int(sbits, 16) == 0x3C00:
            assert int(oracle.code_fl32(np.float32([float(w)]), 1.0)[0]) == int(expected), w


def test_fl32_blocks_exact_halves_closed_form():
    """Blocks whose maximum is 127 * 2^e: d32 = 2^e exactly, so a weight
    (k + 1/2) 2^e has the exact quotient k + 1/2 and the code k + 1."""
    import oracle
    for e in [-10, -3, 0, 2]:
        step = np.float32(2.0 ** e)
        ks = np.arange(31, dtype=np.float32)
        blk = np.concatenate([(ks + np.float32(0.5)) * step, [np.float32(127.0) * step]]).astype(np.float32)
        w = np.stack([blk, -blk])
        q, s, fl = oracle.quantize_rows_fl32(w)
        assert fl == 0
        want = np.concatenate([np.arange(1, 32), [127]])
        assert q[0].tolist() == want.tolist() and q[1].tolist() == (-want).tolist()
        assert int(s[0, 0]) == int(oracle.f32_to_f16(np.float32([step]))[0])


def test_fl32_blocks_match_exact_arithmetic_and_flags():
    """Whole blocks: scale as in the exact mode, codes by the exact
    re-derivation, zero / non-finite blocks as in the exact mode."""
    import oracle
    from fractions import Fraction
    w = synth.weights(6, 256, 0, "fl32.blocks")
    w[2, 32:64] = 0.0
    w[3, 0] = np.inf
    w[4, 64:96] *= np.float32(1e-38)
    q, s, fl = oracle.quantize_rows_fl32(w, with_flags=True)
    q_e, s_e, fl_e = oracle.quantize_rows(w, with_flags=True)
    assert np.array_equal(s, s_e) and np.array_equal(fl, fl_e)
    for r in range(6):
        for b in range(8):
            blk = w[r, 32 * b:32 * b + 32]
            if fl[r, b] or s[r, b] == 0:
                assert not q[r, 32 * b:32 * b + 32].any()
                continue
            d32 = np.float32(np.max(np.abs(blk)) / np.float32(127.0))
            want = [_half_away_code(_fl32_of_fraction(Fraction(float(v)) / Fraction(float(d32)))) for v in blk]
            assert q[r, 32 * b:32 * b + 32].tolist() == want


# ---------------------------------------------------------------------------
# W8A8 reference
# ---------------------------------------------------------------------------
def _bf16_bits(v):
    return (np.asarray(v, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def test_w8a8_integer_activations_reduce_to_w8a16(oracle):
    """Activations that are integers in [-127, 127] with 127 in every block
    quantize to themselves (scale 1, codes = values), so W8A8 equals the
    W8A16 reference on them."""
    rng = np.random.default_rng(7)
    N, K, M = 37, 128, 3
    q, s, _ = oracle.quantize_rows(synth.weights(N, K, 0, "w8a8i"))
    xv = rng.integers(-126, 127, size=(M, K)).astype(np.float32)
    xv[:, ::32] = 127.0
    y8, B8 = oracle.matmul_w8a8(q, s, _bf16_bits(xv))
    y16, B16 = oracle.matmul(q, s, _bf16_bits(xv))
    assert np.allclose(y8, y16, rtol=1e-13, atol=0)
    assert np.allclose(B8, B16, rtol=1e-13, atol=0)


def test_w8a8_brute_force_exact(oracle):
    """Tiny random case against exact rational arithmetic written out block
    by block (each activation block's scale and codes from the Q8_0 rule of
    its binary32 values): a transposed scale or a wrong block index fails."""
    N, K, M = 3, 64, 2
    q, s, _ = oracle.quantize_rows(synth.weights(N, K, 0, "w8a8b"))
    x = synth.activations(M, K, 0, "w8a8bx")
    xf = (x.astype(np.uint32) << 16).view(np.float32)
    qx, sx, _ = oracle.quantize_rows(xf)
    y, _ = oracle.matmul_w8a8(q, s, x)
    f16 = lambda bits: Fraction(float(np.uint16(bits).view(np.float16)))
    for m in range(M):
        for n in range(N):
            exact = sum(f16(s[n, b]) * f16(sx[m, b]) *
                        sum(int(q[n, k]) * int(qx[m, k]) for k in range(32 * b, 32 * b + 32))
                        for b in range(K // 32))
            assert abs(y[m, n] - float(exact)) <= 1e-12 * max(1.0, abs(float(exact)))
