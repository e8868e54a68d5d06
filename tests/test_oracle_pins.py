"""Pins for the CPU oracle: each function is held to something other than itself.

* packing: hand-worked words (golden file) and the pack/unpack round trip;
* dequantization: hand-worked values (golden file), an exhaustive (q, z) x
  scale sweep against exact rational round-to-nearest-even, and closed-form
  cases that fail on a wrong group or column index;
* the product: exact rational brute force at K = 8, the fp32 accumulation
  bound, and closed-form special cases (zero weights, one-hot copy);
* W4A8: hand-worked quantization examples (golden file), invariants of the
  per-token scale, and brute-force integer sums.
"""

import os
from fractions import Fraction
from math import floor

import numpy as np

import oracle
from bit_weight_only_awq_gb300 import synth


# ---------------------------------------------------------------- helpers
def fp16_rn_exact(v: Fraction) -> Fraction:
    """IEEE binary16 round-to-nearest-even of an exact rational (finite range only)."""
    if v == 0:
        return Fraction(0)
    sign = -1 if v < 0 else 1
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -14)                      # subnormals share the 2^-24 spacing
    ulp = Fraction(2) ** (e - 10)
    m = a / ulp
    f = floor(m)
    r = m - f
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and f % 2 == 1):
        f += 1
    return sign * f * ulp


def half_from_hex(h: int) -> np.float16:
    return np.array([h], dtype=np.uint16).view(np.float16)[0]


def read_golden(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as fh:
        return [ln.strip() for ln in fh if ln.strip() and not ln.startswith("#")]


# ---------------------------------------------------------------- packing
def test_unpack_pack_golden(golden_dir):
    n_unpack = n_pack = 0
    for line in read_golden(golden_dir, "awq_order_words.txt"):
        kind, rest = line.split(None, 1)
        lhs, rhs = (s.strip() for s in rest.split(":"))
        if kind == "unpack":
            word = np.array([[int(lhs, 16)]], dtype=np.uint32).view(np.int32)
            want = [int(t) for t in rhs.split()]
            assert oracle.unpack(word)[0].tolist() == want, line
            n_unpack += 1
        else:
            codes = np.array([[int(t) for t in lhs.split()]], dtype=np.uint8)
            got = int(oracle.pack(codes).view(np.uint32)[0, 0])
            assert got == int(rhs, 16), (line, hex(got))
            n_pack += 1
    assert n_unpack >= 5 and n_pack >= 5


def test_pack_unpack_round_trip():
    codes = synth.random_codes(37, 96, seed=11)
    assert np.array_equal(oracle.unpack(oracle.pack(codes)), codes)
    words = synth.random_words(np.random.default_rng(5), 19, 24)
    assert np.array_equal(oracle.pack(oracle.unpack(words)), words)


def test_pack_clamps_codes_above_15():
    codes = synth.random_codes(8, 64, seed=12, high=64)
    assert np.array_equal(oracle.unpack(oracle.pack(codes)), np.minimum(codes, 15))


def test_unpack_column_order_is_a_permutation_per_word():
    # every word's 8 nibbles land in 8 distinct columns of that word's block
    words = np.array([[0x76543210, 0xFEDCBA98]], dtype=np.uint32).view(np.int32)
    u = oracle.unpack(words)[0]
    assert sorted(u[:8].tolist()) == list(range(8))
    assert sorted(u[8:].tolist()) == list(range(8, 16))


# ---------------------------------------------------------------- dequant
def _one_word_problem(q, z, s_half):
    """A single group (g = 1) of 8 columns with every code q, zero z and scale s."""
    codes = np.full((1, 8), q, dtype=np.uint8)
    zeros = np.full((1, 8), z, dtype=np.uint8)
    scales = np.full((1, 8), s_half, dtype=np.float16)
    return oracle.pack(codes), oracle.pack(zeros), scales


def test_dequant_golden(golden_dir):
    rows = read_golden(golden_dir, "dequant_examples.txt")
    for line in rows:
        lhs, want = line.split("->")
        q, z, sh = lhs.split()
        qw, qz, sc = _one_word_problem(int(q), int(z), half_from_hex(int(sh, 16)))
        w = oracle.dequant(qw, qz, sc, group_size=1)
        assert np.all(w.astype(np.float64) == float(want.strip())), line
    assert len(rows) >= 8


def test_dequant_exhaustive_against_exact_rounding():
    # all 16 x 16 (q, z) pairs against a sweep of fp16 scales incl. subnormal and tie-prone ones
    rng = np.random.default_rng(3)
    sweep = [0x0001, 0x0003, 0x03FF, 0x0400, 0x1819, 0x251F, 0x3C01, 0x3C03, 0x3BFF, 0x4A3D, 0x57FF]
    sweep += rng.integers(0x0001, 0x5800, size=24).tolist()
    qs, zs = np.meshgrid(np.arange(16), np.arange(16), indexing="ij")
    qs, zs = qs.ravel(), zs.ravel()
    codes = qs.astype(np.uint8)[None, :]          # 1 row x 256 columns, one group
    zeros = zs.astype(np.uint8)[None, :]
    for h in sweep:
        s = half_from_hex(int(h))
        scales = np.full((1, 256), s, dtype=np.float16)
        w = oracle.dequant(oracle.pack(codes), oracle.pack(zeros), scales, group_size=1)
        s_exact = Fraction(float(s))
        for i in range(256):
            want = fp16_rn_exact((int(qs[i]) - int(zs[i])) * s_exact)
            assert Fraction(float(w[0, i])) == want, (hex(h), qs[i], zs[i])


def test_dequant_symmetric_uses_zero_eight():
    codes = np.arange(16, dtype=np.uint8).repeat(8)[None, :]          # 1 x 128
    scales = np.ones((1, 128), dtype=np.float16)
    w = oracle.dequant(oracle.pack(codes), None, scales, group_size=1)
    assert np.array_equal(w[0].astype(np.int64), codes[0].astype(np.int64) - 8)


def test_dequant_group_index_closed_form():
    # K = 3 groups of 4 rows; codes 9 everywhere; zeros 8, 7, 6 per group;
    # scales 1, 2, 4 per group -> rows of group j equal (j + 1) * 2^j.
    g, n = 4, 16
    codes = np.full((3 * g, n), 9, dtype=np.uint8)
    zeros = np.stack([np.full(n, 8 - j, dtype=np.uint8) for j in range(3)])
    scales = np.stack([np.full(n, 2.0 ** j, dtype=np.float16) for j in range(3)])
    w = oracle.dequant(oracle.pack(codes), oracle.pack(zeros), scales, group_size=g)
    for k in range(3 * g):
        j = k // g
        assert np.all(w[k] == (j + 1) * 2 ** j), k


def test_dequant_per_column_scale_and_zero_not_transposed():
    # distinct per-column zero points and scales: column n has z = n % 16 and s = 2^-(n % 4)
    n = 32
    codes = np.full((1, n), 15, dtype=np.uint8)
    zeros = (np.arange(n) % 16).astype(np.uint8)[None, :]
    scales = (2.0 ** -(np.arange(n) % 4)).astype(np.float16)[None, :]
    w = oracle.dequant(oracle.pack(codes), oracle.pack(zeros), scales, group_size=1)
    want = (15 - (np.arange(n) % 16)) * 2.0 ** -(np.arange(n) % 4)
    assert np.array_equal(w[0].astype(np.float64), want)


# ---------------------------------------------------------------- product
def test_linear_bruteforce_exact_rationals():
    p = synth.awq_problem(3, 8, 24, seed=21, group_size=8)
    w = oracle.dequant(p["qweight"], p["qzeros"], p["scales"], 8)
    y64 = oracle.linear_f64(p["x"], w)
    y32 = oracle.linear_f32acc(p["x"], w)
    assert y64.shape == (3, 24)
    for m in range(3):
        for n in range(24):
            terms = [Fraction(float(p["x"][m, k])) * Fraction(float(w[k, n])) for k in range(8)]
            exact = sum(terms)
            mag = sum(abs(t) for t in terms)
            assert abs(Fraction(float(y64[m, n])) - exact) <= mag * Fraction(8, 2 ** 53)
            assert abs(Fraction(float(y32[m, n])) - exact) <= mag * Fraction(8, 2 ** 24)


def test_linear_zero_weights_give_zero():
    # every row of each group carries the group's zero points as codes: q == z everywhere
    p = synth.awq_problem(4, 256, 64, seed=22)
    codes = synth.random_codes(256, 64, seed=23)
    same = np.repeat(codes[:1], 256, axis=0)
    w = oracle.dequant(oracle.pack(same), oracle.pack(same[:2]), p["scales"], 128)
    assert np.all(w == 0)
    assert np.all(oracle.linear_f64(p["x"], w) == 0)


def test_linear_one_hot_copies_integer_row():
    k_dim, n = 128, 64
    codes = synth.random_codes(k_dim, n, seed=24)
    zeros = np.zeros((1, n), dtype=np.uint8)
    scales = np.ones((1, n), dtype=np.float16)
    w = oracle.dequant(oracle.pack(codes), oracle.pack(zeros), scales, 128)
    x = np.zeros((2, k_dim), dtype=np.float16)
    x[0, 5] = 1.0
    x[1, 77] = 1.0
    y = oracle.linear_f64(x, w)
    assert np.array_equal(y[0], codes[5].astype(np.float64))
    assert np.array_equal(y[1], codes[77].astype(np.float64))


def test_awq_linear_word_column_locality():
    p = synth.awq_problem(5, 256, 40, seed=25)
    y = oracle.awq_linear(p["x"], p["qweight"], p["qzeros"], p["scales"], 128)
    assert y.shape == (5, 40)
    # outputs 8c..8c+7 depend only on word column c: zeroing word column 2 (codes and zeros)
    # changes exactly those outputs, to zero
    qw = p["qweight"].copy()
    qz = p["qzeros"].copy()
    qw[:, 2] = 0
    qz[:, 2] = 0
    y2 = oracle.awq_linear(p["x"], qw, qz, p["scales"], 128)
    assert np.array_equal(y2[:, :16], y[:, :16]) and np.array_equal(y2[:, 24:], y[:, 24:])
    assert np.all(y2[:, 16:24] == 0)


# ---------------------------------------------------------------- W4A8
def test_quant_act_golden(golden_dir):
    rows = read_golden(golden_dir, "w4a8_quant_examples.txt")
    for line in rows:
        xs, s_want, q_want = (part.strip() for part in line.split(";"))
        x = np.array([[float(t) for t in xs.split()]], dtype=np.float16)
        xq, s = oracle.quant_act(x)
        assert float(s[0]) == float(s_want), line
        assert xq[0].tolist() == [int(t) for t in q_want.split()], line
    assert len(rows) >= 4


def test_quant_act_invariants():
    x = synth.activations(np.random.default_rng(7), 16, 1000)
    xq, s = oracle.quant_act(x)
    assert xq.dtype == np.int8 and s.dtype == np.float32
    assert np.all(np.abs(xq.astype(np.int32)) <= 127)
    am = np.argmax(np.abs(x.astype(np.float32)), axis=1)
    assert np.all(np.abs(xq[np.arange(16), am].astype(np.int32)) == 127)
    # reconstruction error at most half a step (plus the fp16 rounding of the scale)
    err = np.abs(xq.astype(np.float64) * s[:, None] - x.astype(np.float64))
    assert np.all(err <= 0.5 * s[:, None] * (1 + 1e-3) + 1e-7)


def test_w4a8_accumulate_bruteforce():
    p = synth.w4a8_problem(3, 24, 16, seed=31)
    xq, _ = oracle.quant_act(p["x"])
    acc = oracle.w4a8_accumulate(xq, p["wq"])
    words = p["wq"].view(np.uint32)
    for m in range(3):
        for n in range(16):
            total = 0
            for k in range(24):
                word = int(words[k, n // 8])
                slot = oracle.AWQ_ORDER.index(n % 8)
                u = (word >> (4 * slot)) & 0xF
                total += int(xq[m, k]) * (u - 8)
            assert acc[m, n] == total


def test_w4a8_unit_scales_return_integers():
    # s_tok = s_ch = 1 and small accumulators: the fp16 output is the integer accumulator itself
    p = synth.w4a8_problem(2, 8, 16, seed=32)
    xq = np.array([[1, -1, 2, 0, 0, 3, -2, 1], [0, 0, 0, 0, 0, 0, 0, 5]], dtype=np.int8)
    y, acc = oracle.w4a8_linear(xq, np.ones(2, np.float32), p["wq"], np.ones(16, np.float16))
    assert np.array_equal(y.astype(np.float64), acc.astype(np.float64))
    # linearity of the accumulator in the activation codes
    acc2 = oracle.w4a8_accumulate((2 * xq).astype(np.int8), p["wq"])
    assert np.array_equal(acc2, 2 * acc)


def test_w4a8_extremes_fit_int32_at_k21760():
    # worst case |acc| <= K * 128 * 8 stays below 2^31 at the largest K of the workloads
    assert 21760 * 128 * 8 < 2 ** 31


# ---------------------------------------------------------------- W4A8 output epilogue
def _binary_fraction(text: str) -> Fraction:
    """'n/2^e' (or '-n/2^e') as an exact rational."""
    num, den = text.split("/")
    base, exp = den.split("^")
    assert base.strip() == "2"
    return Fraction(int(num)) / Fraction(2) ** int(exp)


def _codes_for_accumulator(target: int, k: int):
    """Activation codes xq (int8) and signed weights q (-8..7) over k rows with sum xq * q == target.

    target = n * (127 * 7) + b * 7 + c with 0 <= b <= 126 and 0 <= c <= 6: n rows of 127 x 7, one of
    b x 7 and one of c x 1 (negated codes for a negative target).
    """
    sign = -1 if target < 0 else 1
    t = abs(target)
    n, r = divmod(t, 127 * 7)
    b, c = divmod(r, 7)
    assert n + 2 <= k
    xq = np.zeros(k, dtype=np.int64)
    q = np.zeros(k, dtype=np.int64)
    xq[:n], q[:n] = 127, 7
    xq[n], q[n] = b, 7
    xq[n + 1], q[n + 1] = c, 1
    xq *= sign
    assert int(np.dot(xq, q)) == target
    return xq.astype(np.int8), q


def test_w4a8_epilogue_golden(golden_dir):
    # y = fp16(fp32(fp32(fp32(acc) * s_tok) * s_ch)) on hand-worked cases where an fp16 intermediate,
    # a direct fp16 rounding of the exact product, the scale product taken first, an unrounded
    # accumulator past 2^24 or a dropped token scale each give a different fp16 value
    lines = read_golden(golden_dir, "w4a8_epilogue_examples.txt")
    assert len(lines) == 6
    for line in lines:
        acc_t, st_t, sc_t, y_t, _ = (s.strip() for s in line.split(";"))
        target = int(acc_t)
        s_tok, s_ch, want = _binary_fraction(st_t), _binary_fraction(sc_t), _binary_fraction(y_t)
        k = abs(target) // (127 * 7) + 2 + 6
        xq, q = _codes_for_accumulator(target, k)
        # one packed word: 8 output columns with the same weights and scale
        wq = oracle.pack(np.repeat((q + 8)[:, None], 8, axis=1).astype(np.uint8))
        st32 = np.array([float(s_tok)], dtype=np.float32)
        sc16 = np.full(8, float(s_ch), dtype=np.float16)
        assert Fraction(float(st32[0])) == s_tok and Fraction(float(sc16[0])) == s_ch  # exact inputs
        y, acc = oracle.w4a8_linear(xq[None, :], st32, wq, sc16)
        assert np.all(acc == target)
        assert all(Fraction(float(v)) == want for v in y[0]), (line, y[0])


# ---------------------------------------------------------------- bfloat16 variant
def _bf16_value(bits: int) -> Fraction:
    """Exact value of a bf16 bit pattern (finite), decoded field by field."""
    sign = -1 if bits & 0x8000 else 1
    exp = (bits >> 7) & 0xFF
    frac = bits & 0x7F
    if exp == 0:
        return sign * Fraction(frac, 128) * Fraction(2) ** -126
    return sign * (1 + Fraction(frac, 128)) * Fraction(2) ** (exp - 127)


def test_bf16_golden(golden_dir):
    n_round = n_deq = 0
    for line in read_golden(golden_dir, "bf16_examples.txt"):
        lhs, rhs = (s.strip() for s in line.split(":"))
        want = int(rhs, 16)
        parts = lhs.split()
        if parts[0] == "round":
            f = np.array([int(parts[1], 16)], dtype=np.uint32).view(np.float32)
            assert int(oracle.bf16_round(f)[0]) == want, line
            n_round += 1
        else:
            q, z, sbits = int(parts[1]), int(parts[2]), int(parts[3], 16)
            codes = np.zeros((128, 8), dtype=np.uint8)
            codes[:, 0] = q
            zc = np.zeros((1, 8), dtype=np.uint8)
            zc[0, 0] = z
            scales = np.full((1, 8), sbits, dtype=np.uint16)
            w = oracle.dequant_bf16(oracle.pack(codes), oracle.pack(zc), scales, 128)
            assert np.all(w[:, 0] == want), line
            n_deq += 1
    assert n_round == 7 and n_deq == 4


def test_bf16_round_is_the_nearest_bf16():
    # brute force: for random finite float32 values, the result is the nearer of the two bf16 values
    # around the input (exact rational distances), the one with an even last bit on a tie
    rng = np.random.default_rng(11)
    bits = rng.integers(0, 2 ** 32, size=3000, dtype=np.uint64).astype(np.uint32)
    bits = bits[((bits >> 23) & 0xFF) < 0xFE]            # finite and below the top binade
    ties = (rng.integers(0, 2 ** 16, size=200, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000
    ties = ties[((ties >> 23) & 0xFF) < 0xFE]
    bits = np.concatenate([bits, ties]).astype(np.uint32)
    got = oracle.bf16_round(bits.view(np.float32))
    for b, g in zip(bits.tolist(), got.tolist()):
        v = Fraction(float(np.array([b], dtype=np.uint32).view(np.float32)[0]))
        lo = b >> 16                                      # same sign, magnitude truncated
        cands = [lo, lo + 1]
        dist = [abs(_bf16_value(c) - v) for c in cands]
        if dist[0] < dist[1]:
            best = cands[0]
        elif dist[1] < dist[0]:
            best = cands[1]
        else:
            best = cands[0] if cands[0] % 2 == 0 else cands[1]
        assert g == best, hex(b)


def test_dequant_bf16_exhaustive_against_exact_rounding():
    # every (q, z) pair x bf16 scales spanning several binades: the exact product rounded to the nearest
    # bf16 (ties to even) by a search over exact rationals
    rng = np.random.default_rng(12)
    sbits = np.concatenate([rng.integers(0x3A00, 0x3D80, size=6), [0x3F83, 0x3CA4]]).astype(np.uint16)
    q = np.repeat(np.arange(16), 16).astype(np.uint8)        # 256 rows: every (q, z)
    zz = np.tile(np.arange(16), 16).astype(np.uint8)
    for sb in sbits.tolist():
        codes = np.zeros((256, 8), dtype=np.uint8)
        codes[:, 3] = q
        # one group per row: group size 1 makes every row its own zero point
        zc = np.zeros((256, 8), dtype=np.uint8)
        zc[:, 3] = zz
        scales = np.full((256, 8), sb, dtype=np.uint16)
        w = oracle.dequant_bf16(oracle.pack(codes), oracle.pack(zc), scales, 1)
        s = _bf16_value(sb)
        for r in range(256):
            exact = (int(q[r]) - int(zz[r])) * s
            if exact == 0:
                assert _bf16_value(int(w[r, 3])) == 0
                continue
            mag = abs(exact)
            e = mag.numerator.bit_length() - mag.denominator.bit_length()
            while Fraction(2) ** e > mag:
                e -= 1
            while Fraction(2) ** (e + 1) <= mag:
                e += 1
            ulp = Fraction(2) ** (e - 7)
            m = mag / ulp
            f = floor(m)
            if m - f > Fraction(1, 2) or (m - f == Fraction(1, 2) and f % 2 == 1):
                f += 1
            want = (1 if exact > 0 else -1) * f * ulp
            assert _bf16_value(int(w[r, 3])) == want, (sb, r)


def test_dequant_bf16_symmetric_and_group_index():
    # symmetric: z = 8; group g of rows [128 g, 128 g + 128) takes scale row g
    codes = np.full((256, 8), 12, dtype=np.uint8)
    scales = np.zeros((2, 8), dtype=np.uint16)
    scales[0, :] = 0x3F80   # 1.0
    scales[1, :] = 0x4000   # 2.0
    w = oracle.bf16_to_float(oracle.dequant_bf16(oracle.pack(codes), None, scales, 128))
    assert np.all(w[:128] == 4.0) and np.all(w[128:] == 8.0)


def test_linear_bf16_bruteforce_exact_rationals():
    p = synth.awq_problem_bf16(2, 8, 8, seed=13, group_size=8)
    w = oracle.dequant_bf16(p["qweight"], p["qzeros"], p["scales"], 8)
    y = oracle.awq_linear_bf16(p["x"], p["qweight"], p["qzeros"], p["scales"], 8)
    for m in range(2):
        for n in range(8):
            exact = sum(_bf16_value(int(p["x"][m, k])) * _bf16_value(int(w[k, n])) for k in range(8))
            assert abs(Fraction(float(y[m, n])) - exact) <= abs(exact) * Fraction(1, 2 ** 52) + Fraction(1, 2 ** 120)


# ---------------------------------------------------------------- W4A8 with per-group weight scales
def test_w4a8_group_accumulate_bruteforce():
    p = synth.w4a8_group_problem(3, 16, 16, seed=14, group_size=8)
    xq, _ = oracle.quant_act(p["x"])
    acc = oracle.w4a8_group_accumulate(xq, p["wq"], p["s3"], 8)
    words = p["wq"].view(np.uint32)
    for m in range(3):
        for n in range(16):
            total = 0
            for k in range(16):
                slot = oracle.AWQ_ORDER.index(n % 8)
                u = (int(words[k, n // 8]) >> (4 * slot)) & 0xF
                total += int(xq[m, k]) * (u - 8) * int(p["s3"][k // 8, n])
            assert acc[m, n] == total


def test_w4a8_group_factor_16_is_the_per_channel_kernel():
    # s3 = 16 on every group is the per-channel kernel's shift by 4: the accumulator is 16 times the
    # per-channel one, and with s2 = s_ch / 16 (exact) the fp16 outputs are identical
    p = synth.w4a8_problem(4, 256, 64, seed=15)
    xq, s = oracle.quant_act(p["x"])
    s3 = np.full((2, 64), 16, dtype=np.float16)
    acc_g = oracle.w4a8_group_accumulate(xq, p["wq"], s3, 128)
    assert np.array_equal(acc_g, 16 * oracle.w4a8_accumulate(xq, p["wq"]))
    s2 = (p["s_ch"].astype(np.float32) / 16).astype(np.float16)
    assert np.array_equal(s2.astype(np.float32) * 16, p["s_ch"].astype(np.float32))
    y_g, _ = oracle.w4a8_group_linear(xq, s, p["wq"], s3, s2, 128)
    y_c, _ = oracle.w4a8_linear(xq, s, p["wq"], p["s_ch"])
    assert np.array_equal(y_g.view(np.uint16), y_c.view(np.uint16))


def test_w4a8_group_rejects_non_integer_factors():
    p = synth.w4a8_group_problem(1, 128, 8, seed=16)
    xq, _ = oracle.quant_act(p["x"])
    bad = p["s3"].copy()
    bad[0, 0] = 1.5
    for s3 in (bad, np.zeros_like(p["s3"]), np.full_like(p["s3"], 17)):
        try:
            oracle.w4a8_group_accumulate(xq, p["wq"], s3, 128)
        except ValueError:
            continue
        raise AssertionError("accepted an s3 outside the integers 1..16")


def test_new_order_map_round_trip_and_word():
    # the new format's map: nibble slot i holds column 8c + i, so codes 0..7 pack to 0x76543210
    q = np.arange(8, dtype=np.uint8)[None, :]
    assert int(oracle.pack(q, oracle.AWQ_ORDER_NEW).view(np.uint32)[0, 0]) == 0x76543210
    assert int(oracle.pack(q).view(np.uint32)[0, 0]) == 0x75316420
    codes = synth.random_codes(5, 64, seed=17)
    assert np.array_equal(oracle.unpack(oracle.pack(codes, oracle.AWQ_ORDER_NEW), oracle.AWQ_ORDER_NEW), codes)


# ---------------------------------------------------------------- decode prepack layout
def _unit_words(buf, unit):
    base = unit * oracle.PREPACK_UNIT_BYTES
    return buf[base:base + 16384].view(np.uint32), buf[base + 16384:base + 16512].view(np.uint32), \
        buf[base + 16512:base + oracle.PREPACK_UNIT_BYTES].view(np.float16)


def _codes_to_qweight(q):
    return oracle.pack(q.astype(np.uint8))


def test_prepack_words_for_row_and_column_patterns():
    # codes equal to the row index mod 16: word (w, i, l, b) holds rows 2t, 2t, 2t+8, 2t+8, 2t+1, 2t+1,
    # 2t+9, 2t+9 (lowest nibble first), whatever w, i, b: lane 0 (t = 0) reads 0x99118800 and lane 1
    # (t = 1) 0xBB33AA22
    K, N = 256, 512
    rows = (np.arange(K)[:, None] % 16 + np.zeros((1, N), int)).astype(np.uint8)
    buf = oracle.prepack_gemv(_codes_to_qweight(rows), None, np.ones((K // 128, N), np.float16))
    for unit in range(4):
        words, _, _ = _unit_words(buf, unit)
        w = words.reshape(4, 8, 32, 4)
        assert np.all(w[:, :, 0, :] == 0x99118800) and np.all(w[:, :, 1, :] == 0xBB33AA22)
    # codes equal to the column index mod 16: block b of lane g reads columns 8g + 2b (even positions)
    # and 8g + 2b + 1 (odd positions): g = 0, b = 0 -> 0x10101010; b = 1 -> 0x32323232; g = 1, b = 0 ->
    # 0x98989898
    cols = (np.zeros((K, 1), int) + np.arange(N)[None, :] % 16).astype(np.uint8)
    buf = oracle.prepack_gemv(_codes_to_qweight(cols), None, np.ones((K // 128, N), np.float16))
    w = _unit_words(buf, 3)[0].reshape(4, 8, 32, 4)
    assert np.all(w[:, :, 0:4, 0] == 0x10101010) and np.all(w[:, :, 0:4, 1] == 0x32323232)
    assert np.all(w[:, :, 4:8, 0] == 0x98989898)


def test_prepack_zero_and_scale_placement():
    # zero point of column n = n mod 16: word (w, g) holds columns 64 w + 8 g + c in nibble c, so even g
    # reads 0x76543210 and odd g 0xFEDCBA98; the symmetric layout holds 8 everywhere; scales sit in the
    # same column order; columns beyond N hold zero point 0 and scale 0
    K, N = 128, 480                                      # two tiles, the second one 224 columns wide
    zc = (np.arange(N)[None, :] % 16).astype(np.uint8)
    sc = (np.arange(N)[None, :] * 0.25).astype(np.float16)
    buf = oracle.prepack_gemv(np.zeros((K, N // 8), np.int32), oracle.pack(zc), sc)
    z0, s0 = _unit_words(buf, 0)[1].reshape(4, 8), _unit_words(buf, 0)[2].reshape(4, 8, 8)
    assert np.all(z0[:, 0::2] == 0x76543210) and np.all(z0[:, 1::2] == 0xFEDCBA98)
    assert np.array_equal(s0.reshape(-1), (np.arange(256) * 0.25).astype(np.float16))
    z1, s1 = _unit_words(buf, 1)[1].reshape(-1), _unit_words(buf, 1)[2].reshape(-1)
    assert np.all(z1[28:] == 0) and np.all(s1[224:] == 0)            # columns 480..511 are padding
    assert np.array_equal(s1[:224], ((256 + np.arange(224)) * 0.25).astype(np.float16))
    sym = oracle.prepack_gemv(np.zeros((K, N // 8), np.int32), None, sc)
    assert np.all(_unit_words(sym, 0)[1] == 0x88888888)


def test_prepack_is_a_permutation_of_the_codes():
    # every unit holds exactly the codes of its 128 x 256 block, each once
    p = synth.awq_problem(1, 256, 768, seed=18)
    q = oracle.unpack(p["qweight"])
    buf = oracle.prepack_gemv(p["qweight"], p["qzeros"], p["scales"])
    for unit in range(6):
        tile, grp = divmod(unit, 2)
        words = _unit_words(buf, unit)[0]
        nib = np.stack([(words >> np.uint32(4 * j)) & np.uint32(15) for j in range(8)]).ravel()
        block = q[128 * grp:128 * grp + 128, 256 * tile:256 * tile + 256].ravel()
        assert np.array_equal(np.bincount(nib, minlength=16), np.bincount(block, minlength=16))
