"""Pins for the oracle's grouped signed-integer formats ("tensor-formats.md", sections 4 to 7):
Q4G64_F16S, Q5G64_F16S, Q6G64_F16S and W8G32_F16S.

What fixes them, independent of the oracle's own arithmetic:
  - the printed integral-rounding examples of the canonical encoder (tests/golden);
  - the printed scheme table (code widths, groups, intervals, qmax; tests/golden);
  - closed forms: a group whose largest magnitude is qmax * 2^j has the exact scale 2^j and
    codes rint(x / 2^j); two's-complement words decode to u or u - 2^b;
  - the special cases the page spells out: an all-zero group (scale +0, codes 0), the 2^-24
    rescue of a scale that rounds to zero, failure on an overflowing scale or a non-finite value,
    W8 never emitting -128, a partial last group scaled from its own values only;
  - the normative order inv = 1 / scale, x * inv (found cases where x / scale rounds to
    another integer must follow the reciprocal), computed here in numpy float32;
  - decode = numpy float32 product of the binary16 scale and the code; GEMV = fp64 matmul.
"""
import numpy as np
import pytest

from golden_io import rows

Q4, Q5, Q6, W8 = 1104, 1105, 1106, 1108
SCHEMES = {Q4: "Q4G64_F16S", Q5: "Q5G64_F16S", Q6: "Q6G64_F16S", W8: "W8G32_F16S"}


def table():
    t = {}
    for name, bits, G, qmin, qmax, bpw in rows("grouped_schemes.txt"):
        t[name] = (int(bits), int(G), int(qmin), int(qmax), float(bpw))
    return t


def params(type_):
    return table()[SCHEMES[type_]]


def codes_of(oracle, type_, lo, hi, K):
    """Signed codes via decode with every scale 1.0 (0x3C00): w = 1 * q exactly."""
    n = lo.shape[0]
    ns = oracle.grouped_plane_bytes(type_, K)[2]
    ones = np.full((n, ns), 0x3C00, dtype=np.uint16)
    return oracle.dequantize_grouped(type_, lo, hi, ones, n, K).astype(np.int64)


def f16(bits):
    return np.array(bits, dtype=np.uint16).view(np.float16).astype(np.float32)


@pytest.mark.parametrize("type_", [Q4, Q5, Q6, W8])
def test_scheme_table_and_plane_sizes(oracle, type_):
    bits, G, qmin, qmax, bpw = params(type_)
    assert oracle.GROUPED[type_] == (bits, G, qmin, qmax)
    assert bits + 16 / G == bpw  # section 7: b + 16 / G
    K = 4 * G
    lo, hi, ns = oracle.grouped_plane_bytes(type_, K)
    assert (lo + hi) * 8 == bits * K and ns == 4


def test_printed_rounding_examples(oracle):
    """A Q4 group holding 7.0 has scale exactly 1 (7 / 7), so x * inv = x and the code is the
    printed integral rounding of x."""
    ex = [(float(a), int(b)) for a, b in rows("maxabs_rounding_examples.txt")]
    K = 64
    w = np.zeros((1, K), dtype=np.float32)
    w[0, 0] = 7.0
    for i, (x, _) in enumerate(ex):
        w[0, 1 + i] = x
    lo, hi, sc = oracle.quantize_grouped(Q4, w)
    assert sc[0, 0] == 0x3C00
    q = codes_of(oracle, Q4, lo, hi, K)[0]
    assert q[0] == 7
    for i, (_, want) in enumerate(ex):
        assert q[1 + i] == want


@pytest.mark.parametrize("type_", [Q4, Q5, Q6, W8])
@pytest.mark.parametrize("j", [-20, -3, 0, 5, 10])
def test_power_of_two_scale_closed_form(oracle, type_, j):
    bits, G, qmin, qmax, _ = params(type_)
    rng = np.random.default_rng(100 + j)
    K = 2 * G
    s = np.float32(2.0 ** j)
    w = (rng.uniform(-1, 1, size=(3, K)) * qmax * s).astype(np.float32)
    w[:, 0] = qmax * s
    w[:, G] = -qmax * s
    lo, hi, sc = oracle.quantize_grouped(type_, w)
    assert np.all(f16(sc) == s)
    want = np.clip(np.rint(w / s), qmin, qmax)  # the division by a power of two is exact
    assert np.array_equal(codes_of(oracle, type_, lo, hi, K), want.astype(np.int64))


def pack(type_, u):
    """Planes of one row of logical words u (the library layout, as test_plane_bit_order pins it)."""
    K = len(u)
    if type_ == W8:
        return u.astype(np.uint8)[None, :], None
    lo = ((u[0::2] & 15) | ((u[1::2] & 15) << 4)).astype(np.uint8)[None, :]
    if type_ == Q4:
        return lo, None
    if type_ == Q5:
        hb = np.zeros(K // 8, dtype=np.uint8)
        for k in range(K):
            hb[k // 8] |= ((u[k] >> 4) & 1) << (k % 8)
        return lo, hb[None, :]
    hb = np.zeros(K // 4, dtype=np.uint8)
    for k in range(K):
        hb[k // 4] |= ((u[k] >> 4) & 3) << (2 * (k % 4))
    return lo, hb[None, :]


@pytest.mark.parametrize("type_", [Q4, Q5, Q6, W8])
def test_every_word_decodes_twos_complement(oracle, type_):
    """Section 5: q = u for u < 2^(b-1), else u - 2^b, for every word of the width."""
    bits = params(type_)[0]
    n = 1 << bits
    K = max(8, n)
    u = np.arange(K, dtype=np.int64) % n
    lo, hi = pack(type_, u)
    got = codes_of(oracle, type_, lo, hi, K)[0]
    want = np.where(u < n // 2, u, u - n)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("type_", [Q4, Q5, Q6, W8])
def test_decode_is_the_binary32_product(oracle, type_):
    bits, G, qmin, qmax, _ = params(type_)
    rng = np.random.default_rng(7)
    N, K = 5, 2 * G + 16  # partial last group
    lb, hb, ns = oracle.grouped_plane_bytes(type_, K)
    lo = rng.integers(0, 256, size=(N, lb), dtype=np.uint8)
    hi = rng.integers(0, 256, size=(N, hb), dtype=np.uint8) if hb else None
    if type_ == W8:
        lo[lo == 0x80] = 0x7F
    sc = rng.integers(0, 0x7C00, size=(N, ns), dtype=np.uint16)  # finite, sign clear
    sc[0, 0] = 0x0001
    out = oracle.dequantize_grouped(type_, lo, hi, sc, N, K)
    q = codes_of(oracle, type_, lo, hi, K)
    want = np.repeat(f16(sc), G, axis=1)[:, :K] * q.astype(np.float32)
    assert np.array_equal(out.view(np.uint32), want.astype(np.float32).view(np.uint32))


def test_plane_bit_order(oracle):
    """The library layout: nibble plane (even k low), Q5 bit plane (bit k % 8), Q6 2-bit plane."""
    K = 8
    lo = np.array([[0x21, 0x43, 0x65, 0x87]], dtype=np.uint8)  # words 1,2,3,4,5,6,7,8 in the low bits
    q4 = codes_of(oracle, Q4, lo, None, K)[0]
    assert list(q4) == [1, 2, 3, 4, 5, 6, 7, -8]
    hi5 = np.array([[0b10000001]], dtype=np.uint8)  # bit 4 set for k = 0 and k = 7
    q5 = codes_of(oracle, Q5, lo, hi5, K)[0]
    assert list(q5) == [1 + 16 - 32, 2, 3, 4, 5, 6, 7, 8 + 16 - 32]
    hi6 = np.array([[0b00000011, 0b01000000]], dtype=np.uint8)  # k = 0 -> 3, k = 7 -> 1
    q6 = codes_of(oracle, Q6, lo, hi6, K)[0]
    assert list(q6) == [1 + 48 - 64, 2, 3, 4, 5, 6, 7, 8 + 16]


@pytest.mark.parametrize("type_", [Q4, Q5, Q6, W8])
def test_all_zero_group(oracle, type_):
    _, G, _, _, _ = params(type_)
    w = np.zeros((2, 2 * G), dtype=np.float32)
    w[1, :G] = -0.0
    w[1, G] = 1.0
    lo, hi, sc = oracle.quantize_grouped(type_, w)
    assert sc[0, 0] == 0 and sc[0, 1] == 0 and sc[1, 0] == 0 and sc[1, 1] != 0
    q = codes_of(oracle, type_, lo, hi, 2 * G)
    assert np.all(q[0] == 0) and np.all(q[1, :G] == 0)


@pytest.mark.parametrize("type_", [Q4, Q5, Q6, W8])
def test_tiny_scale_rescue(oracle, type_):
    """amax / qmax below half the smallest binary16 subnormal rounds to +0: the scale is 0x0001."""
    _, G, _, qmax, _ = params(type_)
    w = np.zeros((1, G), dtype=np.float32)
    w[0, 3] = np.float32(2.0 ** -26) * qmax
    lo, hi, sc = oracle.quantize_grouped(type_, w)
    assert sc[0, 0] == 0x0001


@pytest.mark.parametrize("type_", [Q4, Q5, Q6, W8])
def test_overflow_and_non_finite_fail(oracle, type_):
    _, G, _, qmax, _ = params(type_)
    w = np.zeros((1, G), dtype=np.float32)
    w[0, 0] = np.float32(65520.0) * qmax  # raw scale 65520 rounds to binary16 infinity
    with pytest.raises(ValueError):
        oracle.quantize_grouped(type_, w)
    w[0, 0] = np.float32(65504.0) * qmax  # the largest finite scale is accepted
    lo, hi, sc = oracle.quantize_grouped(type_, w)
    assert sc[0, 0] == 0x7BFF
    for bad in (np.inf, -np.inf, np.nan):
        w[0, 0] = bad
        with pytest.raises(ValueError):
            oracle.quantize_grouped(type_, w)


def test_w8_never_emits_minus_128(oracle):
    rng = np.random.default_rng(3)
    w = rng.standard_normal((64, 256)).astype(np.float32)
    w[:, ::32] = -np.abs(w[:, ::32]) * 3  # most negative value is the group's amax
    lo, _, _ = oracle.quantize_grouped(W8, w)
    assert not np.any(lo == 0x80)


@pytest.mark.parametrize("type_", [Q4, Q5, Q6, W8])
def test_partial_last_group_uses_its_own_values(oracle, type_):
    _, G, _, qmax, _ = params(type_)
    K = G + 8
    rng = np.random.default_rng(11)
    w = rng.standard_normal((4, K)).astype(np.float32)
    w[:, :G] *= 1000.0  # the full group's amax must not leak into the partial one
    lo, hi, sc = oracle.quantize_grouped(type_, w)
    amax_tail = np.abs(w[:, G:]).max(axis=1)
    raw = (amax_tail / np.float32(qmax)).astype(np.float32)
    assert np.array_equal(sc[:, 1], raw.astype(np.float16).view(np.uint16))


def near_tie_values(qmax, rng, want=8):
    """(scale, x) pairs, scale a binary16 value, x within a few float32 ulps of (k + 1/2) * scale,
    for which rint(x * fl(1 / scale)) != rint(x / scale) in float32 (numpy's IEEE arithmetic)."""
    out = []
    while len(out) < want:
        s = np.float32(np.float16(rng.uniform(0.01, 4.0)))
        inv = np.float32(1.0) / s
        k = rng.integers(-qmax, qmax)
        x0 = np.float32((k + 0.5) * np.float64(s))
        for d in range(-3, 4):
            x = np.float32(x0)
            for _ in range(abs(d)):
                x = np.nextafter(x, np.float32(np.inf if d > 0 else -np.inf), dtype=np.float32)
            if abs(x) > qmax * s:
                continue
            if np.rint(np.float32(x * inv)) != np.rint(np.float32(x / s)):
                out.append((s, x))
    return out


@pytest.mark.parametrize("type_", [Q4, Q5, Q6, W8])
def test_reciprocal_multiply_order(oracle, type_):
    """Section 7 makes inv = fl(1 / scale) then fl(x * inv) normative: at values where x / scale
    would round to another integer, the oracle's code is the reciprocal one."""
    bits, G, qmin, qmax, _ = params(type_)
    rng = np.random.default_rng(21 + bits)
    cases = near_tie_values(qmax, rng)
    w = np.zeros((len(cases), G), dtype=np.float32)
    for i, (s, x) in enumerate(cases):
        w[i, 0] = np.float32(qmax) * s  # exact: the group's scale is s
        w[i, 1] = x
    lo, hi, sc = oracle.quantize_grouped(type_, w)
    q = codes_of(oracle, type_, lo, hi, G)
    for i, (s, x) in enumerate(cases):
        assert f16(sc[i, 0]) == s
        inv = np.float32(1.0) / s
        assert q[i, 1] == np.clip(np.rint(np.float32(x * inv)), qmin, qmax)
        assert q[i, 1] != np.clip(np.rint(np.float32(x / s)), qmin, qmax) or abs(np.rint(np.float32(x / s))) > qmax


@pytest.mark.parametrize("type_", [Q4, Q5, Q6, W8])
def test_gemv_against_fp64_matmul(oracle, type_):
    _, G, _, _, _ = params(type_)
    rng = np.random.default_rng(5)
    N, K, M = 19, 3 * G + 24, 3
    w = rng.standard_normal((N, K)).astype(np.float32)
    lo, hi, sc = oracle.quantize_grouped(type_, w)
    Wd = oracle.dequantize_grouped(type_, lo, hi, sc, N, K).astype(np.float64)
    X = rng.standard_normal((M, K)).astype(np.float32)
    Y, A = oracle.gemv_grouped(type_, lo, hi, sc, N, K, X)
    ref = X.astype(np.float64) @ Wd.T
    aref = np.abs(X.astype(np.float64)) @ np.abs(Wd).T
    assert np.all(np.abs(Y - ref) <= 1e-12 * aref)
    assert np.allclose(A, aref, rtol=1e-12)
    k = 37
    e = np.zeros((1, K), dtype=np.float32)
    e[0, k] = 1.0
    Y1, _ = oracle.gemv_grouped(type_, lo, hi, sc, N, K, e)
    assert np.array_equal(Y1[0], Wd[:, k])


@pytest.mark.parametrize("type_", [Q4, Q5, Q6, W8])
def test_validity(oracle, type_):
    bits, G, _, _, _ = params(type_)
    rng = np.random.default_rng(9)
    N, K = 8, 2 * G
    w = rng.standard_normal((N, K)).astype(np.float32)
    lo, hi, sc = oracle.quantize_grouped(type_, w)
    assert not oracle.validate_grouped(type_, lo, hi, sc, N, K).any()
    sc2 = sc.copy()
    sc2[1, 0] |= 0x8000           # negative scale
    sc2[2, 1] = 0x7C00            # infinity
    sc2[3, 0] = 0x7E00            # NaN
    sc2[4, 1] = 0x0000            # +0 scale over nonzero codes
    lo2 = lo.copy()
    if type_ == W8:
        lo2[5, 3] = 0x80          # the word of -128
    flags = oracle.validate_grouped(type_, lo2, hi, sc2, N, K)
    want = np.zeros(N, dtype=np.int32)
    want[[1, 2, 3]] = 1
    want[4] = 1 if np.any(codes_of(oracle, type_, lo[4:5], None if hi is None else hi[4:5], K)[0, G:] != 0) else 0
    if type_ == W8:
        want[5] = 1
    assert np.array_equal(flags, want)
