"""Pins for the oracle's PN decode and validation ("PN weight format" page).

The layout check builds blocks from the page's Block layout *table* (bit ranges
per t, tests/golden/pn_layout_table.txt), not from the shift formula the oracle
uses, and rejects the documented wrong decoder (shift by element index).
"""
import numpy as np
import pytest

from golden_io import rows
from block_quantized_weight_pn3t_gb300 import synth

PN3T, PN4T = 124, 125
NAMES = {"pn3t": PN3T, "pn4t": PN4T}
BLK = {PN3T: 80, PN4T: 64}
CPW = {PN3T: 10, PN4T: 8}
Z = {PN3T: 4, PN4T: 8}


def layout():
    tab = {}
    for name, t, lo, hi in rows("pn_layout_table.txt"):
        tab[(NAMES[name], int(t))] = (int(lo), int(hi))
    return tab


def build_block(type_, d_bits, codes, tab):
    """34-byte block from per-element codes, placing each code by the printed table."""
    words = [0] * 8
    for e, c in enumerate(codes):
        lo, hi = tab[(type_, e % CPW[type_])]
        assert c < (1 << (hi - lo + 1))
        words[e // CPW[type_]] |= c << lo
    out = bytearray(d_bits.to_bytes(2, "little"))
    for w in words:
        out += w.to_bytes(4, "little")
    return np.frombuffer(bytes(out), dtype=np.uint8)


def fp16_value(bits):
    return float(np.uint16(bits).view(np.float16))


@pytest.mark.parametrize("type_", [PN3T, PN4T])
def test_layout_table_every_position(oracle, type_):
    """A single non-zero code at element e decodes only at e, with value d*(v - z)."""
    tab = layout()
    z, blk = Z[type_], BLK[type_]
    d_bits = 0x3C00  # 1.0
    for e in range(blk):
        for v in range(2 * z):
            codes = [z] * blk
            codes[e] = v
            W = build_block(type_, d_bits, codes, tab)
            out = oracle.dequantize(type_, W, 1, blk)[0]
            expect = np.zeros(blk, dtype=np.float32)
            expect[e] = v - z
            assert np.array_equal(out, expect), (e, v)


@pytest.mark.parametrize("type_", [PN3T, PN4T])
def test_elemshift_decoder_is_rejected(oracle, type_):
    """Negative control: the wrong decoder (shift = BITS * t) fails the layout check."""
    tab = layout()
    z, blk = Z[type_], BLK[type_]
    failures = 0
    for e in range(blk):
        codes = [z] * blk
        codes[e] = z + 1
        W = build_block(type_, 0x3C00, codes, tab)
        bad = oracle.dequantize_elemshift(type_, W, 1, blk)[0]
        good = oracle.dequantize(type_, W, 1, blk)[0]
        expect = np.zeros(blk, dtype=np.float32)
        expect[e] = 1.0
        assert np.array_equal(good, expect)
        failures += not np.array_equal(bad, expect)
    # the layout check rejects the wrong decoder at most positions (for pn4t it is a
    # permutation of each word's slots with fixed points t = 0 and t = 7)
    assert failures >= blk // 2
    # and on random blocks the wrong decoder differs on most weights
    W = synth.pn_random_blocks(type_, 8, blk * 4, seed=5).numpy()
    a = oracle.dequantize(type_, W, 8, blk * 4)
    b = oracle.dequantize_elemshift(type_, W, 8, blk * 4)
    assert np.mean(a != b) > 0.5


@pytest.mark.parametrize("type_", [PN3T, PN4T])
def test_decode_ranges_and_grid(oracle, type_):
    """Codes decode to -z*d .. (z-1)*d, each an integer multiple of d."""
    K = BLK[type_] * 16
    W = synth.pn_random_blocks(type_, 32, K, seed=11).numpy()
    out = oracle.dequantize(type_, W, 32, K).astype(np.float64)
    nb = K // BLK[type_]
    dbits = W.reshape(32, nb, 34)[:, :, 0:2].copy().view(np.uint16)[..., 0]
    d = dbits.view(np.float16).astype(np.float64)
    q = out.reshape(32, nb, BLK[type_]) / d[..., None]
    assert np.all(q >= -Z[type_]) and np.all(q <= Z[type_] - 1)
    assert np.array_equal(q, np.round(q))
    # every code value occurs (uniform codes): the full range is reached
    assert set(np.unique(q).astype(int)) == set(range(-Z[type_], Z[type_]))


def test_decode_exact_in_fp32_for_every_fp16_d():
    """The page: both steps are exact in fp32 (d has 11 significant bits, n - z at most 4)."""
    d = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16).astype(np.float64)
    d = d[np.isfinite(d)]
    for k in range(-8, 8):
        prod = d * k
        assert np.array_equal(prod.astype(np.float32).astype(np.float64), prod)


@pytest.mark.parametrize("type_", [PN3T, PN4T])
def test_signed_zero(oracle, type_):
    """Code z with negative d decodes to -0.0; with positive d to +0.0."""
    tab = layout()
    z, blk = Z[type_], BLK[type_]
    for d_bits, neg in ((0xBC00, True), (0x3C00, False), (0x8000, True), (0x0000, False)):
        W = build_block(type_, d_bits, [z] * blk, tab)
        out = oracle.dequantize(type_, W, 1, blk)[0]
        assert np.all(out == 0.0)
        assert np.all(np.signbit(out) == neg)


@pytest.mark.parametrize("name,type_", [("pn3t", PN3T), ("pn4t", PN4T)])
def test_canonical_zero_words(oracle, name, type_):
    want = {r[0]: (int(r[1], 16), int(r[2], 16)) for r in rows("pn_canonical_zero.txt")}
    d_bits, word = want[name]
    tab = layout()
    W = build_block(type_, d_bits, [Z[type_]] * BLK[type_], tab)
    assert int.from_bytes(bytes(W[0:2]), "little") == d_bits
    for i in range(8):
        assert int.from_bytes(bytes(W[2 + 4 * i: 6 + 4 * i]), "little") == word
    # and the quantizer writes exactly these bytes for an all-zero group
    q = oracle.quantize(type_, np.zeros((1, BLK[type_]), dtype=np.float32))
    assert np.array_equal(q[0], W)


@pytest.mark.parametrize("type_", [PN3T, PN4T])
def test_validate_rules(oracle, type_):
    tab = layout()
    z, blk = Z[type_], BLK[type_]
    K = blk * 3
    good = np.concatenate([build_block(type_, 0x1234, [z] * blk, tab) for _ in range(3)])
    cases = []
    for dbad in (0x7C00, 0xFC00, 0x7E00, 0x7C01, 0xFE00):
        r = good.copy()
        r[34:36] = np.frombuffer(dbad.to_bytes(2, "little"), dtype=np.uint8)
        cases.append((r, 1))
    for d_ok in (0x7BFF, 0xFBFF, 0x0001, 0x8000, 0x0000):
        r = good.copy()
        r[68:70] = np.frombuffer(d_ok.to_bytes(2, "little"), dtype=np.uint8)
        cases.append((r, 0))
    for bit in (15, 31, 14, 30, 0):
        r = good.copy()
        word = int.from_bytes(bytes(r[34 + 2 + 4 * 5: 34 + 6 + 4 * 5]), "little") | (1 << bit)
        r[34 + 2 + 20: 34 + 6 + 20] = np.frombuffer(word.to_bytes(4, "little"), dtype=np.uint8)
        reserved = bit in (15, 31)
        cases.append((r, 1 if (reserved and type_ == PN3T) else 0))
    W = np.stack([c[0] for c in cases])
    flags = oracle.validate(type_, W, len(cases), K)
    assert flags.tolist() == [c[1] for c in cases]


@pytest.mark.parametrize("type_", [PN3T, PN4T])
def test_unaligned_row_bytes(oracle, type_):
    """Decode does not depend on where the blocks sit in memory (odd blocks are only
    2-byte aligned): the same bytes at every offset mod 16 decode identically."""
    K = BLK[type_] * 8
    W = synth.pn_random_blocks(type_, 4, K, seed=3).numpy().reshape(-1)
    ref = oracle.dequantize(type_, W, 4, K)
    for off in (2, 4, 6, 8, 14):
        buf = np.zeros(W.size + 32, dtype=np.uint8)
        view = buf[off: off + W.size]
        view[:] = W
        assert view.ctypes.data % 16 == (buf.ctypes.data + off) % 16
        assert np.array_equal(oracle.dequantize(type_, np.ascontiguousarray(view), 4, K), ref)
