"""Pins for the oracle's scalar codecs (fp16, bf16, E2M1, E4M3FN).

Each codec is checked against something other than itself: the values the
format pages print (tests/golden), or a library conversion (numpy binary16,
torch bfloat16 / float8_e4m3fn) over every bit pattern.
"""
import math

import numpy as np
import torch

from golden_io import rows


def _same(a, b):
    if math.isnan(a) or math.isnan(b):
        return math.isnan(a) and math.isnan(b)
    return a == b and math.copysign(1.0, a) == math.copysign(1.0, b)


def test_fp16_decode_all_words_vs_numpy(oracle):
    words = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = words.view(np.float16).astype(np.float64)
    for h in range(65536):
        assert _same(oracle.fp16_to_double(h), float(ref[h])), hex(h)


def test_fp16_encode_rne_vs_numpy(oracle):
    rng = np.random.default_rng(1)
    # wide dynamic range, both signs, plus exact halfway points between binary16 values
    vals = list(rng.standard_normal(4000) * np.exp2(rng.uniform(-30, 17, 4000)))
    for h in range(0, 0x7C00, 97):
        lo = float(np.uint16(h).view(np.float16))
        hi = float(np.uint16(h + 1).view(np.float16))
        vals += [0.5 * (lo + hi), -0.5 * (lo + hi), lo, np.nextafter(0.5 * (lo + hi), np.inf)]
    vals += [0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e6, -1e6, 2.0 ** -25, 2.0 ** -26,
             3 * 2.0 ** -26, 2.0 ** -24, float("inf"), float("-inf")]
    for v in vals:
        got = oracle.double_to_fp16(float(v))
        with np.errstate(over="ignore"):  # values past 65520 overflow to infinity, as they should
            want = int(np.array([v], dtype=np.float64).astype(np.float16).view(np.uint16)[0])
        assert got == want, (v, hex(got), hex(want))
    assert oracle.double_to_fp16(float("nan")) & 0x7C00 == 0x7C00


def test_bf16_decode_all_words_vs_torch(oracle):
    words = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    ref = words.view(torch.bfloat16).to(torch.float64).numpy()
    for b in range(0, 65536):
        assert _same(oracle.bf16_to_double(b), float(ref[b])), hex(b)


def test_e2m1_matches_printed_grid(oracle):
    table = rows("e2m1_grid.txt")
    assert len(table) == 16
    for code, value in table:
        assert _same(oracle.e2m1_to_double(int(code, 16)), float(value)), code


def test_e4m3fn_printed_cases(oracle):
    for word, value in rows("e4m3fn_cases.txt"):
        assert _same(oracle.e4m3fn_to_double(int(word, 16)), float(value)), word


def test_e4m3fn_all_words_vs_torch(oracle):
    words = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = words.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        assert _same(oracle.e4m3fn_to_double(c), float(ref[c])), hex(c)


def test_e2m1_times_e4m3_is_exact_in_fp16_and_bf16(oracle):
    """Every E2M1 x E4M3FN product has at most 6 significant bits: exactly representable in
    bf16 and (after scaling by 2^-14) in fp16 -- the property the GPU decode relies on."""
    for c in range(16):
        for s in range(256):
            v = oracle.e2m1_to_double(c) * oracle.e4m3fn_to_double(s)
            if math.isnan(v):
                continue
            assert float(np.float64(v).astype(np.float32)) == v
            assert float(torch.tensor(v, dtype=torch.float64).to(torch.bfloat16).double()) == v
            scaled = v * 2.0 ** -14
            assert float(np.float64(scaled).astype(np.float16)) == scaled
