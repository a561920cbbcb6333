"""Pins for the oracle's NVFP4 clip search (TandemLLM "Quantisation and profiles", section "The
clip search": five multipliers per group of 16, the one with the least act_ms-weighted squared
reconstruction error kept).

  - two worked examples computed by hand from the definitions (comments show the arithmetic):
    with equal act_ms the clipped multiplier 0.90 wins; a heavily used outlier channel makes
    the unclipped 1.00 win;
  - brute force on random groups: each of the five candidates is scored with torch's E4M3FN
    rounding and the printed E2M1 grid (tests/golden), and the oracle's choice, scale and codes
    must be the argmin's (the first on ties);
  - an all-zero group gets the zero scale and zero words; decoding the output with the
    separately pinned NVFP4 decoder reproduces the weights the search scored.
"""
import numpy as np
import pytest
import torch

from golden_io import rows


def multipliers():
    return [float(m) for _, m in rows("nvfp4_clip_multipliers.txt")]


def e2m1_grid():
    return {int(c, 16): float(v) for c, v in rows("e2m1_grid.txt")}


def test_multiplier_table():
    assert multipliers() == [1.00, 0.95, 0.90, 0.85, 0.80]


def hand_group():
    # g = 1, act_ms = 1: w = [6, 3.5 x 15], amax = 6, base scale amax / 6 = 1.
    #  1.00: scale 1; 6 -> 6 (err 0); 3.5 is a tie of 3 (word 5) and 4 (word 6) -> 4, err .25 x 15 = 3.75
    #  0.95: t = .95 -> E4M3 .9375; 6/.9375 = 6.4 -> 6, dq 5.625 (err .140625);
    #        3.5/.9375 = 3.73 -> 4, dq 3.75 (err .0625 x 15 = .9375); total 1.078125
    #  0.90: t = .90 -> E4M3 .875; 6/.875 = 6.86 -> 6, dq 5.25 (err .5625); 3.5/.875 = 4 -> exact; total .5625
    #  0.85: t = .85 -> E4M3 .875 (nearer than .8125): the same .5625, a tie kept by 0.90
    #  0.80: t = .80 -> E4M3 .8125; 6 -> 4.875 (err 1.265625); 3.5/.8125 = 4.31 -> 4, dq 3.25 (.9375); 2.203125
    w = np.full((1, 16), 3.5, dtype=np.float32)
    w[0, 0] = 6.0
    return w


def test_worked_example_clip_wins(oracle):
    codes, scales, chosen = oracle.quantize_nvfp4_clip(hand_group(), np.ones(16, np.float32), 1.0)
    assert chosen[0, 0] == 2
    assert scales[0, 0] == 0x36  # .875 = 1.75 * 2^-1: exponent 6, fraction 6
    words = np.stack([codes[0] & 15, codes[0] >> 4], axis=-1).reshape(16)
    assert words[0] == 7 and np.all(words[1:] == 6)  # 6.0 (word 7) and 4.0 (word 6)


def test_worked_example_act_ms_weighting(oracle):
    # act_ms[0] = 100: 1.00 -> 3.75; 0.95 -> 100 x .140625 + .9375 = 15.0; 0.90 -> 56.25; ...
    a = np.ones(16, np.float32)
    a[0] = 100.0
    codes, scales, chosen = oracle.quantize_nvfp4_clip(hand_group(), a, 1.0)
    assert chosen[0, 0] == 0 and scales[0, 0] == 0x38  # 1.0: exponent 7, fraction 0


def torch_e4m3_round(t):
    return torch.tensor(t, dtype=torch.float64).to(torch.float8_e4m3fn)


def nearest_e2m1(a, grid):
    best, bd = 0, np.inf
    for c in range(8):
        d = abs(grid[c] - a)
        if d < bd or (d == bd and c % 2 == 0):
            best, bd = c, d
    return best


def test_brute_force_argmin(oracle):
    grid = e2m1_grid()
    rng = np.random.default_rng(4)
    N, K, g = 6, 64, 0.01
    w = (rng.standard_normal((N, K)) * 0.05).astype(np.float32)
    w[:, ::16] *= 6.0  # an outlier per group
    a = rng.uniform(0.0, 3.0, size=K).astype(np.float32)
    codes, scales, chosen = oracle.quantize_nvfp4_clip(w, a, g)
    for r in range(N):
        for grp in range(K // 16):
            x = w[r, grp * 16:(grp + 1) * 16].astype(np.float64)
            amax = np.abs(x).max()
            errs, cands = [], []
            for mu in multipliers():
                t = ((mu * amax) / 6.0) / np.float64(np.float32(g))
                f8 = torch_e4m3_round(t)
                sv = float(f8.to(torch.float64))
                sc = int(f8.view(torch.uint8))
                mags = [nearest_e2m1(abs(v) / (sv * np.float64(np.float32(g))), grid) if sv else 0 for v in x]
                words = [m | (8 if v < 0 else 0) for m, v in zip(mags, x)]
                dq = np.array([grid[wd] * sv * np.float64(np.float32(g)) for wd in words])
                errs.append(float(np.sum(a[grp * 16:(grp + 1) * 16].astype(np.float64) * (x - dq) ** 2)))
                cands.append((sc, words))
            i = int(np.argmin(errs))  # the first of equal minima
            assert chosen[r, grp] == i
            assert scales[r, grp] == cands[i][0]
            got = np.stack([codes[r, grp * 8:(grp + 1) * 8] & 15, codes[r, grp * 8:(grp + 1) * 8] >> 4], -1).reshape(16)
            assert list(got) == cands[i][1]


def test_zero_group_and_decode_round_trip(oracle):
    rng = np.random.default_rng(6)
    N, K, g = 4, 48, 0.02
    w = (rng.standard_normal((N, K)) * 0.1).astype(np.float32)
    w[1, 16:32] = 0.0
    w[2, :16] = -0.0
    codes, scales, _ = oracle.quantize_nvfp4_clip(w, np.ones(K, np.float32), g)
    assert scales[1, 1] == 0 and np.all(codes[1, 8:16] == 0)
    assert scales[2, 0] == 0 and np.all(codes[2, :8] == 0x88)  # negative-zero words
    dq = oracle.dequantize_nvfp4(codes, scales, g, N, K)
    assert np.all(np.isfinite(dq))
    # every weight decodes within one grid unit (scale * g) of w: half the widest E2M1 gap (4 to
    # 6) is one unit, and the clipped largest weight is at most (1 / 0.8 - 1) * 6 = 1.5 units off
    sv = np.repeat(np.vectorize(oracle.e4m3fn_to_double)(scales), 16, axis=1) * np.float64(np.float32(g))
    assert np.all(np.abs(dq - w) <= 1.5 * sv * (1 + 1e-6) + 1e-30)
