"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This module holds no arithmetic of the formats themselves (no decode, no
quantizer, no dot product). It draws random bits and random real numbers and
lays them out as the inputs' byte structures require:

* a counter-based generator (the SplitMix64 finaliser applied to
  ``seed, stream, index``), written once in torch integer ops so that the same
  call gives the same bits on the host and on a GPU;
* normal variates by the Box-Muller transform in fp64 on the host (small
  inputs only: activations and quantizer inputs);
* |N(0, sigma)| magnitudes for large tensors drawn on the device by an
  inverse-CDF table of 65,536 quantiles, so device generation stays
  integer-only and reproducible on the host row by row.

Workload recipes (shapes and distributions) follow the decode-step workloads
the format pages describe: pn3t / pn4t blocks with d = fp16(+-|N(0, 0.003)|),
codes uniform, pn3t reserved bits clear; NVFP4 with uniform E2M1 codes, E4M3FN
scales |N(0, 1)| rounded to nearest even, global multiplier 0.01; activations
N(0, 1).
"""
from __future__ import annotations

import statistics

import numpy as np
import torch

PN3T, PN4T, NVFP4 = 124, 125, 1004
BLOCK_WEIGHTS = {PN3T: 80, PN4T: 64}
BLOCK_BYTES = 34

_M64 = (1 << 64) - 1
_GOLD = 0x9E3779B97F4A7C15
_C1 = 0xBF58476D1CE4E5B9
_C2 = 0x94D049BB133111EB
_STREAM = 0xD1B54A32D192ED03


def _s64(v: int) -> int:
    """Reinterpret an unsigned 64-bit integer as a signed one (torch int64 constant)."""
    v &= _M64
    return v - (1 << 64) if v >= (1 << 63) else v


def _srl(z: torch.Tensor, s: int) -> torch.Tensor:
    """Logical right shift of int64 lanes (torch's >> is arithmetic)."""
    return (z >> s) & ((1 << (64 - s)) - 1)


def splitmix64(seed: int, stream: int, idx: torch.Tensor) -> torch.Tensor:
    """64 random bits per index (as int64) from (seed, stream, idx); device follows idx."""
    key = (seed * _GOLD + stream * _STREAM) & _M64
    z = idx.to(torch.int64) * _s64(_GOLD) + _s64(key + _GOLD)
    z = (z ^ _srl(z, 30)) * _s64(_C1)
    z = (z ^ _srl(z, 27)) * _s64(_C2)
    return z ^ _srl(z, 31)


def uniform01(seed: int, stream: int, n: int) -> np.ndarray:
    """n uniforms in (0, 1) from the top 53 bits, fp64, host."""
    z = splitmix64(seed, stream, torch.arange(n, dtype=torch.int64))
    top = _srl(z, 11).numpy().astype(np.float64)
    return (top + 0.5) * (2.0 ** -53)


def normal(seed: int, stream: int, shape, sigma: float = 1.0) -> np.ndarray:
    """N(0, sigma^2) by Box-Muller in fp64 on the host, returned as fp32."""
    n = int(np.prod(shape))
    u1 = uniform01(seed, stream, n)
    u2 = uniform01(seed, stream + 1, n)
    z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
    return (sigma * z).astype(np.float32).reshape(shape)


_abs_normal_cache: dict = {}


def _abs_normal_quantiles() -> np.ndarray:
    """65,536 quantiles of |N(0, 1)| at probabilities (i + 0.5) / 65536, fp64."""
    if "q" not in _abs_normal_cache:
        nd = statistics.NormalDist()
        _abs_normal_cache["q"] = np.array(
            [nd.inv_cdf(0.5 + 0.5 * (i + 0.5) / 65536.0) for i in range(65536)], dtype=np.float64)
    return _abs_normal_cache["q"]


def fp16_abs_normal_table(sigma: float) -> np.ndarray:
    """uint16 bit patterns of fp16(sigma * |N(0,1)| quantile), numpy round-to-nearest-even."""
    q = (sigma * _abs_normal_quantiles()).astype(np.float16)
    return q.view(np.uint16)


def e4m3_abs_normal_table() -> np.ndarray:
    """uint8 E4M3FN words of |N(0,1)| quantiles, rounded to nearest even by torch."""
    q = torch.from_numpy(_abs_normal_quantiles().astype(np.float32))
    return q.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _to_i16(v: torch.Tensor) -> torch.Tensor:
    """int64 values in [0, 65536) -> the int16 with the same 16 bits."""
    v = v & 0xFFFF
    return (v - ((v & 0x8000) << 1)).to(torch.int16)


def pn_random_blocks(type_: int, N: int, K: int, seed: int, stream: int = 0,
                     d_sigma: float = 0.003, device="cpu", rows: torch.Tensor | None = None,
                     out: torch.Tensor | None = None) -> torch.Tensor:
    """Random PN blocks: d = fp16(+-|N(0, d_sigma)|) (random sign per block), codes uniform,
    pn3t reserved bits 15 and 31 clear. Returns uint8 [len(rows) or N][K/BLK * 34].

    ``rows`` selects row indices to generate (default: all); any row is reproducible
    on its own, which is how large device tensors are spot-checked on the host.
    """
    blk = BLOCK_WEIGHTS[type_]
    assert K % blk == 0
    nb = K // blk
    if rows is None:
        rows = torch.arange(N, dtype=torch.int64, device=device)
    else:
        rows = rows.to(device=device, dtype=torch.int64)
    R = rows.numel()
    bidx = (rows[:, None] * nb + torch.arange(nb, dtype=torch.int64, device=device)[None, :]).reshape(-1)
    halves = torch.empty((bidx.numel(), 17), dtype=torch.int16, device=device)
    table = torch.from_numpy(fp16_abs_normal_table(d_sigma).astype(np.int64)).to(device)
    r = splitmix64(seed, stream * 8 + 0, bidx)
    dbits = table[r & 0xFFFF] | (_srl(r, 16) & 1) << 15
    halves[:, 0] = _to_i16(dbits)
    mask = 0x7FFF if type_ == PN3T else 0xFFFF
    for j in range(4):
        z = splitmix64(seed, stream * 8 + 1 + j, bidx)
        for q in range(4):
            halves[:, 1 + 4 * j + q] = _to_i16(_srl(z, 16 * q) & mask)
    blocks = halves.view(torch.uint8).reshape(R, nb * BLOCK_BYTES)
    if out is not None:
        out.copy_(blocks)
        return out
    return blocks


def nvfp4_random(N: int, K: int, seed: int, stream: int = 0, device="cpu",
                 rows: torch.Tensor | None = None):
    """Random NVFP4 weights: codes uniform over the 16 E2M1 words (uint8 [R][K/2], low nibble
    = even k), scales E4M3FN of |N(0,1)| (uint8 [R][K/16]), global multiplier 0.01."""
    assert K % 16 == 0
    if rows is None:
        rows = torch.arange(N, dtype=torch.int64, device=device)
    else:
        rows = rows.to(device=device, dtype=torch.int64)
    R = rows.numel()
    nwords = K // 16  # one 64-bit draw = 8 code bytes = 16 codes
    widx = (rows[:, None] * nwords + torch.arange(nwords, dtype=torch.int64, device=device)[None, :]).reshape(-1)
    z = splitmix64(seed, stream * 8 + 0, widx)
    codes = torch.empty((widx.numel(), 8), dtype=torch.uint8, device=device)
    for q in range(8):
        codes[:, q] = (_srl(z, 8 * q) & 0xFF).to(torch.uint8)
    codes = codes.reshape(R, K // 2)
    table = torch.from_numpy(e4m3_abs_normal_table().astype(np.int64)).to(device)
    sidx = widx  # one scale per 16 weights, same counter space, separate stream
    s = splitmix64(seed, stream * 8 + 1, sidx)
    scales = table[s & 0xFFFF].to(torch.uint8).reshape(R, K // 16)
    return codes, scales, 0.01


def activations(M: int, K: int, seed: int, stream: int = 7) -> np.ndarray:
    """x ~ N(0, 1), fp32 [M][K], host."""
    return normal(seed, stream * 16, (M, K), 1.0)


def activations_bf16(M: int, K: int, seed: int, stream: int = 7) -> np.ndarray:
    """x ~ N(0, 1) rounded to bf16 (torch round-to-nearest-even); raw uint16 words [M][K]."""
    x = torch.from_numpy(activations(M, K, seed, stream))
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def quantizer_weights(N: int, K: int, seed: int, sigma: float = 0.02,
                      outlier_frac: float = 0.001, outlier_mult: float = 8.0) -> np.ndarray:
    """fp32 [N][K] ~ N(0, sigma^2) with a fraction of entries multiplied by outlier_mult;
    row 0 all zero (canonical zero groups); row 1 all positive (every block's largest weight
    is positive, so every block gets a negative d)."""
    w = normal(seed, 3 * 16, (N, K), sigma)
    u = uniform01(seed, 3 * 16 + 5, N * K).reshape(N, K)
    w = np.where(u < outlier_frac, w * np.float32(outlier_mult), w).astype(np.float32)
    if N > 0:
        w[0, :] = 0.0
    if N > 1:
        w[1, :] = np.abs(w[1, :])
    return w
