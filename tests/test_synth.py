"""The seeded input generator (block_quantized_weight_pn3t_gb300/synth.py) on the CPU.

- Its counter-based generator is SplitMix64: output i of the stream seeded with `key` is the
  SplitMix64 finaliser of key + (i + 1) * 0x9E3779B97F4A7C15. Pinned to the published first
  outputs for state 0 and to a plain-Python SplitMix64 written from its definition (stateful
  next(), Python integers), which checks the torch int64 wrap-around and logical shifts.
- Any subset of rows regenerates bit for bit (the GPU parity tests regenerate sampled rows of
  full-size device tensors on the host this way).
- The workload recipes: pn3t reserved bits clear, finite d with random sign, codes over the
  whole range; NVFP4 scales finite E4M3FN magnitudes, g = 0.01; activations N(0, 1).
"""
import numpy as np
import torch

from block_quantized_weight_pn3t_gb300 import synth

M64 = (1 << 64) - 1


class SplitMix64:
    """Plain-Python SplitMix64: state += golden gamma; mix the state."""

    def __init__(self, state):
        self.state = state & M64

    def next(self):
        self.state = (self.state + 0x9E3779B97F4A7C15) & M64
        z = self.state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
        return z ^ (z >> 31)


def u64(t):
    return [int(v) & M64 for v in t]


def test_published_first_outputs_for_state_zero():
    assert u64(synth.splitmix64(0, 0, torch.arange(3))) == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4,
                                                              0x06C45D188009454F]


def test_matches_a_plain_splitmix64():
    for seed, stream in [(0, 0), (1, 0), (20261202, 3), (2**40 + 7, 17), (12345, 2**20)]:
        key = (seed * 0x9E3779B97F4A7C15 + stream * 0xD1B54A32D192ED03) & M64
        ref = SplitMix64(key)
        want = [ref.next() for _ in range(1000)]
        assert u64(synth.splitmix64(seed, stream, torch.arange(1000))) == want
        idx = torch.tensor([5, 999, 0, 123456789, 2**40])
        # output i is the (i + 1)-th step from the key, whatever order the indices come in
        for i, got in zip(idx.tolist(), u64(synth.splitmix64(seed, stream, idx))):
            assert got == SplitMix64(key + i * 0x9E3779B97F4A7C15).next()


def test_pn_rows_regenerate_bit_for_bit():
    for t, K in ((synth.PN3T, 640), (synth.PN4T, 1024)):
        full = synth.pn_random_blocks(t, 300, K, seed=9, stream=2)
        rows = torch.tensor([0, 7, 128, 299, 150])
        assert torch.equal(synth.pn_random_blocks(t, 300, K, seed=9, stream=2, rows=rows), full[rows])
        assert not torch.equal(synth.pn_random_blocks(t, 300, K, seed=9, stream=3), full)


def test_pn_workload_recipe():
    for t, K in ((synth.PN3T, 80 * 64), (synth.PN4T, 64 * 80)):
        W = synth.pn_random_blocks(t, 200, K, seed=4).numpy().reshape(-1, 34)
        d = W[:, 0:2].copy().view(np.uint16).reshape(-1)
        assert np.all((d & 0x7C00) != 0x7C00)  # finite
        neg = (d >> 15).mean()
        assert 0.45 < neg < 0.55  # random sign per block
        dv = np.abs(d.view(np.float16).astype(np.float64))
        assert 0.0015 < np.median(dv) < 0.0025  # |N(0, 0.003)|: median 0.003 * 0.674
        words = W[:, 2:].copy().view(np.uint32)
        if t == synth.PN3T:
            assert np.all(words & 0x80008000 == 0)  # reserved bits 15 and 31 clear
            codes = np.concatenate([(words >> (3 * (j // 2) + 16 * (j % 2))) & 7 for j in range(10)])
            assert set(np.unique(codes)) == set(range(8))
        else:
            assert np.any(words & 0x80008000)  # every bit is a code bit
            codes = np.concatenate([(words >> (4 * (j // 2) + 16 * (j % 2))) & 15 for j in range(8)])
            assert set(np.unique(codes)) == set(range(16))


def test_nvfp4_rows_and_recipe():
    codes, scales, g = synth.nvfp4_random(200, 512, seed=3)
    rows = torch.tensor([1, 199, 50])
    c2, s2, g2 = synth.nvfp4_random(200, 512, seed=3, rows=rows)
    assert torch.equal(c2, codes[rows]) and torch.equal(s2, scales[rows]) and g2 == g == 0.01
    assert codes.shape == (200, 256) and scales.shape == (200, 32)
    nib = np.concatenate([codes.numpy() & 15, codes.numpy() >> 4]).reshape(-1)
    assert set(np.unique(nib)) == set(range(16))
    s = scales.numpy()
    assert np.all(s & 0x80 == 0) and np.all(s & 0x7F != 0x7F)  # positive, finite E4M3FN words
    sv = scales.view(torch.float8_e4m3fn).to(torch.float32).numpy()
    assert 0.55 < np.median(sv) < 0.8  # |N(0, 1)|: median 0.674


def test_activations():
    x = synth.activations(4, 50000, seed=1)
    assert x.dtype == np.float32 and x.shape == (4, 50000)
    assert abs(float(x.mean())) < 0.02 and abs(float(x.std()) - 1.0) < 0.02
    assert np.array_equal(x, synth.activations(4, 50000, seed=1))
    xb = synth.activations_bf16(2, 64, seed=1)
    back = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(back, torch.from_numpy(synth.activations(2, 64, seed=1)).to(torch.bfloat16)
                          .to(torch.float32).numpy())
