"""Pins of the oracle's Philox4x32-10 and bf16 rounding (CPU only)."""
import os

import numpy as np
import pytest
import torch

from oracle import bf16, philox

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _kat_rows():
    rows = []
    with open(os.path.join(GOLDEN, "philox4x32_kat.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].split()
            if line:
                rows.append((int(line[0]), [int(x, 16) for x in line[1:]]))
    return rows


@pytest.mark.parametrize("rounds,vals", _kat_rows())
def test_philox_known_answers(rounds, vals):
    ctr, key, want = vals[0:4], vals[4:6], vals[6:10]
    got = philox.philox4x32([np.array([c], dtype=np.uint32) for c in ctr], key, rounds)
    assert [int(g[0]) for g in got] == want


def test_philox_vectorised_matches_scalar_calls():
    rng = np.random.default_rng(5)
    ctr = [rng.integers(0, 2**32, size=64, dtype=np.uint64) for _ in range(4)]
    key = (0x12345678, 0x9ABCDEF0)
    batch = philox.philox4x32(ctr, key)
    for i in range(64):
        one = philox.philox4x32([np.array([c[i]]) for c in ctr], key)
        assert [int(w[0]) for w in one] == [int(w[i]) for w in batch]


def test_element_uniforms_statistics_and_keying():
    idx = np.arange(1 << 18, dtype=np.int64)
    u = philox.element_uniforms(1234, 0, idx)
    # uniform top byte: chi-square with 255 dof, generous 6-sigma bound
    counts = np.bincount((u >> 24).astype(np.int64), minlength=256)
    exp = idx.size / 256
    chi2 = ((counts - exp) ** 2 / exp).sum()
    assert chi2 < 255 + 6 * np.sqrt(2 * 255)
    # a different seed or offset gives an unrelated stream
    assert np.mean(philox.element_uniforms(1235, 0, idx) == u) < 1e-3
    assert np.mean(philox.element_uniforms(1234, 1, idx) == u) < 1e-3
    # the draw of an element depends on its index only, not on the batch it is in
    sub = idx[1000:1100][::-1]
    assert np.array_equal(philox.element_uniforms(1234, 0, sub), u[sub])


def _f32_samples(n, seed):
    rng = np.random.default_rng(seed)
    bits = rng.integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
    # force exact ties (low half == 0x8000) on a quarter of them
    bits[: n // 4] = (bits[: n // 4] & np.uint32(0xFFFF0000)) | np.uint32(0x8000)
    special = np.array([0.0, -0.0, 1.0, -1.0, np.inf, -np.inf,
                        3.3895313892515355e38, 3.40e38, 1e-40, -1e-45,
                        float.fromhex("0x1.fefffep127"), float.fromhex("0x1.ff0000p127")],
                       dtype=np.float32)
    vals = np.concatenate([bits.view(np.float32), special])
    return vals[np.isfinite(vals) | np.isinf(vals)]


def test_bf16_round_matches_torch_cast_on_float32():
    vals = _f32_samples(200000, 0)
    ours = bf16.bf16_round(vals)
    ref = torch.from_numpy(vals.copy()).to(torch.bfloat16).to(torch.float32).numpy()
    same = (ours.view(np.uint32) == ref.view(np.uint32))
    assert same.all(), vals[~same][:10]


def _all_finite_bf16_sorted():
    bits = np.arange(0, 0x7F80, dtype=np.uint32)     # +0 .. largest finite
    pos = (bits << 16).view(np.float32).astype(np.float64)
    return pos, bits


def _brute_force_round(x):
    """Nearest finite bf16 by search over all of them; ties to even bits."""
    grid, bits = _all_finite_bf16_sorted()
    ax = abs(x)
    if ax >= float.fromhex("0x1.fep127") + 2.0 ** (127 - 8):
        return np.copysign(np.inf, x)
    i = np.searchsorted(grid, ax)
    cands = [j for j in (i - 1, i) if 0 <= j < grid.size]
    best = min(cands, key=lambda j: (abs(grid[j] - ax), bits[j] & 1))
    return np.copysign(grid[best], x)


def test_bf16_round_from_float64_brute_force():
    rng = np.random.default_rng(1)
    grid, _ = _all_finite_bf16_sorted()
    xs = []
    # midpoints between neighbours, and one float64 ulp either side of them:
    # the cases where rounding through float32 first would differ
    for j in rng.integers(1, grid.size - 2, size=300):
        mid = (grid[j] + grid[j + 1]) / 2
        xs += [mid, np.nextafter(mid, 0), np.nextafter(mid, np.inf)]
    xs += list(rng.standard_normal(300) * 10.0 ** rng.integers(-40, 38, size=300))
    xs += [float.fromhex("0x1.fep127") * 1.001, 2.0 ** -133 * 0.5, 2.0 ** -133 * 0.5000001]
    xs = np.array(xs, dtype=np.float64)
    xs = np.concatenate([xs, -xs])
    ours = bf16.bf16_round(xs).astype(np.float64)
    ref = np.array([_brute_force_round(x) for x in xs])
    assert np.array_equal(ours, ref) and np.array_equal(np.signbit(ours), np.signbit(ref))


def test_bf16_bits_round_trip_and_order_key():
    bits = np.arange(0, 0x7F80, dtype=np.uint16)
    vals = bf16.bits_to_f32(bits)
    assert np.array_equal(bf16.f32_to_bits(vals), bits)
    key = bf16.order_key(bits)
    assert np.all(np.diff(key) == 1)
    neg = bf16.order_key(bits | np.uint16(0x8000))
    assert neg[0] == key[0] == 0 and np.all(np.diff(neg) == -1)
    with pytest.raises(ValueError):
        bf16.f32_to_bits(np.array([1.0 + 2 ** -20], dtype=np.float32))
