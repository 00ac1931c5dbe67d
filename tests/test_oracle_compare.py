"""Pins of the parity checker itself (``oracle.compare``), CPU only.

Every tolerance-based GPU parity test goes through these predicates, so each
one is shown here to reject what it must reject: a bf16 result two units in
the last place away (either sign, across zero), an element that only the
magnitude floor could excuse when it is off by more than the floor, a float32
statistic 2e-5 off, a column sum with one term dropped or doubled.  The
magnitudes the oracle hands to the floor are pinned too: they are at least
the value itself, and the floor they give stays below one bf16 ulp of the
value for all but a tiny fraction of elements (a magnitude inflated by a
large factor would turn the floor into the real bar and fail that).
"""
import numpy as np
import pytest

from oracle import bf16
from oracle import boundary as ob
from oracle import compare


def _grid_values(n, seed):
    """Float64 values spread over signs and twenty binades, off the bf16 grid."""
    rng = np.random.default_rng(seed)
    mant = rng.uniform(1.0, 2.0, size=n)
    expo = rng.integers(-10, 10, size=n)
    sign = np.where(rng.random(n) < 0.5, -1.0, 1.0)
    return sign * np.ldexp(mant, expo)


def _step(bits, k):
    """The bf16 value k units in the last place above (k > 0) or below the
    value with these bits, walking the monotone order key (sign aware)."""
    key = bf16.order_key(bits) + k
    mag = np.abs(key).astype(np.uint16)
    return np.where(key < 0, mag | np.uint16(0x8000), mag).astype(np.uint16)


def test_bf16_mismatch_accepts_the_rounded_value_and_one_ulp():
    ref = _grid_values(20000, 1)
    bits = compare.bf16_bits(bf16.bf16_round(ref))
    zero_mag = np.zeros_like(ref)   # no floor: the ulp test alone decides
    for k in (-1, 0, 1):
        assert not compare.bf16_mismatch(_step(bits, k), ref, zero_mag).any(), k


@pytest.mark.parametrize("k", [-3, -2, 2, 3])
def test_bf16_mismatch_flags_two_or_more_ulps_on_both_signs(k):
    ref = _grid_values(20000, 2)
    assert (ref < 0).sum() > 5000 and (ref > 0).sum() > 5000
    bits = compare.bf16_bits(bf16.bf16_round(ref))
    # magnitude = |value|: the floor (2**-16 |value|) is far below one ulp
    bad = compare.bf16_mismatch(_step(bits, k), ref, np.abs(ref))
    assert bad.all()


def test_bf16_mismatch_across_zero():
    tiny = 2.0 ** -133                  # the smallest positive bf16
    ref = np.array([tiny, tiny, -tiny, 0.0, 0.0, 1e-3, -1e-3, tiny])
    gpu = np.array([-tiny, 0.0, 0.0, -0.0, tiny, -1e-3, 1e-3, tiny])
    gpu_bits = compare.bf16_bits(bf16.bf16_round(gpu))
    bad = compare.bf16_mismatch(gpu_bits, ref, np.zeros_like(ref))
    # +tiny vs -tiny are two steps apart through zero; -0 equals +0
    assert bad.tolist() == [True, False, False, False, False, True, True, False]


def test_magnitude_floor_excuses_only_errors_below_it():
    mag = np.ones(4)
    ref = np.full(4, 1e-4)              # a result cancelled far below its terms
    off = np.array([2.0 ** -14, -2.0 ** -14, 2.0 ** -17, -2.0 ** -17])
    gpu_bits = compare.bf16_bits(bf16.bf16_round(ref + off))
    bad = compare.bf16_mismatch(gpu_bits, ref, mag)
    floor_only = compare.bf16_floor_only(gpu_bits, ref, mag)
    assert bad.tolist() == [True, True, False, False]
    assert floor_only.tolist() == [False, False, True, True]
    # the same errors with no floor are all flagged (each is many ulps)
    assert compare.bf16_mismatch(gpu_bits, ref, np.zeros(4)).all()


def test_floor_only_counts_nothing_within_one_ulp():
    ref = _grid_values(5000, 3)
    bits = compare.bf16_bits(bf16.bf16_round(ref))
    assert not compare.bf16_floor_only(_step(bits, 1), ref, np.abs(ref) * 1e6).any()


def test_oracle_magnitudes_are_tight_enough_for_the_floor():
    rng = np.random.default_rng(4)
    n, h, t = 96, 1024, 4
    parts = (rng.standard_normal((t, n, h)) * 0.02).astype(np.float32)
    res = rng.standard_normal((n, h)).astype(np.float32)
    bias = (rng.standard_normal(h) * 0.01).astype(np.float32)
    gamma = (1 + rng.standard_normal(h) * 0.1).astype(np.float32)
    beta = (rng.standard_normal(h) * 0.1).astype(np.float32)
    for norm in ("layernorm", "rmsnorm"):
        fw = ob.forward_rows(parts, res, np.arange(n), bias, gamma, beta, eps=1e-5, p=0.1,
                             seed=7, norm=norm)
        dy = rng.standard_normal((n, h)).astype(np.float32)
        bw = ob.backward_rows(dy, fw["z"], fw["mask"], fw["mean"], fw["rstd"], gamma, None,
                              p=0.1, norm=norm)
        for value, mag in ((fw["out_exact"], fw["out_magnitude"]),
                           (bw["dz"], bw["dz_magnitude"])):
            assert np.all(mag >= np.abs(value) * (1 - 1e-12))
            ulp = np.ldexp(1.0, np.frexp(np.abs(value))[1] - 8)   # bf16 spacing at |value|
            wide = compare.FLOOR_REL * mag >= ulp
            assert wide.mean() < 1e-3, (norm, wide.mean())


def test_float32_layernorm_meets_the_bar_with_few_floor_only_elements():
    """A float32 evaluation of the LayerNorm output (the arithmetic a kernel
    does) passes the bar, and passes it through the floor alone on no more
    elements than floor_only_bound allows."""
    rng = np.random.default_rng(5)
    n, h = 256, 4096
    z = bf16.bf16_round(rng.standard_normal((n, h)))
    gamma = bf16.bf16_round(1 + rng.standard_normal(h) * 0.1)
    beta = bf16.bf16_round(rng.standard_normal(h) * 0.1)
    out, mean, rstd, mag = ob._norm_rows(z.astype(np.float64), gamma, beta, 1e-5, "layernorm")
    m32, r32 = mean.astype(np.float32), rstd.astype(np.float32)
    xh = ((z - m32[:, None]).astype(np.float32) * r32[:, None]).astype(np.float32)
    o32 = ((xh * gamma).astype(np.float32) + beta).astype(np.float32)
    bits = compare.bf16_bits(bf16.bf16_round(o32))
    assert not compare.bf16_mismatch(bits, out, mag).any()
    assert compare.bf16_floor_only(bits, out, mag).sum() <= compare.floor_only_bound(out.size)


@pytest.mark.parametrize("rel", [2e-5, -2e-5, 5e-5])
def test_f32_rel_mismatch_flags_2e5(rel):
    ref = np.array([10.0, -250.0, 0.1, -0.5, 1.0])
    gpu = np.where(np.abs(ref) >= 1, ref * (1 + rel), ref + rel)
    assert compare.f32_rel_mismatch(gpu, ref).all()


@pytest.mark.parametrize("rel", [0.0, 5e-6, -9e-6])
def test_f32_rel_mismatch_accepts_below_1e5(rel):
    ref = np.array([10.0, -250.0, 0.1, -0.5, 1.0])
    gpu = np.where(np.abs(ref) >= 1, ref * (1 + rel), ref + rel)
    assert not compare.f32_rel_mismatch(gpu, ref).any()


def _column_sums(seed, n=16384, h=64):
    rng = np.random.default_rng(seed)
    terms = rng.standard_normal((n, h))
    ref = terms.sum(axis=0)
    rss = np.sqrt((terms * terms).sum(axis=0))
    # float32 partial sums over 152 contiguous blocks, then float32 over blocks
    t32 = terms.astype(np.float32)
    parts = np.stack([blk.sum(axis=0, dtype=np.float32) for blk in np.array_split(t32, 152)])
    gpu = parts.sum(axis=0, dtype=np.float32)
    return terms, ref, rss, gpu


def test_colsum_mismatch_accepts_float32_rounding_at_the_70b_scale():
    terms, ref, rss, gpu = _column_sums(6)
    assert 120 < rss.mean() < 136            # sqrt(16384) = 128: the 70B-shape scale
    assert not compare.colsum_mismatch(gpu, ref, rss).any()


@pytest.mark.parametrize("how", ["dropped", "doubled", "sign"])
def test_colsum_mismatch_flags_one_wrong_term(how):
    terms, ref, rss, gpu = _column_sums(7)
    row = terms[1234]
    delta = {"dropped": -row, "doubled": row, "sign": -2 * row}[how]
    bad = compare.colsum_mismatch(gpu + delta.astype(np.float32), ref, rss)
    visible = np.abs(delta) > 2e-5 * rss   # beyond the tolerance plus float32 noise
    assert visible.sum() >= 60
    assert bad[visible].all()
