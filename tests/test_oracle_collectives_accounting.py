"""Pins of the oracle's collectives and accounting (CPU only).

Against the lesson "第 7 课：序列并行 SP": the ring identity and volume law of
§4, the shape-trace exercise's printed result, and the 70B arithmetic.
"""
import os

import numpy as np
import pytest

from oracle import accounting as acc
from oracle import collectives as coll

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16_like(rng, shape, scale=1.0):
    # values with few significant bits so bf16 storage is exact
    return (np.round(rng.standard_normal(shape) * 64) / 64 * scale).astype(np.float32)


@pytest.mark.parametrize("t,b,s,h", [(1, 1, 8, 8), (2, 1, 16, 8), (3, 2, 9, 16),
                                     (8, 1, 64, 24), (8, 2, 37, 8), (5, 1, 3, 8)])
def test_allreduce_equals_allgather_of_reducescatter(t, b, s, h):
    rng = np.random.default_rng(t * 100 + s)
    partials = [_bf16_like(rng, (b, s, h)) for _ in range(t)]
    shards, _ = coll.reduce_scatter_seq(partials)
    gathered, _ = coll.all_gather_seq(shards)
    ar = coll.all_reduce(partials)
    for j in range(t):
        assert gathered[j].shape == (b, s, h)
        assert np.array_equal(gathered[j].view(np.uint32), ar[j].view(np.uint32))


@pytest.mark.parametrize("t,b,s,h", [(2, 1, 16, 8), (4, 2, 32, 16), (8, 1, 64, 8)])
def test_counted_volume_matches_volume_law(t, b, s, h):
    rng = np.random.default_rng(7)
    partials = [_bf16_like(rng, (b, s, h)) for _ in range(t)]
    size = b * s * h * 2
    shards, rs_bytes = coll.reduce_scatter_seq(partials)
    _, ag_bytes = coll.all_gather_seq(shards)
    assert rs_bytes == [acc.volume_reduce_scatter(size, t)] * t
    assert ag_bytes == [acc.volume_all_gather(size, t)] * t
    # an all-reduce costs exactly one reduce-scatter plus one all-gather
    assert rs_bytes[0] + ag_bytes[0] == acc.volume_all_reduce(size, t)


def test_volume_of_tp_equals_tp_plus_sp():
    for t in (2, 4, 8, 16):
        for (b, s, h) in ((1, 4096, 4096), (1, 16384, 8192), (2, 2048, 5120)):
            assert acc.volume_per_block(b, s, h, t, sp=True) == \
                acc.volume_per_block(b, s, h, t, sp=False)
            size = b * s * h * 2
            assert acc.volume_per_block(b, s, h, t, sp=False) == 4 * (t - 1) * size // t
    # 70B layer input (b=1, s=16384, h=8192, bf16), t=8: 7/8 of 268,435,456 B
    assert acc.volume_reduce_scatter(16384 * 8192 * 2, 8) == 234_881_024


def test_uneven_shards_cover_every_token_once():
    for n in (1, 7, 42823, 4096):
        for t in (1, 3, 8, 16):
            o = coll.shard_offsets(n, t)
            assert o[0] == 0 and o[-1] == n
            sizes = np.diff(o)
            assert sizes.min() >= 0 and sizes.max() - sizes.min() <= 1


def test_transpose_identity_allgather_vs_seq_sum():
    rng = np.random.default_rng(3)
    t, b, s, h = 4, 2, 10, 8
    x = [rng.standard_normal((b, e, h)) for e in np.diff(coll.shard_offsets(s, t))]
    y = [rng.standard_normal((b, s, h)) for _ in range(t)]
    ag, _ = coll.all_gather_seq(x)
    rs = coll.sum_seq_shards(y, t)
    lhs = sum(float((a * c).sum()) for a, c in zip(ag, y))
    rhs = sum(float((a * c).sum()) for a, c in zip(x, rs))
    assert lhs == pytest.approx(rhs, rel=1e-12)


def _golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].split()
            if line:
                rows.append(line)
    return rows


def test_shape_trace_reproduces_printed_result():
    seq = hidden = 4096
    tp = 8
    traces = {"tp_only": acc.block_shape_trace(seq, hidden, tp, enable_sp=False),
              "sp": acc.block_shape_trace(seq, hidden, tp, enable_sp=True)}
    peaks = {}
    for row in _golden("trace_block_s4096_h4096_t8.txt"):
        mode, kind = row[0], row[1]
        if kind == "shape":
            region, s, h = row[2], int(row[3]), int(row[4])
            hits = [e for e in traces[mode] if e.region == region and e.resident]
            assert hits and (hits[0].s, hits[0].h) == (s, h), (mode, region)
        elif kind == "peak_mb":
            peaks[mode] = float(row[2])
    m_tp = acc.peak_resident_bytes(traces["tp_only"])
    m_sp = acc.peak_resident_bytes(traces["sp"])
    assert round(m_tp / 1e6, 1) == peaks["tp_only"]
    assert round(m_sp / 1e6, 1) == peaks["sp"]
    assert m_tp == 33_554_432 and m_sp == 4_194_304 and m_sp * tp == m_tp
    # the transient full-sequence buffers of g, the row output and g*
    transient = [e.region for e in traces["sp"] if not e.resident]
    assert transient == ["g (all-gather seq)", "row_linear", "row_out (full h)",
                         "g* (reduce-scatter seq)"]


@pytest.mark.parametrize("tp", [2, 4, 8])
def test_shape_trace_peak_ratio_is_tp(tp):
    for seq, hidden in ((2048, 1024), (8192, 4096)):
        m_tp = acc.peak_resident_bytes(acc.block_shape_trace(seq, hidden, tp, False))
        m_sp = acc.peak_resident_bytes(acc.block_shape_trace(seq, hidden, tp, True))
        assert m_sp * tp == m_tp


def test_activation_memory_70b_example():
    g = {r[0]: float(r[1]) for r in _golden("activation_70b.txt")}
    s, h, t, L = int(g["seq"]), int(g["hidden"]), int(g["tp"]), int(g["layers"])
    tp_layer = acc.non_tp_activation_bytes(s, 1, h, t, sp=False)
    sp_layer = acc.non_tp_activation_bytes(s, 1, h, t, sp=True)
    assert tp_layer == 1_342_177_280 and sp_layer == 167_772_160
    assert round(tp_layer / 1e9, 2) == g["tp_only_layer_gb"]
    assert round(L * tp_layer / 1e9, 1) == g["tp_only_total_gb"]
    assert round(sp_layer / 1e6, 1) == g["sp_layer_mb"]
    assert round(L * sp_layer / 1e9, 1) == g["sp_total_gb"]
    assert round(L * (tp_layer - sp_layer) / 1e9) == g["saved_gb"]
    assert 1 - sp_layer / tp_layer == g["saved_fraction_t8"]
