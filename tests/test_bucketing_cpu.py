"""Host-side length bucketing (CPU only): the properties the reading promises."""
import numpy as np
import pytest

from sp_boundary_norm_gb300 import bucketing as bk
from sp_boundary_norm_gb300 import workloads as wl


def test_length_cv_definition():
    assert bk.length_cv([]) == 0.0 and bk.length_cv([7]) == 0.0
    assert bk.length_cv([5, 5, 5]) == 0.0
    # population std / mean: [2, 4] -> std 1, mean 3
    assert bk.length_cv([2, 4]) == pytest.approx(1 / 3)
    # the packed workload's lengths: CV 0.34, above the page's 0.18 bound
    assert bk.length_cv(wl.ragged_lengths()) == pytest.approx(0.3433, abs=1e-4)


@pytest.mark.parametrize("max_cv", [0.0, 0.05, 0.15, 0.3, 10.0])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_buckets_partition_and_respect_the_bound(max_cv, seed):
    rng = np.random.default_rng(seed)
    lens = [int(x) for x in np.clip(np.rint(rng.lognormal(np.log(4096), 0.6, 64)), 512, 32768)]
    buckets = bk.bucket_by_tokens(lens, max_cv=max_cv)
    seen = sorted(i for b in buckets for i in b.indices)
    assert seen == list(range(len(lens)))
    for b in buckets:
        assert b.length_cv <= max_cv + 1e-12
        assert list(b.lengths) == [lens[i] for i in b.indices]
        assert b.tokens == sum(b.lengths)
        assert b.cu_seqlens[0] == 0 and b.cu_seqlens[-1] == b.tokens
        assert np.all(np.diff(b.cu_seqlens) == np.array(b.lengths))
    # buckets are runs of consecutive lengths in sorted order
    flat = [lens[i] for b in buckets for i in b.indices]
    assert flat == sorted(lens)
    if max_cv >= 10:
        assert len(buckets) == 1


def test_greedy_cut_is_maximal():
    """A bucket is closed only when the next sequence would break the bound."""
    lens = [100, 101, 102, 150, 151, 400]
    buckets = bk.bucket_by_tokens(lens, max_cv=0.05)
    for a, b in zip(buckets, buckets[1:]):
        nxt = lens[b.indices[0]]
        assert bk.length_cv(list(a.lengths) + [nxt]) > 0.05
    assert [b.lengths for b in buckets] == [(100, 101, 102), (150, 151), (400,)]


def test_token_budget():
    lens = [1000] * 10 + [5000]
    buckets = bk.bucket_by_tokens(lens, max_cv=1.0, max_tokens=3000)
    assert all(b.tokens <= 3000 or len(b.lengths) == 1 for b in buckets)
    assert [b.tokens for b in buckets] == [3000, 3000, 3000, 1000, 5000]


def test_packed_workload_is_split_below_the_bound():
    lens = wl.ragged_lengths()
    buckets = bk.bucket_by_tokens(lens, max_cv=0.15)
    assert len(buckets) > 1 and all(b.length_cv <= 0.15 for b in buckets)
    assert sum(b.tokens for b in buckets) == sum(lens)


def test_invalid_arguments():
    with pytest.raises(ValueError):
        bk.bucket_by_tokens([1, 2], max_cv=-1)
    with pytest.raises(ValueError):
        bk.bucket_by_tokens([1, -2])
    with pytest.raises(ValueError):
        bk.bucket_by_tokens([1, 2], max_tokens=0)


def test_regroup_packed_moves_whole_sequences_and_reshards():
    import torch
    lens = (5, 17, 3, 40, 1, 9)
    w = wl.Workload("rg", t=4, b=1, s=sum(lens), h=8, seqlens=lens, draw_seed=3)
    inp = wl.forward_inputs(w, "cpu")
    dy = wl.backward_inputs(w, "cpu")["dy"]
    cu = wl.cu_seqlens(lens)
    order, blens = (3, 0, 5), (40, 5, 9)
    wb, parts, (res, dyb) = wl.regroup_packed(w, order, blens, inp["partials"],
                                              [inp["residual"], dy])
    assert wb.s == 54 and wb.seqlens == blens and wb.t == w.t
    assert [x.shape[1] for x in res] == wb.shard_sizes() == [x.shape[1] for x in dyb]
    full_res = torch.cat(inp["residual"], dim=1)
    got_res = torch.cat(res, dim=1)
    pos = 0
    for i, n in zip(order, blens):
        assert torch.equal(got_res[:, pos:pos + n], full_res[:, cu[i]:cu[i + 1]])
        for P, Pb in zip(inp["partials"], parts):
            assert torch.equal(Pb[:, pos:pos + n], P[:, cu[i]:cu[i + 1]])
        pos += n
    with pytest.raises(ValueError):
        wl.regroup_packed(w, (3,), (41,), inp["partials"], [])
    with pytest.raises(ValueError):
        wl.regroup_packed(w.with_(seqlens=()), (0,), (5,), inp["partials"], [])


def test_regroup_packed_of_the_buckets_covers_every_token_once():
    import torch
    w = wl.WORKLOADS["ragged"].with_(h=8)
    inp = wl.forward_inputs(w, "cpu")
    tok = torch.arange(w.s, dtype=torch.float32).reshape(1, -1, 1).expand(1, w.s, 8)
    seen = []
    for b in bk.bucket_by_tokens(w.seqlens, max_cv=0.15):
        _, parts, _ = wl.regroup_packed(w, b.indices, b.lengths, [tok], [])
        seen.append(parts[0][0, :, 0])
    assert torch.equal(torch.sort(torch.cat(seen)).values, torch.arange(w.s, dtype=torch.float32))
