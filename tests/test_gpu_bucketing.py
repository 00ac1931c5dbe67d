"""The boundary on length buckets: host bucketing feeding the packed entry points.

"分布式训练为什么一开 Sequence Parallel 就开始省显存却抖吞吐" (coreui.cn), section
on shape drift: its first lever is to tighten the length buckets
(``bucket_by_tokens(batch, max_cv=0.15)``) before the sequence-parallel
step.  Here the packed workload's eight sequences (length CV 0.34) are
bucketed with that bound, each bucket is laid out as a packed batch of its
own (the sequences' tokens moved, not recomputed), and the fused forward and
the backward run on it with the bucket's ``cu_seqlens``; every element of
every bucket is compared with the oracle.  With dropout off, every token's
results in the buckets equal its results in the unbucketed batch bit for
bit: bucketing regroups tokens and changes no token-wise value ("第 7 课：
序列并行 SP" §3).
"""
import numpy as np
import pytest
import torch

from sp_boundary_norm_gb300 import bucketing as bk
from sp_boundary_norm_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

C = pytest.importorskip("_cases")


@pytest.fixture(scope="module", autouse=True)
def _built(lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield


def _buckets(w):
    buckets = bk.bucket_by_tokens(w.seqlens, max_cv=0.15)
    assert len(buckets) >= 2 and all(b.length_cv <= 0.15 for b in buckets)
    assert sorted(i for b in buckets for i in b.indices) == list(range(len(w.seqlens)))
    return buckets


def test_boundary_on_each_length_bucket_every_element():
    w = wl.WORKLOADS["ragged"]
    inp = wl.forward_inputs(w, C.DEV)
    dy = wl.backward_inputs(w, C.DEV)["dy"]
    for b in _buckets(w):
        wb, parts, (res, dyb) = wl.regroup_packed(w, b.indices, b.lengths, inp["partials"],
                                                  [inp["residual"], dy])
        assert wb.s == b.tokens and np.array_equal(wl.cu_seqlens(wb.seqlens), b.cu_seqlens)
        ib = dict(inp, partials=parts, residual=res)
        cu = torch.from_numpy(b.cu_seqlens).to(C.DEV)
        fwd = C.run_fwd(wb, ib, n_gather=1, cu_seqlens=cu)
        torch.cuda.synchronize()
        C.sp.check_device_status(C.DEV)
        f = C.full_fwd_check(wb, ib, fwd)
        out = C.run_bwd(wb, fwd, ib["gamma"], dyb, None, n_gather=1, cu_seqlens=cu)
        torch.cuda.synchronize()
        C.sp.check_device_status(C.DEV)
        g = C.full_bwd_check(wb, fwd, ib["gamma"], dyb, None, out)
        print(f"\nbucket {b.lengths} (CV {b.length_cv:.3f}, {b.tokens} tokens): "
              f"forward {f}, backward {g}")


def test_bucketing_changes_no_token_wise_result_without_dropout():
    w = wl.WORKLOADS["ragged"].with_(p=0.0)
    inp = wl.forward_inputs(w, C.DEV)
    whole = C.run_fwd(w, inp, n_gather=1)
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    for b in _buckets(w):
        wb, parts, (res, z_exp, mean_exp, rstd_exp) = wl.regroup_packed(
            w, b.indices, b.lengths, inp["partials"],
            [inp["residual"], whole["z"], [m[..., None] for m in whole["mean"]],
             [r[..., None] for r in whole["rstd"]]])
        _, _, (o_exp,) = wl.regroup_packed(w, b.indices, b.lengths, [], [whole["gathered"]])
        ib = dict(inp, partials=parts, residual=res)
        got = C.run_fwd(wb, ib, n_gather=1, cu_seqlens=torch.from_numpy(b.cu_seqlens).to(C.DEV))
        torch.cuda.synchronize()
        C.sp.check_device_status(C.DEV)
        cat = lambda lst: torch.cat(list(lst), dim=1)
        assert torch.equal(cat(got["z"]).view(torch.int16), cat(z_exp).view(torch.int16))
        assert bool((cat(got["mask"]) == 1).all())
        assert torch.equal(cat(got["mean"]), cat(mean_exp)[..., 0])
        assert torch.equal(cat(got["rstd"]), cat(rstd_exp)[..., 0])
        assert torch.equal(got["gathered"][0].view(torch.int16), cat(o_exp).view(torch.int16))
