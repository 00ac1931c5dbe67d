"""Host-side pieces of bench.py on CPU: the algorithmic byte counts, the
launch count a step claims, and the bucketed step's composition."""
import os
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from sp_boundary_norm_gb300 import bucketing as bk  # noqa: E402
from sp_boundary_norm_gb300 import workloads as wl  # noqa: E402


def test_byte_counts_of_the_70b_shape():
    # forward 23h + 8, backward 9h + 8 per token at t = 8, one gathered copy
    assert bench.fwd_bytes_per_token(8, 8192, 1) * 16384 == 3_087_138_816
    assert bench.bwd_bytes_per_token(8192, 1) * 16384 == 1_208_090_624
    # RMSNorm stores no mean: 4 bytes fewer per token in each direction
    assert bench.fwd_bytes_per_token(8, 8192, 1, "rmsnorm") == 23 * 8192 + 4
    # one gathered copy per rank adds 2h per extra copy
    assert bench.fwd_bytes_per_token(8, 8192, 8) - bench.fwd_bytes_per_token(8, 8192, 1) \
        == 7 * 2 * 8192
    # the unfused forward moves 31h + 8, the unfused backward through g 27h + 8
    assert bench.unfused_fwd_bytes_per_token(8, 8192, 1) == 31 * 8192 + 8
    assert bench.bwd_g_bytes_per_token(8, 8192, 1, fused=False) == 27 * 8192 + 8
    assert bench.bwd_g_bytes_per_token(8, 8192, 1, fused=True) == 23 * 8192 + 8


@pytest.mark.parametrize("fused,n_gather,entry,want", [
    (True, 1, "shard", 3),   # forward; backward + parameter reduce
    (True, 8, "shard", 3),
    (False, 1, "shard", 5),  # reduce-scatter, shard norm, all-gather; backward + reduce
    (False, 0, "shard", 4),
    (True, 1, "g", 3),       # the backward through g is one kernel + its reduce
    (False, 1, "g", 6),      # ... or a separate reduce-scatter first
])
def test_launches_per_step(fused, n_gather, entry, want):
    assert bench.launches_per_step(fused, n_gather, entry) == want


def test_bucketed_step_covers_the_batch(lib):
    w = wl.WORKLOADS["ragged"].with_(h=64)
    buckets = bk.bucket_by_tokens(w.seqlens, max_cv=0.15)
    step = bench.BucketedStep(w, torch.device("cpu"), buckets)
    assert [st.w.s for st in step.steps] == [b.tokens for b in buckets]
    assert sum(st.w.s for st in step.steps) == w.s
    for st, b in zip(step.steps, buckets):
        assert st.w.seqlens == tuple(b.lengths)
        assert st.cu is not None and st.cu.tolist() == b.cu_seqlens.tolist()
    # what a caller copies in and out per step: every bucket's tensors
    one = step.steps[0]
    assert len(step.inputs()) == len(buckets) * len(one.inputs())
    assert len(step.outputs()) == len(buckets) * len(one.outputs())
    assert sum(x.numel() for x in step.inputs()) == \
        (w.t * w.s * w.h) + 2 * (w.s * w.h)   # partials, residual, dY


@pytest.mark.parametrize("mask,entry,fwd,bwd", [
    ("stored", "shard", 23 * 8192 + 8, 9 * 8192 + 8),
    ("bits", "shard", 22 * 8192 + 1024 + 8, 8 * 8192 + 1024 + 8),   # h / 8 bytes of mask
    ("regen", "shard", 22 * 8192 + 8, 8 * 8192 + 8),                # no mask at all
    ("stored", "g", 23 * 8192 + 8, 23 * 8192 + 8),   # t = 8 partial gradients read
    ("bits", "g", 22 * 8192 + 1024 + 8, 22 * 8192 + 1024 + 8),
])
def test_step_bytes_of_each_mask_mode(mask, entry, fwd, bwd):
    w = wl.WORKLOADS["70b"]
    assert bench.step_bytes_per_token(w, 1, "fused", mask, entry) == (fwd, bwd)


def test_recorded_traffic_belongs_to_the_default_line_only():
    """The profiled DRAM traffic is that of the default line's forward kernel:
    a line whose forward is another kernel (another mask format, workload,
    norm or number of gathered copies) reports none."""
    base = dict(workload="70b", s=0, h=0, p=None, norm=None, n_gather=1, mask="stored")
    ns = lambda **kw: type("A", (), {**base, **kw})
    assert bench.profiled_workload(ns())
    for change in (dict(mask="bits"), dict(mask="regen"), dict(workload="ragged"),
                   dict(norm="rmsnorm"), dict(n_gather=8), dict(s=2048), dict(p=0.0)):
        assert not bench.profiled_workload(ns(**change)), change
