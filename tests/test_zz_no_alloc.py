"""The allocate-nothing backward (sp_norm_bwd_noalloc) against sp_norm_bwd.

sp_norm_bwd_noalloc serves callers that have no way to obtain device scratch
memory themselves (for example a plugin whose host framework reserves all
device memory and gives it no workspace): the library keeps the
parameter-gradient partials in a fixed array of its own device memory.  These
tests call it through the C ABI, twice in a row with different inputs, and
check every output against the ordinary entry point, which takes a caller
workspace.  Both run the same kernels with the same grid and summation order,
so every output, the float32 parameter gradients included, must agree bit
for bit.

This file is collected last on purpose: a failure here leaves every other
test already run.
"""
import numpy as np
import pytest
import torch

from oracle import compare
from sp_boundary_norm_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

C = pytest.importorskip("_cases")


@pytest.fixture(scope="module", autouse=True)
def _built(lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield


def _noalloc(w, fwd, gamma, dy, skip, n_gather=1):
    out = C.alloc_bwd(w, n_gather)
    C.sp.sp_norm_bwd_noalloc(dy, fwd["z"], fwd["mask"], fwd["mean"], fwd["rstd"], gamma, skip,
                             s=w.s, p=w.p, norm=w.norm, dresidual=out["dres"],
                             dgathered=out["dgat"], dgamma=out["dgamma"],
                             dbeta=out["dbeta"] if w.norm == "layernorm" else None,
                             dbias=out["dbias"])
    return out


def _same(w, a, b):
    for x, y in zip(a["dres"] + a["dgat"], b["dres"] + b["dgat"]):
        assert np.array_equal(compare.bf16_bits(x), compare.bf16_bits(y))
    names = ["dgamma", "dbias"] + (["dbeta"] if w.norm == "layernorm" else [])
    for name in names:
        # the same kernel, grid and summation order run in both, so the
        # parameter gradients must be identical bit for bit: a partial or
        # stale overwrite of the shared scratch would show here
        assert torch.equal(a[name].view(torch.int32), b[name].view(torch.int32)), name


@pytest.mark.parametrize("norm,with_skip,n_gather", [("layernorm", False, 1),
                                                    ("rmsnorm", True, 1),
                                                    ("layernorm", False, 3)])
def test_noalloc_backward_matches_workspace_backward_twice(norm, with_skip, n_gather):
    w = wl.Workload("na", t=4, b=1, s=2048, h=8192, norm=norm,
                    eps=1e-5 if norm == "layernorm" else 1e-6, draw_seed=51)
    inp = wl.forward_inputs(w, C.DEV)
    fwd = C.run_fwd(w, inp, n_gather=0)
    for call in range(2):   # two calls in a row, different upstream gradients
        b = wl.backward_inputs(w, C.DEV, seed=60 + call, with_skip=with_skip)
        ref = C.run_bwd(w, fwd, inp["gamma"], b["dy"], b["dz_skip"], n_gather=n_gather)
        got = _noalloc(w, fwd, inp["gamma"], b["dy"], b["dz_skip"], n_gather)
        torch.cuda.synchronize()
        C.sp.check_device_status(C.DEV)
        _same(w, got, ref)


def test_noalloc_backward_at_70b_shape():
    """h = 8192: the stored-mask backward runs one block per SM, 152 x 3 x h
    float32 partials (14.9 MB), inside the fixed scratch."""
    w = wl.WORKLOADS["bwd70b"]
    inp = wl.forward_inputs(w, C.DEV)
    fwd = C.run_fwd(w, inp, n_gather=0)
    dy = wl.backward_inputs(w, C.DEV)["dy"]
    ref = C.run_bwd(w, fwd, inp["gamma"], dy, None, n_gather=1)
    got = _noalloc(w, fwd, inp["gamma"], dy, None)
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    _same(w, got, ref)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    w = wl.Workload("big", t=2, b=1, s=4096, h=16384, draw_seed=52)
    assert C.sp.sp_norm_bwd_workspace_bytes(w.b, w.s, w.h, w.t) > C.sp.NOALLOC_WORKSPACE_BYTES
    inp = wl.forward_inputs(w, C.DEV)
    fwd = C.run_fwd(w, inp, n_gather=0)
    dy = wl.backward_inputs(w, C.DEV)["dy"]
    with pytest.raises(C.sp.SpError) as e:
        _noalloc(w, fwd, inp["gamma"], dy, None)
    assert e.value.name == "SP_ERR_UNSUPPORTED"
