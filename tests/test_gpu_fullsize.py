"""Full-size parity: every element of the full-size workloads against the oracle.

The 70B-shape forward (LayerNorm, and the RMSNorm workload of the backward
configuration) and the packed workload (42,823 tokens, h = 5120) run in the
launch configuration the benchmark times (one gathered copy); Z and the
dropout mask are compared bit for bit on every element, mean / rstd on every
token, and the gathered O on every element at the bf16 bar.  The backward of
the same workloads is compared on every dResidual and dYpre element, and its
parameter gradients summed over every token.  "第 7 课：序列并行 SP" §3: the
token-wise operators give the same result whichever rank holds a token, so
the sharded outputs must equal the oracle's per-token results everywhere;
answer to Q1: the masks agree element for element.

The oracle runs over chunks of tokens in a thread pool on the host cores
(see ``_cases.full_fwd_check``); each test prints its counts, including how
many elements passed through the magnitude floor alone.
"""
import time

import pytest
import torch

from sp_boundary_norm_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

C = pytest.importorskip("_cases")


@pytest.fixture(scope="module", autouse=True)
def _built(lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield


@pytest.mark.parametrize("name", ["70b", "bwd70b_rms", "ragged"])
def test_forward_full_size_every_element(name):
    w = wl.WORKLOADS[name]
    inp = wl.forward_inputs(w, C.DEV)
    out = C.run_fwd(w, inp, n_gather=1)
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    t0 = time.perf_counter()
    tot = C.full_fwd_check(w, inp, out)
    print(f"\nfull-size forward {name}: {tot} ({time.perf_counter() - t0:.1f} s, "
          f"{C.host_threads()} threads)")


@pytest.mark.parametrize("name", ["bwd70b", "bwd70b_rms", "ragged", "trace4k"])
def test_backward_full_size_every_element(name):
    w = wl.WORKLOADS[name]
    inp = wl.forward_inputs(w, C.DEV)
    fwd = C.run_fwd(w, inp, n_gather=0)
    dy = wl.backward_inputs(w, C.DEV)["dy"]
    out = C.run_bwd(w, fwd, inp["gamma"], dy, None, n_gather=1)
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    t0 = time.perf_counter()
    tot = C.full_bwd_check(w, fwd, inp["gamma"], dy, None, out)
    print(f"\nfull-size backward {name}: {tot} ({time.perf_counter() - t0:.1f} s, "
          f"{C.host_threads()} threads)")


@pytest.mark.parametrize("name", ["bwd70b", "ragged"])
def test_mask_free_backward_full_size_every_element(name):
    """The mask-free backward at full size, every element against the oracle
    run with the forward's stored mask: the keep decisions it draws again
    must be the forward's (answer to Q1: one seed, the same mask everywhere).
    At h = 8192 it runs its own launch shape (256 threads x 4 chunks, terms in
    tensor memory), so its float32 row sums may round differently from the
    stored-mask backward's; the bar is the oracle's, not bit equality."""
    w = wl.WORKLOADS[name]
    inp = wl.forward_inputs(w, C.DEV)
    fwd = C.run_fwd(w, inp, n_gather=0)
    dy = wl.backward_inputs(w, C.DEV)["dy"]
    got = C.alloc_bwd(w, 1)
    cu = torch.from_numpy(wl.cu_seqlens(w.seqlens)).to(C.DEV) if w.ragged else None
    C.sp.sp_norm_bwd_philox(dy, fwd["z"], fwd["mean"], fwd["rstd"], inp["gamma"], None, s=w.s,
                            p=w.p, seed=w.seed, offset=w.offset, norm=w.norm, cu_seqlens=cu,
                            dresidual=got["dres"], dgathered=got["dgat"], dgamma=got["dgamma"],
                            dbeta=got["dbeta"], dbias=got["dbias"], workspace=got["ws"])
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    t0 = time.perf_counter()
    tot = C.full_bwd_check(w, fwd, inp["gamma"], dy, None, got)
    print(f"\nfull-size mask-free backward {name}: {tot} ({time.perf_counter() - t0:.1f} s)")


@pytest.mark.parametrize("name", ["bwd70b", "ragged"])
def test_rs_norm_bwd_full_size_every_element(name):
    """The backward entered through g at full size (the 70B shape, and the
    packed workload with its uneven shards): dY is the float32
    rank-ascending sum of the t ranks' partial gradients of the gathered
    input (the reduce-scatter that is the gradient of g, "第 7 课" §3.B),
    fused into the norm backward; every element against the oracle."""
    w = wl.WORKLOADS[name]
    inp = wl.forward_inputs(w, C.DEV)
    fwd = C.run_fwd(w, inp, n_gather=0)
    gen = wl.make_generator(97, C.DEV)
    parts = [(torch.randn((w.b, w.s, w.h), generator=gen, device=C.DEV) * 0.35).to(torch.bfloat16)
             for _ in range(w.t)]
    out = C.alloc_bwd(w, 1)
    cu = torch.from_numpy(wl.cu_seqlens(w.seqlens)).to(C.DEV) if w.ragged else None
    C.sp.sp_rs_norm_bwd(parts, fwd["z"], fwd["mask"], fwd["mean"], fwd["rstd"], inp["gamma"],
                        None, p=w.p, norm=w.norm, cu_seqlens=cu, dresidual=out["dres"],
                        dgathered=out["dgat"], dgamma=out["dgamma"], dbeta=out["dbeta"],
                        dbias=out["dbias"], workspace=out["ws"])
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    t0 = time.perf_counter()
    tot = C.full_bwd_check(w, fwd, inp["gamma"], None, None, out, dy_partials=parts)
    print(f"\nfull-size backward through g, {name}: {tot} ({time.perf_counter() - t0:.1f} s)")


def test_70b_one_gathered_copy_per_rank_every_element():
    """n_gather = t at the 70B shape (the --n-gather 8 bench line): every
    element of every rank's gathered O and gathered dYpre against the oracle."""
    w = wl.WORKLOADS["70b"]
    inp = wl.forward_inputs(w, C.DEV)
    fwd = C.run_fwd(w, inp, n_gather=w.t)
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    t0 = time.perf_counter()
    f = C.full_fwd_check(w, inp, fwd)
    del fwd["gathered"]
    dy = wl.backward_inputs(w, C.DEV)["dy"]
    out = C.run_bwd(w, fwd, inp["gamma"], dy, None, n_gather=w.t)
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    g = C.full_bwd_check(w, fwd, inp["gamma"], dy, None, out)
    print(f"\nfull-size n_gather={w.t}: forward {f}, backward {g} "
          f"({time.perf_counter() - t0:.1f} s)")


@pytest.mark.parametrize("name", ["70b", "ragged"])
def test_unfused_pipeline_full_size_every_element(name):
    """The unfused boundary (reduce-scatter, norm on the shards, all-gather:
    the ablation of the fusion) at full size, every element against the
    oracle: the bf16 shards of the reduce-scatter, Z, mask, statistics, O and
    the gathered copy."""
    w = wl.WORKLOADS[name]
    inp = wl.forward_inputs(w, C.DEV)
    y, o, out = C.run_unfused(w, inp)
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    t0 = time.perf_counter()
    tot = C.full_unfused_fwd_check(w, inp, y, o, out)
    print(f"\nfull-size unfused forward {name}: {tot} ({time.perf_counter() - t0:.1f} s)")


@pytest.mark.parametrize("name", ["70b", "ragged"])
def test_bit_mask_pair_full_size_equals_byte_mask_pair(name):
    """At full size the bit-mask forward and backward give the byte mask packed
    and every other output bit for bit as the byte-mask pair, which the
    tests above check against the oracle on every element."""
    w = wl.WORKLOADS[name]
    cu = torch.from_numpy(wl.cu_seqlens(w.seqlens)).to(C.DEV) if w.ragged else None
    inp = wl.forward_inputs(w, C.DEV)
    dy = wl.backward_inputs(w, C.DEV)["dy"]
    fwd_b = C.run_fwd(w, inp, n_gather=1)
    bwd_b = C.run_bwd(w, fwd_b, inp["gamma"], dy, None, n_gather=1)
    fwd_k, bwd_k = C.run_bitmask_pair(w, inp, dy, None, 1, 1, cu_seqlens=cu)
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    C.assert_bitmask_pair_matches(w, fwd_b, bwd_b, fwd_k, bwd_k)


def test_rs_norm_bwd_bit_mask_full_size_equals_byte_mask():
    """The backward entered through g at the 70B shape, reading the bit-packed
    mask, equals the byte-mask call (checked against the oracle above) bit for
    bit."""
    w = wl.WORKLOADS["bwd70b"]
    inp = wl.forward_inputs(w, C.DEV)
    fwd = C.run_fwd(w, inp, n_gather=0)
    gen = wl.make_generator(97, C.DEV)
    parts = [(torch.randn((w.b, w.s, w.h), generator=gen, device=C.DEV) * 0.35).to(torch.bfloat16)
             for _ in range(w.t)]
    ref = C.alloc_bwd(w, 1)
    C.sp.sp_rs_norm_bwd(parts, fwd["z"], fwd["mask"], fwd["mean"], fwd["rstd"], inp["gamma"],
                        None, p=w.p, norm=w.norm, dresidual=ref["dres"], dgathered=ref["dgat"],
                        dgamma=ref["dgamma"], dbeta=ref["dbeta"], dbias=ref["dbias"],
                        workspace=ref["ws"])
    got = C.run_rs_bwd_bitmask(w, fwd, inp, parts, None, C.oracle_mask_bits(fwd["mask"]), 1)
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    C.assert_bwd_outputs_equal(w, ref, got)


def test_tensors_beyond_2_31_elements():
    """Tensors of more than 2^31 elements (t = 2, s = 266,240 tokens of
    h = 8192: 2.18 G elements per partial, about 38 GB in all): every element
    of rows on both sides of element 2^31 (token 262,144), of the shard
    boundary and of the first and last rows, forward and backward, against
    the oracle -- the kernels' 64-bit index arithmetic; and the bit-mask pair
    on the same inputs, bit for bit the byte-mask pair on every element."""
    import numpy as np
    w = wl.Workload("big", t=2, b=1, s=266240, h=8192, draw_seed=77)
    assert w.s * w.h > 2 ** 31
    inp = wl.forward_inputs(w, C.DEV)
    fwd = C.run_fwd(w, inp, n_gather=1)
    dy = wl.backward_inputs(w, C.DEV)["dy"]
    bwd = C.run_bwd(w, fwd, inp["gamma"], dy, None, n_gather=1)
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    edge = 2 ** 31 // w.h
    tokens = np.array(sorted({0, 1, edge - 2, edge - 1, edge, edge + 1, w.s // 2 - 1, w.s // 2,
                              w.s - 2, w.s - 1} | set(range(edge - 8, edge + 8, 3))),
                      dtype=np.int64)
    C.check_fwd_rows(w, inp, fwd, tokens)
    C.check_bwd_rows(w, fwd, inp["gamma"], dy, None, bwd, tokens)
    for name in ("dgamma", "dbeta", "dbias"):
        assert torch.isfinite(bwd[name]).all(), name
    # the bit-packed mask at this size: every output of the pair bit for bit
    fwd_k, bwd_k = C.run_bitmask_pair(w, inp, dy, None, 1, 1)
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    C.assert_bitmask_pair_matches(w, fwd, bwd, fwd_k, bwd_k)
