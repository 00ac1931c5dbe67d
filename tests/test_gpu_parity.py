"""GPU parity: the CUDA boundary (through the C ABI) against the CPU oracle.

Bit-exact: shard indexing, gathered layout, Z (pinned float32 order), the
dropout mask.  Tolerances (``oracle.compare``): bf16 outputs within 1 ulp (or
float32-accuracy floor on cancellation), float32 stats 1e-5 relative,
parameter-gradient sums 1e-5 of their terms' root-sum-square.
"""
import numpy as np
import pytest
import torch

from oracle import boundary as ob
from oracle import compare
from sp_boundary_norm_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

C = pytest.importorskip("_cases")


@pytest.fixture(scope="module", autouse=True)
def _built(lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield


_full_fwd_compare = C.fwd_compare_all


@pytest.mark.parametrize("name", ["tiny", "trace4k"])
def test_forward_full_compare(name):
    w = wl.WORKLOADS[name]
    inp = wl.forward_inputs(w, C.DEV)
    out = C.run_fwd(w, inp)
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    _full_fwd_compare(w, inp, out)


@pytest.mark.parametrize("variant", [dict(), dict(b=2, s=36, t=3), dict(norm="rmsnorm", eps=1e-6)])
def test_forward_equals_unsharded_path_sliced_by_token(variant):
    """Sequence parallelism leaves every token-wise result unchanged: the GPU
    boundary equals the TP-only path (all-reduce of the partials, then bias,
    dropout, residual and the norm on every token) sliced by shard; Z and the
    mask bit for bit, the statistics and O within the stated tolerances."""
    w = wl.Workload("us", t=4, b=1, s=64, h=1024, draw_seed=131).with_(**variant)
    inp = wl.forward_inputs(w, C.DEV)
    out = C.run_fwd(w, inp)
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    offs = [(k * w.s) // w.t for k in range(w.t + 1)]
    residual_full = np.concatenate([C.f32(r) for r in inp["residual"]], axis=1)
    ref = ob.unsharded_fwd([C.f32(x) for x in inp["partials"]], residual_full,
                           C.f32(inp["bias"]), C.f32(inp["gamma"]), C.f32(inp["beta"]),
                           eps=w.eps, p=w.p, seed=w.seed, offset=w.offset, norm=w.norm)
    for k in range(w.t):
        sl = slice(offs[k], offs[k + 1])
        assert np.array_equal(compare.bf16_bits(out["z"][k]), compare.bf16_bits(ref["z"][:, sl])), k
        assert np.array_equal(out["mask"][k].cpu().numpy(), ref["mask"][:, sl]), k
        assert not compare.f32_rel_mismatch(out["rstd"][k].cpu().numpy(), ref["rstd"][:, sl]).any()
        if w.norm == "layernorm":
            assert not compare.f32_rel_mismatch(out["mean"][k].cpu().numpy(),
                                                ref["mean"][:, sl]).any()
    C.assert_bf16(compare.bf16_bits(out["gathered"][0]), ref["out_exact"], ref["out_magnitude"],
                  "gathered[0]")


@pytest.fixture
def fwd_split():
    """Split every forward row over a thread-block cluster of `split` CTAs
    (forcing the threads per CTA if given) for one test; the automatic choice
    is restored afterwards."""
    def force(split, threads=0):
        C.sp.sp_debug_tune(0, 0, 0, threads, split)
    yield force
    C.sp.sp_debug_tune(0, 0, 0, 0, 0)


@pytest.mark.parametrize("split", [1, 2])
def test_layernorm_rows_with_large_mean(fwd_split, split):
    """The forward takes the LayerNorm variance as E[Z^2] - mean^2 only where
    mean^2 <= var / 4 and recomputes it from (Z - mean)^2 elsewhere.  Residual
    rows shifted by 0 to 300 standard deviations (either sign, several near the
    switch at 0.5) put tokens on both sides; all must meet the tolerances.
    With split = 2 each row is split over a CTA pair, so the recomputation
    takes a second exchange of row sums between the two CTAs."""
    if split == 2:
        fwd_split(2, 128)
    w = wl.Workload("lm", t=4, b=1, s=288, h=1024, draw_seed=97)
    inp = wl.forward_inputs(w, C.DEV)
    shifts = [0.0, 0.25, 0.45, 0.49, 0.5, 0.51, 0.55, 0.7, 1.0, 3.0, 30.0, 300.0, -0.5, -40.0]
    offs = [(k * w.s) // w.t for k in range(w.t + 1)]
    for k, r in enumerate(inp["residual"]):
        g = torch.arange(offs[k], offs[k + 1], device=C.DEV)
        c = torch.tensor(shifts, device=C.DEV)[g % len(shifts)]
        inp["residual"][k] = (r.float() + c[None, :, None]).to(torch.bfloat16)
    out = C.run_fwd(w, inp)
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    ref = _full_fwd_compare(w, inp, out)
    ratio = np.concatenate([m * m / (1.0 / (r * r) - w.eps) for m, r in
                            zip(ref["mean"], ref["rstd"])], axis=1)
    assert (ratio < 0.2).any() and (ratio > 0.3).any() and (ratio > 1e3).any()
    assert C.sp.sp_debug_last_shape(0)["cluster"] == split


@pytest.mark.parametrize("variant,threads", [
    (dict(), 128),
    (dict(norm="rmsnorm", eps=1e-6), 128),
    (dict(t=3, s=48), 128),
    (dict(b=3, s=40, t=4), 128),
    (dict(h=16, s=16), 128),
    (dict(h=528, s=32), 128),
    (dict(p=0.0), 128),
    (dict(n_gather=2), 128),
    (dict(seed=2**40 + 17, offset=2**33 + 5), 128),
    (dict(h=4096, s=64, t=8), 0),
    (dict(h=8192, s=64, t=8), 0),
    (dict(h=8192, s=16, t=8), 256),
    (dict(h=16384, s=8), 0),
])
def test_forward_row_split_over_a_cta_pair(fwd_split, variant, threads):
    """The forward with every token row split over a thread-block cluster of
    two CTAs (h / 2 channels each, the row sums exchanged through distributed
    shared memory): Z and the mask bit for bit, the statistics and O within
    the tolerances, against the oracle."""
    fwd_split(2, threads)
    w = wl.Workload("cp", t=2, b=1, s=64, h=512, draw_seed=141).with_(**variant)
    inp = wl.forward_inputs(w, C.DEV)
    out = C.run_fwd(w, inp)
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    shape = C.sp.sp_debug_last_shape(0)
    assert shape["cluster"] == 2 and shape["grid"] % 2 == 0, shape
    _full_fwd_compare(w, inp, out)


def test_forward_row_split_ragged_and_70b_every_element(fwd_split):
    """The CTA-pair forward on packed uneven shards and on the 70B shape,
    every element against the oracle (the 70B check through the chunked,
    thread-pooled oracle), and the drop rate."""
    fwd_split(2, 128)
    lengths = (33, 64, 7, 1, 90, 12)
    w = wl.Workload("rp", t=5, b=1, s=sum(lengths), h=512, seqlens=lengths, draw_seed=142)
    inp = wl.forward_inputs(w, C.DEV)
    out = C.run_fwd(w, inp)
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    assert C.sp.sp_debug_last_shape(0)["cluster"] == 2
    _full_fwd_compare(w, inp, out)
    del inp, out
    fwd_split(2)
    w = wl.WORKLOADS["70b"]
    inp = wl.forward_inputs(w, C.DEV)
    out = C.run_fwd(w, inp)
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    assert C.sp.sp_debug_last_shape(0)["cluster"] == 2
    C.full_fwd_check(w, inp, out)
    kept = sum(int(m.sum()) for m in out["mask"])
    n = w.tokens * w.h
    assert abs((1 - kept / n) - w.p) < 5 * np.sqrt(w.p * (1 - w.p) / n)


@pytest.mark.parametrize("variant", [
    dict(norm="rmsnorm", eps=1e-6),
    dict(p=0.0),
    dict(t=1),
    dict(t=1, p=0.0),
    dict(t=3, s=48),
    dict(t=16, s=64),
    dict(b=3, s=40, t=4),
    dict(h=8, s=16),
    dict(h=24, s=16),
    dict(h=520, s=32),
    dict(h=2056, s=16),
    dict(h=5120, s=32),
    dict(h=16384, s=8),
    dict(n_gather=2),
    dict(n_gather=0),
    dict(seed=2**40 + 17, offset=2**33 + 5),
    dict(p=0.9),
])
def test_forward_variants_full_compare(variant):
    base = wl.Workload("v", t=2, b=1, s=64, h=512, draw_seed=21)
    w = base.with_(**variant)
    inp = wl.forward_inputs(w, C.DEV)
    out = C.run_fwd(w, inp)
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    _full_fwd_compare(w, inp, out)


def test_forward_gathered_copies_identical_and_layout():
    w = wl.Workload("g", t=4, b=2, s=32, h=256, n_gather=4, draw_seed=22)
    inp = wl.forward_inputs(w, C.DEV)
    out = C.run_fwd(w, inp)
    g0 = out["gathered"][0]
    for g in out["gathered"][1:]:
        assert torch.equal(g.view(torch.int16), g0.view(torch.int16))


@pytest.mark.parametrize("lengths,t,extra", [((5, 17, 3, 40), 8, {}), ((3,), 8, {}),
                                             ((100, 1, 1), 3, {}),
                                             ((33, 64, 7, 1, 90, 12), 5, {}),
                                             ((33, 64, 7, 1, 90, 12), 5,
                                              dict(norm="rmsnorm", eps=1e-6)),
                                             ((5, 17, 3, 40), 8, dict(n_gather=3)),
                                             ((50, 13, 9), 8, dict(h=5120))])
def test_forward_ragged_packed_full_compare(lengths, t, extra):
    w = wl.Workload("r", t=t, b=1, s=sum(lengths), h=512, seqlens=tuple(lengths),
                    draw_seed=23).with_(**extra)
    inp = wl.forward_inputs(w, C.DEV)
    out = C.run_fwd(w, inp)
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    _full_fwd_compare(w, inp, out)


def test_forward_ragged_workload_sampled():
    w = wl.WORKLOADS["ragged"]
    inp = wl.forward_inputs(w, C.DEV)
    out = C.run_fwd(w, inp)
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    C.check_fwd_rows(w, inp, out, C.sample_tokens(w, 160))


@pytest.mark.parametrize("name", ["70b", "bwd70b_rms"])
def test_forward_70b_sampled_and_properties(name):
    """The 70B-shape forward at full size in the bench's launch configuration
    (LayerNorm, and the RMSNorm workload of the backward config): sampled
    tokens against the oracle, whole-tensor properties."""
    w = wl.WORKLOADS[name]
    inp = wl.forward_inputs(w, C.DEV)
    out = C.run_fwd(w, inp)
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    C.check_fwd_rows(w, inp, out, C.sample_tokens(w, 96))
    # properties over the whole output: drop rate, finiteness, gathered == shards
    kept = sum(int(m.sum()) for m in out["mask"])
    n = w.tokens * w.h
    assert abs((1 - kept / n) - w.p) < 5 * np.sqrt(w.p * (1 - w.p) / n)
    g = out["gathered"][0]
    assert torch.isfinite(g.float()).all()
    offs = [(k * w.s) // w.t for k in range(w.t + 1)]
    for k in range(w.t):
        blk = g[:, offs[k]:offs[k + 1], :].float()
        assert torch.isfinite(out["z"][k].float()).all()
        # finite statistics on every token
        assert torch.isfinite(out["rstd"][k]).all()
        if w.norm == "layernorm":
            assert torch.isfinite(out["mean"][k]).all()
        assert blk.shape[1] == w.shard_sizes()[k]


def test_forward_empty_and_tiny_sequences():
    w = wl.Workload("e", t=4, b=1, s=0, h=64)
    inp = wl.forward_inputs(w, C.DEV)
    out = C.run_fwd(w, inp)
    torch.cuda.synchronize()
    assert all(z.numel() == 0 for z in out["z"])


def test_forward_mask_independent_of_t_on_gpu():
    masks = []
    for t in (1, 2, 8):
        w = wl.Workload("m", t=t, b=1, s=64, h=256, draw_seed=24)
        inp = wl.forward_inputs(w, C.DEV)
        out = C.run_fwd(w, inp)
        masks.append(torch.cat(out["mask"], dim=1))
    assert torch.equal(masks[0], masks[1]) and torch.equal(masks[0], masks[2])


def test_forward_deterministic_and_writes_only_its_outputs():
    w = wl.Workload("d", t=4, b=1, s=128, h=1024, n_gather=2, draw_seed=25)
    inp = wl.forward_inputs(w, C.DEV)
    # outputs poisoned first: every element must be overwritten
    out1 = C.run_fwd(w, inp, out=C.alloc_fwd(w, 2, fill=float("nan")))
    out2 = C.run_fwd(w, inp, out=C.alloc_fwd(w, 2, fill=-7.0))
    torch.cuda.synchronize()
    for key in ("z", "gathered"):
        for a, b in zip(out1[key], out2[key]):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    for key in ("mask", "mean", "rstd"):
        for a, b in zip(out1[key], out2[key]):
            assert torch.equal(a, b)


def test_guard_bands_untouched():
    """Outputs carved from larger buffers: bytes around them keep their pattern."""
    w = wl.Workload("gb", t=2, b=1, s=96, h=264, n_gather=1, draw_seed=26)
    inp = wl.forward_inputs(w, C.DEV)
    pad = 4096
    sizes = w.shard_sizes()

    def carve(shape, dtype):
        n = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
        raw = torch.full((n + 2 * pad,), 0x5A, dtype=torch.uint8, device=C.DEV)
        return raw, raw[pad:pad + n].view(dtype).view(shape)

    bufs, out = [], {"z": [], "mask": [], "mean": [], "rstd": [], "gathered": []}
    for n in sizes:
        for key, shape, dt in (("z", (1, n, w.h), torch.bfloat16), ("mask", (1, n, w.h), torch.uint8),
                               ("mean", (1, n), torch.float32), ("rstd", (1, n), torch.float32)):
            raw, v = carve(shape, dt)
            bufs.append(raw)
            out[key].append(v)
    raw, v = carve((1, w.s, w.h), torch.bfloat16)
    bufs.append(raw)
    out["gathered"].append(v)
    C.run_fwd(w, inp, out=out)
    torch.cuda.synchronize()
    for raw in bufs:
        assert bool((raw[:pad] == 0x5A).all()) and bool((raw[-pad:] == 0x5A).all())


def test_invalid_cu_seqlens_flagged_on_device():
    w = wl.Workload("bad", t=2, b=1, s=20, h=64, seqlens=(10, 10), draw_seed=27)
    inp = wl.forward_inputs(w, C.DEV)
    bad = torch.tensor([0, 10, 19], dtype=torch.int32, device=C.DEV)   # ends at 19 != 20
    C.run_fwd(w, inp, cu_seqlens=bad)
    torch.cuda.synchronize()
    with pytest.raises(C.sp.SpError) as e:
        C.sp.check_device_status(C.DEV)
    assert e.value.name == "SP_ERR_DEVICE_CHECK"
    C.run_fwd(w, inp)                                                    # a good call after
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)


def test_injected_failure_launches_nothing():
    w = wl.WORKLOADS["tiny"]
    inp = wl.forward_inputs(w, C.DEV)
    out = C.alloc_fwd(w, 1, fill=3.0)
    C.sp.sp_debug_inject(4)
    with pytest.raises(C.sp.SpError) as e:
        C.run_fwd(w, inp, out=out)
    assert e.value.name == "SP_ERR_CUDA"
    torch.cuda.synchronize()
    assert bool((out["gathered"][0].float() == 3.0).all())
    C.run_fwd(w, inp, out=out)                                           # hook disarmed


def test_forward_bounded_wait_reports_timeout():
    """The SP_ERR_TIMEOUT test hook makes block 0's copy producer withhold its
    first chunk: that block's bounded waits give up after about a second, the
    status word reads SP_ERR_TIMEOUT, nothing hangs or faults, and the next
    call is exact again."""
    import time
    w = wl.Workload("to", t=2, b=1, s=64, h=512, draw_seed=121)
    inp = wl.forward_inputs(w, C.DEV)
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    C.sp.sp_debug_inject(5)                                            # SP_ERR_TIMEOUT
    t0 = time.perf_counter()
    C.run_fwd(w, inp)
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 10.0
    with pytest.raises(C.sp.SpError) as e:
        C.sp.check_device_status(C.DEV)
    assert e.value.name == "SP_ERR_TIMEOUT"
    out = C.run_fwd(w, inp)                                            # hook disarmed
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    _full_fwd_compare(w, inp, out)


# ------------------------------------------------------------------ backward

def _bwd_setup(w, with_skip=False, n_gather=1):
    inp = wl.forward_inputs(w, C.DEV)
    fwd = C.run_fwd(w, inp, n_gather=0)
    b = wl.backward_inputs(w, C.DEV, with_skip=with_skip)
    out = C.run_bwd(w, fwd, inp["gamma"], b["dy"], b["dz_skip"], n_gather=n_gather)
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    return inp, fwd, b, out


@pytest.mark.parametrize("variant", [
    dict(),
    dict(norm="rmsnorm", eps=1e-6),
    dict(p=0.0),
    dict(t=1),
    dict(t=3, s=48),
    dict(b=2, s=40, t=4),
    dict(h=8, s=16),
    dict(h=520, s=32),
    dict(h=5120, s=24),
    dict(h=16384, s=8),
    dict(n_gather=3),
    dict(n_gather=0),
])
@pytest.mark.parametrize("with_skip", [False, True])
def test_backward_full_compare(variant, with_skip):
    base = wl.Workload("b", t=2, b=1, s=64, h=512, draw_seed=31)
    w = base.with_(**variant)
    inp, fwd, b, out = _bwd_setup(w, with_skip, n_gather=w.n_gather)
    toks = np.arange(w.tokens, dtype=np.int64)
    C.check_bwd_rows(w, fwd, inp["gamma"], b["dy"], b["dz_skip"], out, toks)
    C.check_param_grads(w, fwd, inp["gamma"], b["dy"], b["dz_skip"], out)


@pytest.mark.parametrize("variant", [
    dict(),
    dict(norm="rmsnorm", eps=1e-6),
    dict(skip=True),
    dict(n_gather=2),
    dict(h=5120, t=8),
])
def test_backward_ragged_packed(variant):
    """Packed uneven shards through the backward, every token compared, with
    RMSNorm, the skip-path gradient, two gathered copies and the h = 5120
    tensor-memory shape."""
    v = dict(variant)
    skip = v.pop("skip", False)
    lengths = (5, 17, 3, 40, 1, 9)
    w = wl.Workload("rb", t=4, b=1, s=sum(lengths), h=256, seqlens=lengths,
                    draw_seed=32).with_(**v)
    inp, fwd, b, out = _bwd_setup(w, skip, n_gather=w.n_gather)
    C.check_bwd_rows(w, fwd, inp["gamma"], b["dy"], b["dz_skip"], out, np.arange(w.tokens))
    C.check_param_grads(w, fwd, inp["gamma"], b["dy"], b["dz_skip"], out)


@pytest.mark.parametrize("name", ["bwd70b", "bwd70b_rms"])
def test_backward_70b_sampled_and_param_grads(name):
    w = wl.WORKLOADS[name]
    inp, fwd, b, out = _bwd_setup(w)
    C.check_bwd_rows(w, fwd, inp["gamma"], b["dy"], None, out, C.sample_tokens(w, 64))
    C.check_param_grads(w, fwd, inp["gamma"], b["dy"], None, out)


def test_70b_one_gathered_copy_per_rank():
    """The 70B shape with n_gather = t (one gathered copy per rank, the
    bench's --n-gather 8 line): forward and backward sampled against the
    oracle through copy 0, and every copy bit-identical to copy 0."""
    w = wl.WORKLOADS["70b"]
    inp = wl.forward_inputs(w, C.DEV)
    fwd = C.run_fwd(w, inp, n_gather=w.t)
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    C.check_fwd_rows(w, inp, fwd, C.sample_tokens(w, 48))
    for g in fwd["gathered"][1:]:
        assert torch.equal(g.view(torch.int16), fwd["gathered"][0].view(torch.int16))
    del fwd["gathered"]
    b = wl.backward_inputs(w, C.DEV)
    out = C.run_bwd(w, fwd, inp["gamma"], b["dy"], None, n_gather=w.t)
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    C.check_bwd_rows(w, fwd, inp["gamma"], b["dy"], None, out, C.sample_tokens(w, 48))
    for g in out["dgat"][1:]:
        assert torch.equal(g.view(torch.int16), out["dgat"][0].view(torch.int16))


@pytest.mark.parametrize("variant,n_gather", [
    (dict(), 2),
    (dict(s=4096), 3),                       # several rows per block: both row buffers reused
    (dict(t=8, s=64, h=8192), 8),            # the 70B row width, one row per block
    (dict(t=8, s=4096, h=8192), 8),
    (dict(t=8, s=512, h=5120), 4),           # the tensor-memory shape
    (dict(t=8, s=1024, h=4096, norm="rmsnorm", eps=1e-6), 2),
    (dict(skip=True, s=1000), 5),
    (dict(seqlens=(300, 17, 683), s=1000, t=3), 3),
    (dict(b=2, s=512, t=4), 2),              # gathered rows of two batch rows
    (dict(t=3, s=999, h=2056), 3),           # a row width that leaves chunks partial
    (dict(s=64, h=16384), 2),                # the widest rows: 4 chunks, ring of 2
    (dict(s=64, h=16384, skip=True), 3),     # ... with the skip gradient: ring of 1
])
def test_backward_bulk_gathered_copies_equal_per_thread_stores(variant, n_gather):
    """With several gathered copies the backward writes each row's dYpre once
    into shared memory and sends it to every copy with bulk copies.  Every
    copy must equal, bit for bit, the copy the per-thread stores write with a
    single gathered copy; dResidual and the parameter gradients are
    unchanged; nothing outside the copies is written."""
    v = dict(variant)
    skip = v.pop("skip", False)
    w = wl.Workload("bk", t=2, b=1, s=256, h=512, draw_seed=37).with_(**v)
    inp = wl.forward_inputs(w, C.DEV)
    fwd = C.run_fwd(w, inp, n_gather=0)
    bi = wl.backward_inputs(w, C.DEV, with_skip=skip)
    one = C.run_bwd(w, fwd, inp["gamma"], bi["dy"], bi["dz_skip"], n_gather=1)
    torch.cuda.synchronize()
    shape_one = C.sp.sp_debug_last_shape(1)
    pad = 4096
    nbytes = w.tokens * w.h * 2
    raws = [torch.full((nbytes + 2 * pad,), 0x5A, dtype=torch.uint8, device=C.DEV)
            for _ in range(n_gather)]
    for raw in raws:
        raw[pad:pad + nbytes] = 0xFF   # NaN bf16 pattern: every element must be written
    out = C.alloc_bwd(w, 0)
    out["dgat"] = [raw[pad:pad + nbytes].view(torch.bfloat16).view(w.b, w.s, w.h) for raw in raws]
    C.run_bwd(w, fwd, inp["gamma"], bi["dy"], bi["dz_skip"], out=out)
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    shape_many = C.sp.sp_debug_last_shape(1)
    stage = ((w.h * 2 + 15) // 16) * 16
    tmem = (shape_many["threads"], shape_many["chunks"]) in ((320, 2), (256, 4), (128, 4))
    if not tmem:   # (tensor-memory shapes pad their shared memory to a fixed size)
        assert shape_many["smem"] >= shape_one["smem"] + 2 * stage or shape_many["stages"] != \
            shape_one["stages"], (shape_one, shape_many)   # the bulk variant ran
    ref = one["dgat"][0].view(torch.int16)
    for g in out["dgat"]:
        assert torch.equal(g.view(torch.int16), ref)
    for raw in raws:
        assert bool((raw[:pad] == 0x5A).all()) and bool((raw[-pad:] == 0x5A).all())
    for a, b in zip(out["dres"], one["dres"]):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    names = ["dgamma", "dbias"] + (["dbeta"] if w.norm == "layernorm" else [])
    for name in names:
        if shape_many["grid"] == shape_one["grid"]:
            assert torch.equal(out[name], one[name]), name
        else:
            assert torch.allclose(out[name], one[name], rtol=1e-5, atol=1e-4), name


def test_backward_ragged_workload_sampled_and_param_grads():
    """The packed workload at full size in the bench's launch configuration
    (h = 5120 runs the tensor-memory shape, 320 threads x 2 chunks):
    sampled rows, including the first and last of every shard, and every
    parameter gradient over all 42,823 tokens."""
    w = wl.WORKLOADS["ragged"]
    inp, fwd, b, out = _bwd_setup(w)
    C.check_bwd_rows(w, fwd, inp["gamma"], b["dy"], None, out, C.sample_tokens(w, 96))
    C.check_param_grads(w, fwd, inp["gamma"], b["dy"], None, out)


def test_backward_deterministic():
    w = wl.Workload("det", t=4, b=1, s=512, h=2048, draw_seed=33)
    inp = wl.forward_inputs(w, C.DEV)
    fwd = C.run_fwd(w, inp, n_gather=0)
    dy = wl.backward_inputs(w, C.DEV)["dy"]
    o1 = C.run_bwd(w, fwd, inp["gamma"], dy)
    o2 = C.run_bwd(w, fwd, inp["gamma"], dy)
    torch.cuda.synchronize()
    for key in ("dgamma", "dbeta", "dbias"):
        assert torch.equal(o1[key], o2[key]), key
    for a, c in zip(o1["dres"], o2["dres"]):
        assert torch.equal(a.view(torch.int16), c.view(torch.int16))


def test_backward_empty_gives_zero_param_grads():
    w = wl.Workload("e", t=2, b=1, s=0, h=64)
    inp = wl.forward_inputs(w, C.DEV)
    fwd = C.run_fwd(w, inp, n_gather=0)
    dy = wl.backward_inputs(w, C.DEV)["dy"]
    out = C.alloc_bwd(w, 1)
    for key in ("dgamma", "dbeta", "dbias"):
        out[key].fill_(5.0)
    C.run_bwd(w, fwd, inp["gamma"], dy, out=out)
    torch.cuda.synchronize()
    for key in ("dgamma", "dbeta", "dbias"):
        assert bool((out[key] == 0).all())


# --------------------------------------------------------- collectives alone

@pytest.mark.parametrize("t,b,s,h,n_gather", [(2, 1, 64, 512, 1), (8, 1, 256, 1024, 8),
                                              (3, 2, 33 * 3, 40, 2), (4, 1, 4096, 4096, 1)])
def test_allgather_and_reduce_scatter_bit_exact(t, b, s, h, n_gather):
    from oracle import collectives as coll
    w = wl.Workload("c", t=t, b=b, s=s, h=h, draw_seed=41)
    inp = wl.forward_inputs(w, C.DEV)
    sizes = w.shard_sizes()
    shards = [torch.empty((b, n, h), dtype=torch.bfloat16, device=C.DEV) for n in sizes]
    C.sp.sp_reduce_scatter_seq(inp["partials"], shards)
    gathered = [torch.empty((b, s, h), dtype=torch.bfloat16, device=C.DEV) for _ in range(n_gather)]
    C.sp.sp_allgather_seq(shards, gathered, s=s)
    torch.cuda.synchronize()
    ref_shards, _ = coll.reduce_scatter_seq([C.f32(x) for x in inp["partials"]])
    from oracle.bf16 import bf16_round
    for k in range(t):
        assert np.array_equal(compare.bf16_bits(shards[k]),
                              compare.bf16_bits(bf16_round(ref_shards[k])))
    full = np.concatenate([bf16_round(x) for x in ref_shards], axis=1)
    for g in gathered:
        assert np.array_equal(compare.bf16_bits(g), compare.bf16_bits(full))


def test_fused_gather_equals_unfused_gather_of_shards():
    """g fused into the norm kernel == g applied afterwards to the shards' O."""
    w = wl.Workload("fu", t=4, b=1, s=256, h=1024, n_gather=1, draw_seed=42)
    inp = wl.forward_inputs(w, C.DEV)
    out = C.run_fwd(w, inp, n_gather=1)
    offs = [(k * w.s) // w.t for k in range(w.t + 1)]
    o_shards = [out["gathered"][0][:, offs[k]:offs[k + 1], :].contiguous() for k in range(w.t)]
    g2 = [torch.empty_like(out["gathered"][0])]
    C.sp.sp_allgather_seq(o_shards, g2, s=w.s)
    torch.cuda.synchronize()
    assert torch.equal(g2[0].view(torch.int16), out["gathered"][0].view(torch.int16))


def test_device_philox_matches_oracle():
    from oracle import philox
    rng = np.random.default_rng(3)
    n = 4096
    words = rng.integers(0, 2**32, size=(n, 6), dtype=np.uint64).astype(np.uint32)
    words[0] = 0
    words[1] = 0xFFFFFFFF
    dev_out = C.sp.sp_debug_philox(torch.from_numpy(words.view(np.int32)).to(C.DEV))
    got = dev_out.cpu().numpy().view(np.uint32)
    for i in range(0, n, 97):
        ref = philox.philox4x32([np.array([words[i, j]]) for j in range(4)],
                                (int(words[i, 4]), int(words[i, 5])))
        assert [int(r[0]) for r in ref] == list(got[i])
    ref = philox.philox4x32([words[:, j] for j in range(4)], (0, 0))   # vectorised key 0 rows
    zero_key = (words[:, 4] == 0) & (words[:, 5] == 0)
    for j in range(4):
        assert np.array_equal(got[zero_key, j], ref[j][zero_key])


# ----------------------------------------------- unfused boundary (ablation)

@pytest.mark.parametrize("variant", [dict(), dict(norm="rmsnorm", eps=1e-6), dict(t=3, s=48),
                                     dict(b=2, s=40, t=4), dict(h=5120, s=32), dict(p=0.0)])
def test_unfused_pipeline_matches_oracle(variant):
    w = wl.Workload("uf", t=2, b=1, s=64, h=512, draw_seed=61).with_(**variant)
    inp = wl.forward_inputs(w, C.DEV)
    y, o, out = C.run_unfused(w, inp)
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    ref = ob.unfused_fwd([C.f32(x) for x in inp["partials"]], [C.f32(x) for x in inp["residual"]],
                         C.f32(inp["bias"]), C.f32(inp["gamma"]), C.f32(inp["beta"]), eps=w.eps,
                         p=w.p, seed=w.seed, offset=w.offset, norm=w.norm, n_gather=1)
    for k in range(w.t):
        assert np.array_equal(compare.bf16_bits(y[k]), compare.bf16_bits(ref["y_shards"][k]))
        assert np.array_equal(compare.bf16_bits(out["z"][k]), compare.bf16_bits(ref["z"][k]))
        assert np.array_equal(out["mask"][k].cpu().numpy(), ref["mask"][k])
        assert not compare.f32_rel_mismatch(out["rstd"][k].cpu().numpy(), ref["rstd"][k]).any()
        mag = ob._norm_rows(ref["z"][k].reshape(-1, w.h).astype(np.float64), C.f32(inp["gamma"]),
                            C.f32(inp["beta"]), w.eps, w.norm)[3].reshape(ref["z"][k].shape)
        C.assert_bf16(compare.bf16_bits(o[k]), ref["out_exact"][k], mag, f"o[{k}]")
    full = np.concatenate(ref["out"], axis=1)
    got = compare.bf16_bits(out["gathered"][0])
    # the gathered copy is the shards' O laid out along s (bit-exact copy of o)
    assert np.array_equal(got, np.concatenate([compare.bf16_bits(x) for x in o], axis=1))
    assert got.shape == compare.bf16_bits(full).shape


def test_unfused_pipeline_70b_sampled():
    """The unfused boundary (bench --pipeline unfused) at the 70B shape in the
    bench's launch configuration, on sampled tokens: the reduce-scatter's bf16
    shard rows equal the oracle's rank-ascending float32 sum rounded to bf16,
    and the shard step's Z and mask (bit for bit), statistics and O (within
    the tolerances) equal the oracle's token-wise forward of those rows."""
    from oracle import bf16 as obf
    from oracle import collectives as oc
    w = wl.WORKLOADS["70b"]
    inp = wl.forward_inputs(w, C.DEV)
    y, o, out = C.run_unfused(w, inp)
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    tokens = C.sample_tokens(w, 48)
    toks = torch.from_numpy(tokens).to(C.DEV)
    prow = [C.f32(P.reshape(-1, w.h).index_select(0, toks))[None] for P in inp["partials"]]
    y16 = obf.bf16_round(np.concatenate(oc.reduce_scatter_seq(prow)[0], axis=1)[0])
    locs = [C.token_shard(w, g) for g in tokens]
    row = lambda lst, k, l: lst[k].reshape(-1, w.h)[l]
    got_y = np.stack([compare.bf16_bits(row(y, k, l)) for k, l in locs])
    assert np.array_equal(got_y, compare.bf16_bits(y16)), "reduce-scatter rows"
    rrow = np.stack([C.f32(row(inp["residual"], k, l)) for k, l in locs])
    ref = ob.forward_rows(y16[None], rrow, tokens, C.f32(inp["bias"]), C.f32(inp["gamma"]),
                          C.f32(inp["beta"]), eps=w.eps, p=w.p, seed=w.seed, offset=w.offset,
                          norm=w.norm)
    z = np.stack([compare.bf16_bits(row(out["z"], k, l)) for k, l in locs])
    assert np.array_equal(z, compare.bf16_bits(ref["z"])), "Z"
    m = np.stack([row(out["mask"], k, l).cpu().numpy() for k, l in locs])
    assert np.array_equal(m, ref["mask"]), "mask"
    rs = np.array([float(out["rstd"][k].reshape(-1)[l]) for k, l in locs])
    assert not compare.f32_rel_mismatch(rs, ref["rstd"]).any(), "rstd"
    mu = np.array([float(out["mean"][k].reshape(-1)[l]) for k, l in locs])
    assert not compare.f32_rel_mismatch(mu, ref["mean"]).any(), "mean"
    got_o = np.stack([compare.bf16_bits(row(o, k, l)) for k, l in locs])
    C.assert_bf16(got_o, ref["out_exact"], ref["out_magnitude"], "O")
    g = compare.bf16_bits(out["gathered"][0].reshape(-1, w.h).index_select(0, toks))
    assert np.array_equal(g, got_o), "gathered rows are the shards' O"


def test_unfused_mask_equals_fused_mask():
    w = wl.Workload("ufm", t=4, b=1, s=128, h=1024, draw_seed=62)
    inp = wl.forward_inputs(w, C.DEV)
    _, _, un = C.run_unfused(w, inp)
    fu = C.run_fwd(w, inp)
    torch.cuda.synchronize()
    for a, b in zip(un["mask"], fu["mask"]):
        assert torch.equal(a, b)


def test_graph_replay_of_a_step_equals_eager_calls():
    """A step (forward, then the backward that reads its Z, mask and stats,
    then the parameter reduce) captured in one CUDA graph, as bench.py times
    it, and replayed twice gives the eager results bit for bit."""
    w = wl.Workload("gr", t=4, b=1, s=2048, h=4096, draw_seed=111)
    inp = wl.forward_inputs(w, C.DEV)
    dy = wl.backward_inputs(w, C.DEV)["dy"]
    fwd_e = C.run_fwd(w, inp)
    bwd_e = C.run_bwd(w, fwd_e, inp["gamma"], dy, None, n_gather=1)
    torch.cuda.synchronize()
    fwd_g, bwd_g = C.alloc_fwd(w, 1, fill=7.0), C.alloc_bwd(w, 1)
    for t in fwd_g["z"] + fwd_g["gathered"] + bwd_g["dres"] + bwd_g["dgat"]:
        t.fill_(7.0)
    C.run_fwd(w, inp, out=fwd_g)                      # warm-up outside the capture
    C.run_bwd(w, fwd_g, inp["gamma"], dy, None, n_gather=1, out=bwd_g)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        C.run_fwd(w, inp, out=fwd_g)
        C.run_bwd(w, fwd_g, inp["gamma"], dy, None, n_gather=1, out=bwd_g)
    for _ in range(2):
        for t in fwd_g["z"] + fwd_g["gathered"] + bwd_g["dres"] + bwd_g["dgat"]:
            t.fill_(7.0)
        g.replay()
        torch.cuda.synchronize()
        C.sp.check_device_status(C.DEV)
        for key in ("z", "mask", "mean", "rstd", "gathered"):
            for a, b in zip(fwd_e[key], fwd_g[key]):
                assert torch.equal(a, b), key
        for key in ("dres", "dgat"):
            for a, b in zip(bwd_e[key], bwd_g[key]):
                assert torch.equal(a, b), key
        for key in ("dgamma", "dbeta", "dbias"):
            assert torch.equal(bwd_e[key], bwd_g[key]), key


# ------------------------------------- tensor-memory parameter-gradient terms

@pytest.fixture
def bwd_shape():
    """Force the backward's launch shape (threads, chunks per row, ring rows)
    for one test; the automatic choice is restored afterwards."""
    def force(threads, chunks, ring=2):
        C.sp.sp_debug_tune(1, ring, 0, threads, chunks)
    yield force
    C.sp.sp_debug_tune(1, 0, 0, 0, 0)


@pytest.mark.parametrize("shape,h", [((256, 4), 8192), ((256, 4), 6152), ((128, 4), 4096),
                                     ((128, 4), 3000), ((320, 2), 5120), ((320, 2), 4000)])
def test_backward_tensor_memory_shapes(bwd_shape, shape, h):
    """The shapes that keep each thread's dgamma / dbeta / dbias terms in
    tensor memory: exact rows and a ragged last chunk, several rows per block."""
    bwd_shape(*shape)
    w = wl.Workload("tm", t=2, b=1, s=1216, h=h, draw_seed=101)
    inp, fwd, b, out = _bwd_setup(w)
    got = C.sp.sp_debug_last_shape(1)
    assert (got["threads"], got["chunks"]) == shape, got
    C.check_bwd_rows(w, fwd, inp["gamma"], b["dy"], None, out, C.sample_tokens(w, 96))
    C.check_param_grads(w, fwd, inp["gamma"], b["dy"], None, out)


@pytest.mark.parametrize("variant", [dict(ring=1), dict(ring=3), dict(norm="rmsnorm", eps=1e-6),
                                     dict(skip=True), dict(n_gather=2), dict(t=3, s=96)])
def test_backward_tensor_memory_variants(bwd_shape, variant):
    v = dict(variant)
    bwd_shape(256, 4, v.pop("ring", 2))
    skip = v.pop("skip", False)
    w = wl.Workload("tv", t=2, b=1, s=640, h=8192, draw_seed=102).with_(**v)
    inp, fwd, b, out = _bwd_setup(w, skip, n_gather=w.n_gather)
    got = C.sp.sp_debug_last_shape(1)
    assert (got["threads"], got["chunks"]) == (256, 4), got
    C.check_bwd_rows(w, fwd, inp["gamma"], b["dy"], b["dz_skip"], out, C.sample_tokens(w, 64))
    C.check_param_grads(w, fwd, inp["gamma"], b["dy"], b["dz_skip"], out)


def test_backward_tensor_memory_mask_free_and_deterministic(bwd_shape):
    bwd_shape(256, 4)
    w = wl.Workload("td", t=2, b=1, s=640, h=8192, draw_seed=103)
    inp, fwd, b, first = _bwd_setup(w)
    again = C.run_bwd(w, fwd, inp["gamma"], b["dy"], None, n_gather=1)
    got = C.alloc_bwd(w, 1)
    C.sp.sp_norm_bwd_philox(b["dy"], fwd["z"], fwd["mean"], fwd["rstd"], inp["gamma"], None,
                            s=w.s, p=w.p, seed=w.seed, offset=w.offset, norm=w.norm,
                            dresidual=got["dres"], dgathered=got["dgat"], dgamma=got["dgamma"],
                            dbeta=got["dbeta"], dbias=got["dbias"], workspace=got["ws"])
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    shape = C.sp.sp_debug_last_shape(1)
    assert (shape["threads"], shape["chunks"]) == (256, 4), shape
    for other in (again, got):
        for a, c in zip(first["dres"] + first["dgat"], other["dres"] + other["dgat"]):
            assert torch.equal(a, c)
        for name in ("dgamma", "dbeta", "dbias"):
            assert torch.equal(first[name], other[name]), name


# ------------------------------------------------------ mask-free backward

@pytest.mark.parametrize("variant", [dict(), dict(norm="rmsnorm", eps=1e-6), dict(t=3, s=48),
                                     dict(b=2, s=40, t=4), dict(p=0.0), dict(h=5120, s=24),
                                     dict(seed=2**40 + 3, offset=2**33 + 1)])
@pytest.mark.parametrize("with_skip", [False, True])
def test_mask_free_backward_equals_stored_mask_backward(variant, with_skip):
    w = wl.Workload("mf", t=2, b=1, s=64, h=512, draw_seed=71).with_(**variant)
    inp = wl.forward_inputs(w, C.DEV)
    fwd = C.run_fwd(w, inp, n_gather=0)
    bi = wl.backward_inputs(w, C.DEV, with_skip=with_skip)
    ref = C.run_bwd(w, fwd, inp["gamma"], bi["dy"], bi["dz_skip"], n_gather=1)
    got = C.alloc_bwd(w, 1)
    C.sp.sp_norm_bwd_philox(bi["dy"], fwd["z"], fwd["mean"], fwd["rstd"], inp["gamma"],
                            bi["dz_skip"], s=w.s, p=w.p, seed=w.seed, offset=w.offset,
                            norm=w.norm, dresidual=got["dres"], dgathered=got["dgat"],
                            dgamma=got["dgamma"],
                            dbeta=got["dbeta"] if w.norm == "layernorm" else None,
                            dbias=got["dbias"], workspace=got["ws"])
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    for a, b in zip(got["dres"] + got["dgat"], ref["dres"] + ref["dgat"]):
        assert np.array_equal(compare.bf16_bits(a), compare.bf16_bits(b))
    for name in ("dgamma", "dbias") + (("dbeta",) if w.norm == "layernorm" else ()):
        assert torch.equal(got[name], ref[name]), name
    # and against the oracle (same checks as the stored-mask backward)
    C.check_bwd_rows(w, fwd, inp["gamma"], bi["dy"], bi["dz_skip"], got, np.arange(w.tokens))
    C.check_param_grads(w, fwd, inp["gamma"], bi["dy"], bi["dz_skip"], got)


@pytest.mark.parametrize("variant", [dict(), dict(norm="rmsnorm", eps=1e-6), dict(b=2, s=40, t=4),
                                     dict(p=0.0), dict(h=5120, s=24), dict(n_gather=3),
                                     dict(seqlens=(5, 17, 3, 40, 1, 9), s=75, t=4, h=256)])
@pytest.mark.parametrize("pipeline", ["fused", "unfused"])
def test_forward_without_mask_then_mask_free_backward(variant, pipeline):
    """mask_out = NULL: the forward writes Z, the statistics and O bit for bit
    as it does with the mask, and stores no mask; the mask-free backward of
    its outputs matches the oracle's backward of the stored-mask forward."""
    w = wl.Workload("nm", t=2, b=1, s=64, h=512, draw_seed=72).with_(**variant)
    inp = wl.forward_inputs(w, C.DEV)
    cu = torch.from_numpy(wl.cu_seqlens(w.seqlens)).to(C.DEV) if w.ragged else None
    ng = max(1, w.n_gather)
    if pipeline == "fused":
        ref = C.run_fwd(w, inp, n_gather=ng)
        got = C.alloc_fwd(w, ng, fill=7.0)
        C.sp.sp_rs_norm_fwd(inp["partials"], inp["residual"], inp["bias"], inp["gamma"],
                            inp["beta"], eps=w.eps, p=w.p, seed=w.seed, offset=w.offset,
                            norm=w.norm, cu_seqlens=cu, z_out=got["z"], mask_out=None,
                            mean_out=got["mean"], rstd_out=got["rstd"], gathered=got["gathered"])
        pairs = [("z", ref["z"], got["z"]), ("gathered", ref["gathered"], got["gathered"])]
    else:
        y, o_ref, ref = C.run_unfused(w, inp, n_gather=0)
        got = C.alloc_fwd(w, 0, fill=7.0)
        o_got = [torch.full_like(x, 7.0) for x in o_ref]
        C.sp.sp_shard_norm_fwd(y, inp["residual"], inp["bias"], inp["gamma"], inp["beta"],
                               s=w.s, eps=w.eps, p=w.p, seed=w.seed, offset=w.offset,
                               norm=w.norm, cu_seqlens=cu, z_out=got["z"], mask_out=None,
                               mean_out=got["mean"], rstd_out=got["rstd"], o_shards=o_got)
        pairs = [("z", ref["z"], got["z"]), ("o", o_ref, o_got)]
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    pairs.append(("rstd", ref["rstd"], got["rstd"]))
    if w.norm == "layernorm":
        pairs.append(("mean", ref["mean"], got["mean"]))
    for name, a_list, b_list in pairs:
        for a, b in zip(a_list, b_list):
            assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else
                               a.view(torch.int32),
                               b.view(torch.int16) if b.dtype == torch.bfloat16 else
                               b.view(torch.int32)), name
    if pipeline == "fused":
        C.fwd_compare_all(w, inp, ref)

    bi = wl.backward_inputs(w, C.DEV)
    mf = C.alloc_bwd(w, 1)
    C.sp.sp_norm_bwd_philox(bi["dy"], got["z"], got["mean"], got["rstd"], inp["gamma"], None,
                            s=w.s, p=w.p, seed=w.seed, offset=w.offset, norm=w.norm,
                            cu_seqlens=cu, dresidual=mf["dres"], dgathered=mf["dgat"],
                            dgamma=mf["dgamma"],
                            dbeta=mf["dbeta"] if w.norm == "layernorm" else None,
                            dbias=mf["dbias"], workspace=mf["ws"])
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    # the oracle backward reads the stored-mask forward's mask
    C.check_bwd_rows(w, ref, inp["gamma"], bi["dy"], None, mf, np.arange(w.tokens))
    C.check_param_grads(w, ref, inp["gamma"], bi["dy"], None, mf)


@pytest.mark.parametrize("variant", [dict(), dict(norm="rmsnorm", eps=1e-6), dict(b=2, s=40, t=4),
                                     dict(p=0.0), dict(p=0.9), dict(h=5120, s=24),
                                     dict(h=96, s=16), dict(h=544, s=32), dict(h=16384, s=8),
                                     dict(n_gather=3),
                                     dict(seqlens=(5, 17, 3, 40, 1, 9), s=75, t=4, h=256)])
@pytest.mark.parametrize("with_skip", [False, True])
def test_bit_mask_forward_and_backward(variant, with_skip):
    """The mask stored one bit per element: the forward's bits are the
    oracle-checked byte mask packed by the oracle's definition, its other
    outputs and the backward reading the bits are bit for bit those of the
    byte-mask pair (same launch shapes, same summation order)."""
    w = wl.Workload("bm", t=2, b=1, s=64, h=512, draw_seed=74).with_(**variant)
    inp = wl.forward_inputs(w, C.DEV)
    cu = torch.from_numpy(wl.cu_seqlens(w.seqlens)).to(C.DEV) if w.ragged else None
    bi = wl.backward_inputs(w, C.DEV, with_skip=with_skip)
    ng = max(1, w.n_gather)
    fwd_b = C.run_fwd(w, inp, n_gather=ng)
    bwd_b = C.run_bwd(w, fwd_b, inp["gamma"], bi["dy"], bi["dz_skip"], n_gather=ng)
    fwd_k, bwd_k = C.run_bitmask_pair(w, inp, bi["dy"], bi["dz_skip"], ng, ng, cu_seqlens=cu)
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    C.fwd_compare_all(w, inp, fwd_b)
    C.assert_bitmask_pair_matches(w, fwd_b, bwd_b, fwd_k, bwd_k)


@pytest.mark.parametrize("h", [8, 520, 1000])
def test_bit_mask_refuses_widths_not_a_multiple_of_32(h):
    """The bit-packed mask needs whole 4-byte words of bits per row: other
    widths are refused by both entry points before anything is enqueued, and
    the outputs stay untouched."""
    w = wl.Workload("bx", t=2, b=1, s=16, h=h, draw_seed=75)
    inp = wl.forward_inputs(w, C.DEV)
    dy = wl.backward_inputs(w, C.DEV)["dy"]
    with pytest.raises(C.sp.SpError) as e:
        C.run_bitmask_pair(w, inp, dy, None, 1, 1)
    assert e.value.name == "SP_ERR_UNSUPPORTED"
    fwd = C.run_fwd(w, inp, n_gather=1)
    out = C.alloc_bwd(w, 1)
    for x in out["dres"]:
        x.fill_(3.0)
    bits = [torch.zeros((w.b, n, h // 8), dtype=torch.uint8, device=C.DEV)
            for n in w.shard_sizes()]
    with pytest.raises(C.sp.SpError) as e:
        C.sp.sp_norm_bwd_bitmask(dy, fwd["z"], bits, fwd["mean"], fwd["rstd"], inp["gamma"],
                                 None, s=w.s, p=w.p, norm=w.norm, dresidual=out["dres"],
                                 dgathered=out["dgat"], workspace=out["ws"])
    assert e.value.name == "SP_ERR_UNSUPPORTED"
    torch.cuda.synchronize()
    assert all(bool((x == 3.0).all()) for x in out["dres"])


@pytest.mark.parametrize("shape,ring", [((256, 4), 2), ((256, 4), 3), ((512, 2), 1),
                                        ((512, 2), 2), ((128, 4), 2)])
def test_bit_mask_backward_forced_shapes(bwd_shape, shape, ring):
    """The bit-mask backward in launch shapes other than the default (the
    tensor-memory shapes, shallower rings): with the same shape forced for
    both, it gives the byte-mask backward's outputs bit for bit."""
    bwd_shape(*shape, ring=ring)
    w = wl.Workload("bmf", t=4, b=1, s=96, h=8192 if shape[0] >= 256 else 4096, draw_seed=76)
    inp = wl.forward_inputs(w, C.DEV)
    # (three staged rows of the tensor-memory shape fit beside a second block
    # only without the skip gradient)
    bi = wl.backward_inputs(w, C.DEV, with_skip=ring < 3)
    fwd_b = C.run_fwd(w, inp, n_gather=1)
    bwd_b = C.run_bwd(w, fwd_b, inp["gamma"], bi["dy"], bi["dz_skip"], n_gather=1)
    fwd_k, bwd_k = C.run_bitmask_pair(w, inp, bi["dy"], bi["dz_skip"], 1, 1)
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    got = C.sp.sp_debug_last_shape(1)
    assert (got["threads"], got["chunks"], got["stages"]) == (shape[0], shape[1], ring)
    C.assert_bitmask_pair_matches(w, fwd_b, bwd_b, fwd_k, bwd_k)


def test_mask_free_backward_70b_sampled():
    w = wl.WORKLOADS["bwd70b"]
    inp = wl.forward_inputs(w, C.DEV)
    fwd = C.run_fwd(w, inp, n_gather=0)
    dy = wl.backward_inputs(w, C.DEV)["dy"]
    got = C.alloc_bwd(w, 1)
    C.sp.sp_norm_bwd_philox(dy, fwd["z"], fwd["mean"], fwd["rstd"], inp["gamma"], None, s=w.s,
                            p=w.p, seed=w.seed, offset=w.offset, norm=w.norm,
                            dresidual=got["dres"], dgathered=got["dgat"], dgamma=got["dgamma"],
                            dbeta=got["dbeta"], dbias=got["dbias"], workspace=got["ws"])
    torch.cuda.synchronize()
    C.check_bwd_rows(w, fwd, inp["gamma"], dy, None, got, C.sample_tokens(w, 48))
    C.check_param_grads(w, fwd, inp["gamma"], dy, None, got)


# ------------------------------------------ backward entered through g

_rs_bwd_check = C.rs_bwd_check


def _run_rs_bwd(w, fwd, inp, parts, skip, n_gather=1):
    out = C.alloc_bwd(w, n_gather)
    C.sp.sp_rs_norm_bwd(parts, fwd["z"], fwd["mask"], fwd["mean"], fwd["rstd"], inp["gamma"],
                        skip, p=w.p, norm=w.norm, dresidual=out["dres"], dgathered=out["dgat"],
                        dgamma=out["dgamma"],
                        dbeta=out["dbeta"] if w.norm == "layernorm" else None,
                        dbias=out["dbias"], workspace=out["ws"])
    return out


@pytest.mark.parametrize("variant", [dict(), dict(norm="rmsnorm", eps=1e-6), dict(t=3, s=48),
                                     dict(b=2, s=40, t=4), dict(t=1), dict(h=5120, s=24),
                                     dict(h=8, s=16), dict(h=2056, s=16), dict(p=0.0),
                                     dict(t=16, s=32), dict(n_gather=0), dict(n_gather=3)])
@pytest.mark.parametrize("with_skip", [False, True])
def test_rs_norm_bwd_full_compare(variant, with_skip):
    w = wl.Workload("rsb", t=2, b=1, s=64, h=512, draw_seed=81).with_(**variant)
    inp = wl.forward_inputs(w, C.DEV)
    fwd = C.run_fwd(w, inp, n_gather=0)
    gen = wl.make_generator(99, C.DEV)
    parts = [(torch.randn((w.b, w.s, w.h), generator=gen, device=C.DEV) * 0.5).to(torch.bfloat16)
             for _ in range(w.t)]
    skip = wl.backward_inputs(w, C.DEV, with_skip=True)["dz_skip"] if with_skip else None
    out = _run_rs_bwd(w, fwd, inp, parts, skip, n_gather=w.n_gather)
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    _rs_bwd_check(w, fwd, inp, parts, skip, out)


def test_rs_norm_bwd_ragged_packed():
    lengths = (5, 17, 3, 40, 1, 9)
    w = wl.Workload("rsr", t=4, b=1, s=sum(lengths), h=256, seqlens=lengths, draw_seed=82)
    inp = wl.forward_inputs(w, C.DEV)
    fwd = C.run_fwd(w, inp, n_gather=0)
    gen = wl.make_generator(98, C.DEV)
    parts = [torch.randn((1, w.s, w.h), generator=gen, device=C.DEV).to(torch.bfloat16)
             for _ in range(w.t)]
    out = C.alloc_bwd(w, 1)
    cu = torch.from_numpy(wl.cu_seqlens(lengths)).to(C.DEV)
    C.sp.sp_rs_norm_bwd(parts, fwd["z"], fwd["mask"], fwd["mean"], fwd["rstd"], inp["gamma"],
                        None, p=w.p, norm=w.norm, cu_seqlens=cu, dresidual=out["dres"],
                        dgathered=out["dgat"], dgamma=out["dgamma"], dbeta=out["dbeta"],
                        dbias=out["dbias"], workspace=out["ws"])
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    _rs_bwd_check(w, fwd, inp, parts, None, out)


def test_rs_norm_bwd_70b_sampled():
    w = wl.WORKLOADS["bwd70b"]
    inp = wl.forward_inputs(w, C.DEV)
    fwd = C.run_fwd(w, inp, n_gather=0)
    gen = wl.make_generator(97, C.DEV)
    parts = [(torch.randn((w.b, w.s, w.h), generator=gen, device=C.DEV) * 0.35).to(torch.bfloat16)
             for _ in range(w.t)]
    out = _run_rs_bwd(w, fwd, inp, parts, None)
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    rng = np.random.default_rng(0)
    tokens = np.unique(np.concatenate([[0, 1, 2047], rng.integers(0, 2048, 40)]))
    _rs_bwd_check(w, fwd, inp, parts, None, out, tokens=tokens)


@pytest.mark.parametrize("variant", [dict(), dict(norm="rmsnorm", eps=1e-6), dict(t=3, s=48),
                                     dict(b=2, s=40, t=4), dict(h=5120, s=24), dict(h=96, s=16),
                                     dict(t=16, s=32), dict(n_gather=3), dict(p=0.0),
                                     dict(seqlens=(5, 17, 3, 40, 1, 9), s=75, t=4, h=256)])
@pytest.mark.parametrize("with_skip", [False, True])
def test_rs_norm_bwd_bit_mask_equals_byte_mask(variant, with_skip):
    """The backward entered through g reading the mask as bits (the oracle's
    packing of the stored byte mask) gives every output of the byte-mask call
    bit for bit."""
    w = wl.Workload("rsbits", t=2, b=1, s=64, h=512, draw_seed=83).with_(**variant)
    cu = torch.from_numpy(wl.cu_seqlens(w.seqlens)).to(C.DEV) if w.ragged else None
    inp = wl.forward_inputs(w, C.DEV)
    fwd = C.run_fwd(w, inp, n_gather=0)
    gen = wl.make_generator(96, C.DEV)
    parts = [(torch.randn((w.b, w.s, w.h), generator=gen, device=C.DEV) * 0.5).to(torch.bfloat16)
             for _ in range(w.t)]
    skip = wl.backward_inputs(w, C.DEV, with_skip=True)["dz_skip"] if with_skip else None
    ng = w.n_gather
    ref = C.alloc_bwd(w, ng)
    C.sp.sp_rs_norm_bwd(parts, fwd["z"], fwd["mask"], fwd["mean"], fwd["rstd"], inp["gamma"],
                        skip, p=w.p, norm=w.norm, cu_seqlens=cu, dresidual=ref["dres"],
                        dgathered=ref["dgat"], dgamma=ref["dgamma"],
                        dbeta=ref["dbeta"] if w.norm == "layernorm" else None,
                        dbias=ref["dbias"], workspace=ref["ws"])
    got = C.run_rs_bwd_bitmask(w, fwd, inp, parts, skip, C.oracle_mask_bits(fwd["mask"]), ng,
                               cu_seqlens=cu)
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    C.assert_bwd_outputs_equal(w, ref, got)


@pytest.mark.parametrize("t,h,skip", [(2, 16384, False), (16, 8192, True)])
def test_rs_norm_bwd_rejects_shapes_it_cannot_run(t, h, skip):
    """h above 8192, and t = 16 at h = 8192 with a skip gradient (the t partial
    stages and the row buffers do not fit one SM's shared memory), are
    refused before anything is launched; outputs stay untouched."""
    w = wl.Workload("rsx", t=t, b=1, s=2 * t, h=h, draw_seed=85)
    inp = wl.forward_inputs(w, C.DEV)
    fwd = C.run_fwd(w, inp, n_gather=0)
    gen = wl.make_generator(86, C.DEV)
    parts = [torch.randn((1, w.s, w.h), generator=gen, device=C.DEV).to(torch.bfloat16)
             for _ in range(w.t)]
    sk = wl.backward_inputs(w, C.DEV, with_skip=True)["dz_skip"] if skip else None
    out = C.alloc_bwd(w, 1)
    for x in out["dres"] + out["dgat"]:
        x.fill_(5.0)
    torch.cuda.synchronize()
    with pytest.raises(C.sp.SpError) as e:
        C.sp.sp_rs_norm_bwd(parts, fwd["z"], fwd["mask"], fwd["mean"], fwd["rstd"],
                            inp["gamma"], sk, p=w.p, norm=w.norm, dresidual=out["dres"],
                            dgathered=out["dgat"], dgamma=out["dgamma"], dbeta=out["dbeta"],
                            dbias=out["dbias"], workspace=out["ws"])
    assert e.value.name == "SP_ERR_UNSUPPORTED"
    torch.cuda.synchronize()
    assert all(bool((x.float() == 5.0).all()) for x in out["dres"] + out["dgat"])


def test_rs_norm_bwd_equals_unfused_reduce_then_norm_bwd_within_rounding():
    """The unfused path rounds the reduced dY to bf16 before the norm backward;
    with bf16-exact sums (few significant bits) the two agree bit for bit."""
    w = wl.Workload("rse", t=4, b=1, s=64, h=1024, draw_seed=83)
    inp = wl.forward_inputs(w, C.DEV)
    fwd = C.run_fwd(w, inp, n_gather=0)
    gen = wl.make_generator(96, C.DEV)
    parts = [(torch.randint(-8, 8, (1, w.s, w.h), generator=gen, device=C.DEV) / 64)
             .to(torch.bfloat16) for _ in range(w.t)]
    fused = _run_rs_bwd(w, fwd, inp, parts, None)
    dy = [torch.empty((1, n, w.h), dtype=torch.bfloat16, device=C.DEV) for n in w.shard_sizes()]
    C.sp.sp_reduce_scatter_seq(parts, dy)
    plain = C.run_bwd(w, fwd, inp["gamma"], dy, None, n_gather=1)
    torch.cuda.synchronize()
    for a, b in zip(fused["dres"] + fused["dgat"], plain["dres"] + plain["dgat"]):
        assert np.array_equal(compare.bf16_bits(a), compare.bf16_bits(b))


def test_one_kernel_across_shared_memory_sizes():
    """The same kernel instantiation (run-time t) needs more shared memory for
    more ranks; calls with large, small, then medium needs must all launch."""
    for t in (16, 2, 5, 3, 16):
        w = wl.Workload("sm", t=t, b=1, s=16 * t, h=512, draw_seed=90 + t)
        inp = wl.forward_inputs(w, C.DEV)
        out = C.run_fwd(w, inp)
        torch.cuda.synchronize()
        C.check_fwd_rows(w, inp, out, C.sample_tokens(w, 8))


# ------------------------------------------------------ default launch shapes

@pytest.mark.parametrize("h,fwd_threads,bwd_shape", [(8192, 256, (512, 2)), (5120, 128, (320, 2)),
                                                     (4096, 256, (256, 2))])
def test_default_launch_shapes(h, fwd_threads, bwd_shape):
    """The launch shapes the library picks by default for the workloads'
    row widths (the measured choices): forward threads per block (whole rows,
    no cluster), backward (threads, chunks per row)."""
    w = wl.Workload("ds", t=8, b=1, s=64, h=h, draw_seed=151)
    _bwd_setup(w)
    f = C.sp.sp_debug_last_shape(0)
    assert f["threads"] == fwd_threads and f["cluster"] == 1, f
    b = C.sp.sp_debug_last_shape(1)
    assert (b["threads"], b["chunks"]) == bwd_shape, b
    if h == 8192:
        assert b["stages"] == 3, b   # one block per SM stages three rows
