"""Stream order across the library's calls.

Every kernel of the library is launched with programmatic stream
serialisation: its blocks may be placed on the SMs while the previous kernel
on the stream is still running, and each waits for that kernel to complete
before it touches global memory.  These tests run chains of calls in which
every call reads what the call before it wrote, and writes buffers that the
call before it read (two buffer sets, alternating), and require the chain to
give bit for bit what the same chain gives with the device synchronised after
every call -- back to back on one stream and replayed as one CUDA graph.
Every kernel is deterministic, so any read of a buffer before its producer
finished, or any write before its last reader finished, shows as a changed
bit."""
import pytest
import torch

from sp_boundary_norm_gb300 import binding as sp
from sp_boundary_norm_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

C = pytest.importorskip("_cases")


@pytest.fixture(scope="module", autouse=True)
def _built(lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield

STEPS = 4


def _alloc_set(w, dev):
    """One buffer set: everything one step of the chain writes."""
    sizes = w.shard_sizes()
    e = lambda shape, dt: torch.empty(shape, dtype=dt, device=dev)
    shard = lambda dt: [e((w.b, n, w.h), dt) for n in sizes]
    stats = lambda: [e((w.b, n), torch.float32) for n in sizes]
    full = lambda k: [e((w.b, w.s, w.h), torch.bfloat16) for _ in range(k)]
    vec = lambda: e((w.h,), torch.float32)
    st = {
        # fused forward
        "z": shard(torch.bfloat16), "mask": shard(torch.uint8), "mean": stats(),
        "rstd": stats(), "g": full(w.t),
        # backward from the shards (stored mask) and its parameter gradients
        "d": shard(torch.bfloat16), "dg": full(1), "dgamma": vec(), "dbeta": vec(),
        "dbias": vec(),
        # backward entered through g (the t partial gradients reduce-scattered)
        "d2": shard(torch.bfloat16), "dg2": full(1), "dgamma2": vec(), "dbeta2": vec(),
        "dbias2": vec(),
        # the unfused forward: reduce-scatter, norm on the shards, all-gather
        "y": shard(torch.bfloat16), "z2": shard(torch.bfloat16), "mask2": shard(torch.uint8),
        "mean2": stats(), "rstd2": stats(), "o2": shard(torch.bfloat16), "g2": full(1),
        # the bit-mask forward and backward
        "zk": shard(torch.bfloat16), "bits": [e((w.b, n, w.h // 8), torch.uint8) for n in sizes],
        "meank": stats(), "rstdk": stats(), "gk": full(1), "dk": shard(torch.bfloat16),
        "dgk": full(1), "dgammak": vec(), "dbetak": vec(), "dbiask": vec(),
        # the forward storing no mask and the mask-free backward
        "zn": shard(torch.bfloat16), "meann": stats(), "rstdn": stats(), "gn": full(1),
        "dn": shard(torch.bfloat16), "dgn": full(1), "dgamman": vec(), "dbetan": vec(),
        "dbiasn": vec(),
    }
    if w.norm != "layernorm":   # RMSNorm has no mean and no beta
        for key in ("mean", "mean2", "dbeta", "dbeta2", "meank", "dbetak", "meann", "dbetan"):
            del st[key]
    return st


def _tensors(st):
    for v in st.values():
        if isinstance(v, list):
            yield from v
        else:
            yield v


def _poison(sets):
    for st in sets:
        for x in _tensors(st):
            if x.dtype == torch.uint8:
                x.fill_(0xA5)
            else:
                x.fill_(float("nan"))


def _chain(w, inp, dy, cu, sets, ws, sync):
    """STEPS steps; step i reads set (i - 1) % 2 (the inputs for i = 0) and
    writes set i % 2.  Per step: fused forward -> backward from the shards
    (+ parameter reduce) -> backward through g (+ parameter reduce) ->
    reduce-scatter -> shard norm -> all-gather -> bit-mask forward ->
    bit-mask backward (+ reduce) -> forward storing no mask -> mask-free
    backward (+ reduce); each reads what the call before it wrote."""
    after = (lambda: torch.cuda.synchronize()) if sync else (lambda: None)
    prev = {"g": inp["partials"], "z2": inp["residual"], "d2": dy}
    for i in range(STEPS):
        cur = sets[i % 2]
        sp.sp_rs_norm_fwd(prev["g"], prev["z2"], inp["bias"], inp["gamma"], inp["beta"],
                          eps=w.eps, p=w.p, seed=w.seed, offset=w.offset + i, norm=w.norm,
                          cu_seqlens=cu, z_out=cur["z"], mask_out=cur["mask"],
                          mean_out=cur.get("mean"), rstd_out=cur["rstd"], gathered=cur["g"])
        after()
        sp.sp_norm_bwd(prev["d2"], cur["z"], cur["mask"], cur.get("mean"), cur["rstd"],
                       inp["gamma"], None, s=w.s, p=w.p, norm=w.norm, cu_seqlens=cu,
                       dresidual=cur["d"], dgathered=cur["dg"], dgamma=cur["dgamma"],
                       dbeta=cur.get("dbeta"), dbias=cur["dbias"], workspace=ws)
        after()
        sp.sp_rs_norm_bwd(cur["g"], cur["z"], cur["mask"], cur.get("mean"), cur["rstd"],
                          inp["gamma"], None, p=w.p, norm=w.norm, cu_seqlens=cu,
                          dresidual=cur["d2"], dgathered=cur["dg2"], dgamma=cur["dgamma2"],
                          dbeta=cur.get("dbeta2"), dbias=cur["dbias2"],
                          workspace=ws)
        after()
        sp.sp_reduce_scatter_seq(cur["g"], cur["y"], cu_seqlens=cu)
        after()
        sp.sp_shard_norm_fwd(cur["y"], cur["d"], inp["bias"], inp["gamma"], inp["beta"], s=w.s,
                             eps=w.eps, p=w.p, seed=w.seed, offset=w.offset + 100 + i,
                             norm=w.norm, cu_seqlens=cu, z_out=cur["z2"],
                             mask_out=cur["mask2"], mean_out=cur.get("mean2"),
                             rstd_out=cur["rstd2"], o_shards=cur["o2"])
        after()
        sp.sp_allgather_seq(cur["o2"], cur["g2"], s=w.s, cu_seqlens=cu)
        after()
        sp.sp_rs_norm_fwd_bitmask([cur["g2"][0]] * w.t, cur["z2"], inp["bias"], inp["gamma"],
                                  inp["beta"], eps=w.eps, p=w.p, seed=w.seed,
                                  offset=w.offset + 200 + i, norm=w.norm, cu_seqlens=cu,
                                  z_out=cur["zk"], mask_bits_out=cur["bits"],
                                  mean_out=cur.get("meank"), rstd_out=cur["rstdk"],
                                  gathered=cur["gk"])
        after()
        sp.sp_norm_bwd_bitmask(cur["d2"], cur["zk"], cur["bits"], cur.get("meank"),
                               cur["rstdk"], inp["gamma"], None, s=w.s, p=w.p, norm=w.norm,
                               cu_seqlens=cu, dresidual=cur["dk"], dgathered=cur["dgk"],
                               dgamma=cur["dgammak"], dbeta=cur.get("dbetak"),
                               dbias=cur["dbiask"], workspace=ws)
        after()
        sp.sp_rs_norm_fwd([cur["gk"][0]] * w.t, cur["dk"], inp["bias"], inp["gamma"],
                          inp["beta"], eps=w.eps, p=w.p, seed=w.seed, offset=w.offset + 300 + i,
                          norm=w.norm, cu_seqlens=cu, z_out=cur["zn"], mask_out=None,
                          mean_out=cur.get("meann"), rstd_out=cur["rstdn"], gathered=cur["gn"])
        after()
        sp.sp_norm_bwd_philox(cur["dk"], cur["zn"], cur.get("meann"), cur["rstdn"], inp["gamma"],
                              None, s=w.s, p=w.p, seed=w.seed, offset=w.offset + 300 + i,
                              norm=w.norm, cu_seqlens=cu, dresidual=cur["dn"],
                              dgathered=cur["dgn"], dgamma=cur["dgamman"],
                              dbeta=cur.get("dbetan"), dbias=cur["dbiasn"], workspace=ws)
        after()
        prev = cur


def _snapshot(sets):
    return [[x.clone() for x in _tensors(st)] for st in sets]


def _same(a, b):
    for sa, sb in zip(a, b):
        for x, y in zip(sa, sb):
            if x.dtype == torch.float32:
                x, y = x.view(torch.int32), y.view(torch.int32)
            if not torch.equal(x, y):
                return False
    return True


@pytest.mark.parametrize("variant", [
    dict(t=4, b=1, s=2048, h=4096),
    dict(t=8, b=2, s=1024, h=8192, norm="rmsnorm", eps=1e-6),
    dict(t=4, b=1, s=2048, h=5120, seqlens=(700, 1, 1200, 147)),
])
def test_dependent_calls_back_to_back_and_in_a_graph_equal_synchronised_calls(variant):
    w = wl.Workload("chain", draw_seed=515, p=0.1, **variant)
    inp = wl.forward_inputs(w, C.DEV)
    dy = wl.backward_inputs(w, C.DEV)["dy"]
    cu = torch.from_numpy(wl.cu_seqlens(w.seqlens)).to(C.DEV) if w.ragged else None
    sets = [_alloc_set(w, C.DEV), _alloc_set(w, C.DEV)]
    ws = torch.empty(max(16, sp.sp_norm_bwd_workspace_bytes(w.b, w.s, w.h, w.t, w.norm)),
                     dtype=torch.uint8, device=C.DEV)

    _poison(sets)
    _chain(w, inp, dy, cu, sets, ws, sync=True)
    torch.cuda.synchronize()
    sp.check_device_status(C.DEV)
    ref = _snapshot(sets)
    for st in sets:   # every output written and finite
        for x in _tensors(st):
            if x.dtype != torch.uint8:
                assert torch.isfinite(x.float()).all()

    for rep in range(3):
        _poison(sets)
        _chain(w, inp, dy, cu, sets, ws, sync=False)
        torch.cuda.synchronize()
        sp.check_device_status(C.DEV)
        assert _same(ref, _snapshot(sets)), f"back to back, repetition {rep}"

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _chain(w, inp, dy, cu, sets, ws, sync=False)
    for rep in range(3):
        _poison(sets)
        g.replay()
        torch.cuda.synchronize()
        sp.check_device_status(C.DEV)
        assert _same(ref, _snapshot(sets)), f"graph replay {rep}"


def test_independent_calls_on_separate_streams_equal_serial_calls():
    """Three independent problems (their own inputs, outputs and workspaces),
    each forward + backward on a stream of its own, forked from and joined to
    the current stream as the bench runs length buckets: the bits of the same
    calls run one after another."""
    shapes = [dict(t=8, b=1, s=1024, h=4096), dict(t=4, b=1, s=2048, h=5120,
                                                    seqlens=(700, 1, 1200, 147)),
              dict(t=8, b=2, s=512, h=8192, norm="rmsnorm", eps=1e-6)]
    ws_ = [wl.Workload(f"par{i}", draw_seed=600 + i, **v) for i, v in enumerate(shapes)]
    inps = [wl.forward_inputs(w, C.DEV) for w in ws_]
    dys = [wl.backward_inputs(w, C.DEV)["dy"] for w in ws_]
    cus = [torch.from_numpy(wl.cu_seqlens(w.seqlens)).to(C.DEV) if w.ragged else None
           for w in ws_]

    def run_all(streams):
        outs = []
        main = torch.cuda.current_stream(C.DEV)
        fork = torch.cuda.Event()
        fork.record(main)
        joins = []
        for i, w in enumerate(ws_):
            f = C.alloc_fwd(w, 1, fill=7.0)
            b = C.alloc_bwd(w, 1)
            stream = streams[i] if streams else main
            stream.wait_event(fork)
            with torch.cuda.stream(stream):
                C.run_fwd(w, inps[i], n_gather=1, out=f, cu_seqlens=cus[i])
                C.run_bwd(w, f, inps[i]["gamma"], dys[i], None, n_gather=1, out=b,
                          cu_seqlens=cus[i])
                done = torch.cuda.Event()
                done.record(stream)
            joins.append(done)
            outs.append((f, b))
        for done in joins:
            main.wait_event(done)
        torch.cuda.synchronize()
        C.sp.check_device_status(C.DEV)
        return outs

    serial = run_all(None)
    streams = [torch.cuda.Stream(C.DEV) for _ in ws_]
    for rep in range(3):
        par = run_all(streams)
        for w, (fs, bs), (fp, bp) in zip(ws_, serial, par):
            for key in ("z", "mask", "rstd", "gathered") + (("mean",) if w.norm == "layernorm"
                                                             else ()):
                for a, b in zip(fs[key], fp[key]):
                    assert C.bits_equal(a, b), (w.name, key, rep)
            C.assert_bwd_outputs_equal(w, bs, bp)
