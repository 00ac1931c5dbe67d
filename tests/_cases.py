"""Shared helpers of the GPU parity tests: run the CUDA path, run the oracle,
compare at the tolerances stated in ``oracle.compare``."""
import numpy as np
import torch

from oracle import boundary as ob
from oracle import compare
from sp_boundary_norm_gb300 import binding as sp
from sp_boundary_norm_gb300 import workloads as wl

DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


def f32(x):
    return None if x is None else x.float().cpu().numpy()


def assert_bf16(gpu_bits, ref_exact, magnitude, what):
    """The bf16 bar (1 ulp, or the magnitude floor on cancelled results), and
    no more elements passing through the floor alone than its stated bound."""
    bad = compare.bf16_mismatch(gpu_bits, ref_exact, magnitude)
    assert not bad.any(), f"{what}: {bad.sum()} elements off"
    floor_only = int(compare.bf16_floor_only(gpu_bits, ref_exact, magnitude).sum())
    assert floor_only <= compare.floor_only_bound(bad.size), \
        f"{what}: {floor_only} of {bad.size} elements pass only through the magnitude floor"
    return floor_only


def alloc_fwd(w, n_gather, dev=DEV, fill=None):
    sizes = w.shard_sizes()
    mk = lambda shape, dt: (torch.empty(shape, dtype=dt, device=dev) if fill is None else
                            torch.full(shape, fill, dtype=dt, device=dev) if dt.is_floating_point
                            else torch.full(shape, 0xAB, dtype=dt, device=dev))
    return {
        "z": [mk((w.b, n, w.h), torch.bfloat16) for n in sizes],
        "mask": [mk((w.b, n, w.h), torch.uint8) for n in sizes],
        "mean": [mk((w.b, n), torch.float32) for n in sizes] if w.norm == "layernorm" else None,
        "rstd": [mk((w.b, n), torch.float32) for n in sizes],
        "gathered": [mk((w.b, w.s, w.h), torch.bfloat16) for _ in range(n_gather)],
    }


def run_fwd(w, inp, n_gather=None, out=None, cu_seqlens=None):
    n_gather = w.n_gather if n_gather is None else n_gather
    out = alloc_fwd(w, n_gather) if out is None else out
    if cu_seqlens is None and w.ragged:
        cu_seqlens = torch.from_numpy(wl.cu_seqlens(w.seqlens)).to(DEV)
    sp.sp_rs_norm_fwd(inp["partials"], inp["residual"], inp["bias"], inp["gamma"], inp["beta"],
                      eps=w.eps, p=w.p, seed=w.seed, offset=w.offset, norm=w.norm,
                      cu_seqlens=cu_seqlens, z_out=out["z"], mask_out=out["mask"],
                      mean_out=out["mean"], rstd_out=out["rstd"], gathered=out["gathered"])
    return out


def alloc_bwd(w, n_gather, dev=DEV):
    sizes = w.shard_sizes()
    ws = torch.empty(max(16, sp.sp_norm_bwd_workspace_bytes(w.b, w.s, w.h, w.t, w.norm)),
                     dtype=torch.uint8, device=dev)
    return {
        "dres": [torch.empty((w.b, n, w.h), dtype=torch.bfloat16, device=dev) for n in sizes],
        "dgat": [torch.empty((w.b, w.s, w.h), dtype=torch.bfloat16, device=dev)
                 for _ in range(n_gather)],
        "dgamma": torch.empty(w.h, dtype=torch.float32, device=dev),
        "dbeta": torch.empty(w.h, dtype=torch.float32, device=dev),
        "dbias": torch.empty(w.h, dtype=torch.float32, device=dev),
        "ws": ws,
    }


def run_bwd(w, fwd_out, gamma, dy, dz_skip=None, n_gather=None, out=None, cu_seqlens=None):
    n_gather = w.n_gather if n_gather is None else n_gather
    out = alloc_bwd(w, n_gather) if out is None else out
    if cu_seqlens is None and w.ragged:
        cu_seqlens = torch.from_numpy(wl.cu_seqlens(w.seqlens)).to(DEV)
    sp.sp_norm_bwd(dy, fwd_out["z"], fwd_out["mask"], fwd_out["mean"], fwd_out["rstd"], gamma,
                   dz_skip, s=w.s, p=w.p, norm=w.norm, cu_seqlens=cu_seqlens,
                   dresidual=out["dres"], dgathered=out["dgat"], dgamma=out["dgamma"],
                   dbeta=out["dbeta"] if w.norm == "layernorm" else None, dbias=out["dbias"],
                   workspace=out["ws"])
    return out


def run_unfused(w, inp, n_gather=1):
    """The boundary as three calls: reduce-scatter (bf16 shards), the norm on
    the shards, all-gather of the shards' O.  Returns (y, o, out)."""
    sizes = w.shard_sizes()
    e = lambda shape, dt: torch.empty(shape, dtype=dt, device=DEV)
    y = [e((w.b, n, w.h), torch.bfloat16) for n in sizes]
    out = alloc_fwd(w, n_gather)
    o = [e((w.b, n, w.h), torch.bfloat16) for n in sizes]
    cu = torch.from_numpy(wl.cu_seqlens(w.seqlens)).to(DEV) if w.ragged else None
    sp.sp_reduce_scatter_seq(inp["partials"], y, cu_seqlens=cu)
    sp.sp_shard_norm_fwd(y, inp["residual"], inp["bias"], inp["gamma"], inp["beta"], s=w.s,
                         eps=w.eps, p=w.p, seed=w.seed, offset=w.offset, norm=w.norm,
                         cu_seqlens=cu, z_out=out["z"], mask_out=out["mask"],
                         mean_out=out["mean"], rstd_out=out["rstd"], o_shards=o)
    if n_gather:
        sp.sp_allgather_seq(o, out["gathered"], s=w.s, cu_seqlens=cu)
    return y, o, out


def fwd_compare_all(w, inp, out):
    """Every element of a (small) forward against the oracle: Z and the mask
    bit for bit, the statistics at 1e-5, every gathered copy at the bf16 bar."""
    ref = ob.rs_norm_fwd([f32(x) for x in inp["partials"]], [f32(x) for x in inp["residual"]],
                         f32(inp["bias"]), f32(inp["gamma"]), f32(inp["beta"]), eps=w.eps,
                         p=w.p, seed=w.seed, offset=w.offset, norm=w.norm,
                         n_gather=len(out["gathered"]))
    for k in range(w.t):
        assert np.array_equal(compare.bf16_bits(out["z"][k]), compare.bf16_bits(ref["z"][k])), k
        assert np.array_equal(out["mask"][k].cpu().numpy(), ref["mask"][k]), k
        assert not compare.f32_rel_mismatch(out["rstd"][k].cpu().numpy(), ref["rstd"][k]).any()
        if w.norm == "layernorm":
            assert not compare.f32_rel_mismatch(out["mean"][k].cpu().numpy(), ref["mean"][k]).any()
    out_exact = np.concatenate(ref["out_exact"], axis=1)
    mag = np.concatenate([ob._norm_rows(z.reshape(-1, w.h).astype(np.float64), f32(inp["gamma"]),
                                        f32(inp["beta"]), w.eps, w.norm)[3].reshape(z.shape)
                          for z in ref["z"]], axis=1)
    for j, g in enumerate(out["gathered"]):
        assert_bf16(compare.bf16_bits(g), out_exact, mag, f"gathered[{j}]")
    return ref


def rs_bwd_check(w, fwd, inp, parts, skip, out, tokens=None):
    """dResidual / dYpre rows and parameter sums against the oracle, with dY
    the float32 rank-ascending sum of the partial gradients on each shard."""
    from oracle import collectives as coll
    h = w.h
    flat = [f32(x) for x in parts]
    dy_shards, _ = coll.reduce_scatter_seq(flat)
    offs = [(k * w.s) // w.t for k in range(w.t + 1)]
    g = f32(inp["gamma"])
    acc = {n: np.zeros(h) for n in ("dgamma", "dbeta", "dbias")}
    sq = {n: np.zeros(h) for n in acc}
    scale = float(ob.dropout_scale(w.p))
    for k in range(w.t):
        n = w.b * (offs[k + 1] - offs[k])
        if n == 0:
            continue
        rows = lambda x: x[k].reshape(-1, h)
        one = ob.backward_rows(dy_shards[k].reshape(-1, h), f32(rows(fwd["z"])),
                               rows(fwd["mask"]).cpu().numpy(),
                               None if w.norm != "layernorm" else fwd["mean"][k].reshape(-1).cpu().numpy(),
                               fwd["rstd"][k].reshape(-1).cpu().numpy(), g,
                               None if skip is None else f32(rows(skip)), p=w.p, norm=w.norm)
        sel = np.arange(n) if tokens is None else tokens[(tokens >= 0) & (tokens < n)]
        dres = compare.bf16_bits(out["dres"][k].reshape(-1, h))
        assert_bf16(dres[sel], one["dz"][sel], one["dz_magnitude"][sel], f"dresidual[{k}]")
        for j, dg in enumerate(out["dgat"]):
            blk = compare.bf16_bits(dg[:, offs[k]:offs[k + 1], :].reshape(-1, h))
            assert_bf16(blk[sel], one["dypre_exact"][sel], one["dz_magnitude"][sel] * scale,
                          f"dgathered[{j}] shard {k}")
        for name in acc:
            terms = one[name + "_terms"]
            if terms is not None:
                acc[name] += terms.sum(axis=0)
                sq[name] += (terms * terms).sum(axis=0)
    for name in ("dgamma", "dbias") + (("dbeta",) if w.norm == "layernorm" else ()):
        bad = compare.colsum_mismatch(out[name].cpu().numpy(), acc[name], np.sqrt(sq[name]))
        assert not bad.any(), name


def bits_equal(a, b):
    """Bit-for-bit equality of two tensors (bf16 and float32 compared as integers)."""
    view = {torch.bfloat16: torch.int16, torch.float32: torch.int32}
    if a.dtype in view:
        a, b = a.view(view[a.dtype]), b.view(view[b.dtype])
    return torch.equal(a, b)


def run_bitmask_pair(w, inp, dy, dz_skip, n_gather_fwd, n_gather_bwd, cu_seqlens=None):
    """The forward storing the mask one bit per element and the backward
    reading it.  Returns (fwd outputs with "mask_bits", bwd outputs)."""
    sizes = w.shard_sizes()
    fwd = alloc_fwd(w, n_gather_fwd, fill=7.0)
    fwd["mask_bits"] = [torch.full((w.b, n, w.h // 8), 0xAB, dtype=torch.uint8, device=DEV)
                        for n in sizes]
    sp.sp_rs_norm_fwd_bitmask(inp["partials"], inp["residual"], inp["bias"], inp["gamma"],
                              inp["beta"], eps=w.eps, p=w.p, seed=w.seed, offset=w.offset,
                              norm=w.norm, cu_seqlens=cu_seqlens, z_out=fwd["z"],
                              mask_bits_out=fwd["mask_bits"], mean_out=fwd["mean"],
                              rstd_out=fwd["rstd"], gathered=fwd["gathered"])
    bwd = alloc_bwd(w, n_gather_bwd)
    sp.sp_norm_bwd_bitmask(dy, fwd["z"], fwd["mask_bits"], fwd["mean"], fwd["rstd"],
                           inp["gamma"], dz_skip, s=w.s, p=w.p, norm=w.norm,
                           cu_seqlens=cu_seqlens, dresidual=bwd["dres"], dgathered=bwd["dgat"],
                           dgamma=bwd["dgamma"],
                           dbeta=bwd["dbeta"] if w.norm == "layernorm" else None,
                           dbias=bwd["dbias"], workspace=bwd["ws"])
    return fwd, bwd


def assert_bitmask_pair_matches(w, fwd_bytes, bwd_bytes, fwd_bits, bwd_bits):
    """The bit-mask pair against the byte-mask pair: the bits are the byte
    mask packed by the oracle's definition, every other output bit for bit."""
    for k in range(w.t):
        want = ob.pack_mask_bits(fwd_bytes["mask"][k].cpu().numpy())
        assert np.array_equal(fwd_bits["mask_bits"][k].cpu().numpy(), want), f"mask bits {k}"
    keys = ["z", "rstd", "gathered"] + (["mean"] if w.norm == "layernorm" else [])
    for key in keys:
        for a, b in zip(fwd_bytes[key], fwd_bits[key]):
            assert bits_equal(a, b), key
    for key in ("dres", "dgat"):
        for a, b in zip(bwd_bytes[key], bwd_bits[key]):
            assert bits_equal(a, b), key
    for key in ("dgamma", "dbias") + (("dbeta",) if w.norm == "layernorm" else ()):
        assert bits_equal(bwd_bytes[key], bwd_bits[key]), key


def oracle_mask_bits(byte_masks):
    """The oracle's packing of device byte masks, as device tensors."""
    return [torch.from_numpy(ob.pack_mask_bits(m.cpu().numpy())).to(DEV) for m in byte_masks]


def run_rs_bwd_bitmask(w, fwd, inp, parts, dz_skip, mask_bits, n_gather, cu_seqlens=None):
    out = alloc_bwd(w, n_gather)
    sp.sp_rs_norm_bwd_bitmask(parts, fwd["z"], mask_bits, fwd["mean"], fwd["rstd"], inp["gamma"],
                              dz_skip, p=w.p, norm=w.norm, cu_seqlens=cu_seqlens,
                              dresidual=out["dres"], dgathered=out["dgat"], dgamma=out["dgamma"],
                              dbeta=out["dbeta"] if w.norm == "layernorm" else None,
                              dbias=out["dbias"], workspace=out["ws"])
    return out


def assert_bwd_outputs_equal(w, a, b):
    for key in ("dres", "dgat"):
        for x, y in zip(a[key], b[key]):
            assert bits_equal(x, y), key
    for key in ("dgamma", "dbias") + (("dbeta",) if w.norm == "layernorm" else ()):
        assert bits_equal(a[key], b[key]), key


def token_shard(w, g):
    """(shard k, local row) of global token g for b == 1 or dense b > 1."""
    bi, si = divmod(int(g), w.s)
    offs = [(k * w.s) // w.t for k in range(w.t + 1)]
    k = max(j for j in range(w.t) if offs[j] <= si and offs[j + 1] > si)
    return k, bi * (offs[k + 1] - offs[k]) + (si - offs[k])


def sample_tokens(w, n, seed=0):
    """Spread of tokens incl. the first and last token of every shard."""
    offs = [(k * w.s) // w.t for k in range(w.t + 1)]
    picks = set()
    for bi in range(w.b):
        for k in range(w.t):
            if offs[k + 1] > offs[k]:
                picks.add(bi * w.s + offs[k])
                picks.add(bi * w.s + offs[k + 1] - 1)
    rng = np.random.default_rng(seed)
    picks.update(int(x) for x in rng.integers(0, w.b * w.s, size=max(0, n - len(picks))))
    return np.array(sorted(picks), dtype=np.int64)


def check_fwd_rows(w, inp, out, tokens):
    """Compare the given tokens' outputs with the oracle's per-token forward."""
    t, h = w.t, w.h
    toks = torch.from_numpy(tokens).to(DEV)
    flat = [P.reshape(-1, h) for P in inp["partials"]]
    prow = np.stack([f32(F.index_select(0, toks)) for F in flat])          # (t, n, h)
    locs = [token_shard(w, g) for g in tokens]
    rrow = np.stack([f32(inp["residual"][k].reshape(-1, h)[l]) for k, l in locs])
    ref = ob.forward_rows(prow, rrow, tokens, f32(inp["bias"]), f32(inp["gamma"]),
                          f32(inp["beta"]), eps=w.eps, p=w.p, seed=w.seed, offset=w.offset,
                          norm=w.norm)
    z = np.stack([compare.bf16_bits(out["z"][k].reshape(-1, h)[l]) for k, l in locs])
    assert np.array_equal(z, compare.bf16_bits(ref["z"])), "Z must be bit-exact"
    m = np.stack([out["mask"][k].reshape(-1, h)[l].cpu().numpy() for k, l in locs])
    assert np.array_equal(m, ref["mask"]), "mask must be bit-exact"
    rs = np.array([float(out["rstd"][k].reshape(-1)[l]) for k, l in locs])
    assert not compare.f32_rel_mismatch(rs, ref["rstd"]).any(), "rstd"
    if w.norm == "layernorm":
        mu = np.array([float(out["mean"][k].reshape(-1)[l]) for k, l in locs])
        assert not compare.f32_rel_mismatch(mu, ref["mean"]).any(), "mean"
    for j, g in enumerate(out["gathered"]):
        o = compare.bf16_bits(g.reshape(-1, h).index_select(0, toks))
        assert_bf16(o, ref["out_exact"], ref["out_magnitude"], f"gathered[{j}]")
    return ref


def check_bwd_rows(w, fwd_out, gamma, dy, dz_skip, out, tokens):
    h = w.h
    locs = [token_shard(w, g) for g in tokens]
    pick = lambda lst, k, l: lst[k].reshape(-1, h)[l]
    dyr = np.stack([f32(pick(dy, k, l)) for k, l in locs])
    zr = np.stack([f32(pick(fwd_out["z"], k, l)) for k, l in locs])
    mr = np.stack([pick(fwd_out["mask"], k, l).cpu().numpy() for k, l in locs])
    rs = np.array([float(fwd_out["rstd"][k].reshape(-1)[l]) for k, l in locs])
    mu = (np.array([float(fwd_out["mean"][k].reshape(-1)[l]) for k, l in locs])
          if w.norm == "layernorm" else None)
    sk = None if dz_skip is None else np.stack([f32(pick(dz_skip, k, l)) for k, l in locs])
    ref = ob.backward_rows(dyr, zr, mr, mu, rs, f32(gamma), sk, p=w.p, norm=w.norm)
    dres = np.stack([compare.bf16_bits(pick(out["dres"], k, l)) for k, l in locs])
    assert_bf16(dres, ref["dz"], ref["dz_magnitude"], "dresidual")
    toks = torch.from_numpy(tokens).to(DEV)
    scale = float(ob.dropout_scale(w.p))
    for j, g in enumerate(out["dgat"]):
        o = compare.bf16_bits(g.reshape(-1, h).index_select(0, toks))
        assert_bf16(o, ref["dypre_exact"], ref["dz_magnitude"] * scale, f"dgathered[{j}]")
    return ref


def check_param_grads(w, fwd_out, gamma, dy, dz_skip, out):
    """Full oracle parameter gradients, shard by shard (float64)."""
    h = w.h
    acc = {n: np.zeros(h) for n in ("dgamma", "dbeta", "dbias")}
    sq = {n: np.zeros(h) for n in acc}
    g = f32(gamma)
    for k in range(w.t):
        n = fwd_out["z"][k].numel() // h
        if n == 0:
            continue
        step = 4096
        for lo in range(0, n, step):
            sl = slice(lo, min(n, lo + step))
            rows = lambda x: None if x is None else f32(x[k].reshape(-1, h)[sl])
            one = ob.backward_rows(
                rows(dy), rows(fwd_out["z"]), fwd_out["mask"][k].reshape(-1, h)[sl].cpu().numpy(),
                None if w.norm != "layernorm" else fwd_out["mean"][k].reshape(-1)[sl].cpu().numpy(),
                fwd_out["rstd"][k].reshape(-1)[sl].cpu().numpy(), g, rows(dz_skip), p=w.p,
                norm=w.norm)
            for name in acc:
                terms = one[name + "_terms"]
                if terms is None:
                    continue
                acc[name] += terms.sum(axis=0)
                sq[name] += (terms * terms).sum(axis=0)
    names = ["dgamma", "dbias"] + (["dbeta"] if w.norm == "layernorm" else [])
    for name in names:
        got = out[name].cpu().numpy()
        bad = compare.colsum_mismatch(got, acc[name], np.sqrt(sq[name]))
        assert not bad.any(), f"{name}: {bad.sum()} channels off, max err " \
            f"{np.max(np.abs(got - acc[name])):.3g}"


# ------------------------------------------------ every element at full size
#
# The full-size workloads are checked element by element with the oracle run
# over chunks of tokens in a thread pool: numpy releases the GIL inside its
# array operations, so the chunks run in parallel on the host cores without
# copying the inputs between processes.

CHUNK = 128


def host_threads():
    import os
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:
        n = os.cpu_count() or 1
    return max(1, min(32, n))


def _bits_rows(shards, h):
    """bf16 shard tensors (b, s_k, h) -> host uint16 (b*s, h) in global token order."""
    full = torch.cat([x.reshape(x.shape[0], -1, h) for x in shards], dim=1).reshape(-1, h)
    return full.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _full_bits(x, h):
    return x.reshape(-1, h).contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _u8_rows(shards, h):
    return torch.cat([x.reshape(x.shape[0], -1, h) for x in shards], dim=1).reshape(-1, h) \
        .cpu().numpy()


def _vec_rows(shards):
    return torch.cat([x.reshape(x.shape[0], -1) for x in shards], dim=1).reshape(-1).cpu().numpy()


def _val(bits):
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _pool_map(fn, n_rows):
    from concurrent.futures import ThreadPoolExecutor
    starts = list(range(0, n_rows, CHUNK))
    with ThreadPoolExecutor(max_workers=host_threads()) as ex:
        return list(ex.map(fn, starts))


def _add_counts(parts):
    tot = {}
    for part in parts:
        for key, v in part.items():
            tot[key] = tot.get(key, 0) + v
    return tot


def full_fwd_check(w, inp, out):
    """Every token of a forward against the oracle's per-token forward: Z and
    the mask bit for bit, mean / rstd within 1e-5, each gathered copy within
    the bf16 bar with floor-only elements bounded.  Returns the counts."""
    h, T = w.h, w.tokens
    parts = [_full_bits(P, h) for P in inp["partials"]]
    R = _bits_rows(inp["residual"], h)
    Z = _bits_rows(out["z"], h)
    M = _u8_rows(out["mask"], h)
    RS = _vec_rows(out["rstd"])
    MU = _vec_rows(out["mean"]) if w.norm == "layernorm" else None
    G = [_full_bits(g, h) for g in out["gathered"]]
    bias, gamma, beta = f32(inp["bias"]), f32(inp["gamma"]), f32(inp["beta"])

    def chunk(lo):
        hi = min(T, lo + CHUNK)
        ref = ob.forward_rows(np.stack([_val(P[lo:hi]) for P in parts]), _val(R[lo:hi]),
                              np.arange(lo, hi, dtype=np.int64), bias, gamma, beta, eps=w.eps,
                              p=w.p, seed=w.seed, offset=w.offset, norm=w.norm)
        c = {"z_bad": int((Z[lo:hi] != compare.bf16_bits(ref["z"])).sum()),
             "mask_bad": int((M[lo:hi] != ref["mask"]).sum()),
             "rstd_bad": int(compare.f32_rel_mismatch(RS[lo:hi], ref["rstd"]).sum()),
             "mean_bad": 0 if MU is None else
             int(compare.f32_rel_mismatch(MU[lo:hi], ref["mean"]).sum()),
             "o_bad": 0, "o_floor_only": 0}
        for g in G:
            c["o_bad"] += int(compare.bf16_mismatch(g[lo:hi], ref["out_exact"],
                                                    ref["out_magnitude"]).sum())
            c["o_floor_only"] += int(compare.bf16_floor_only(g[lo:hi], ref["out_exact"],
                                                             ref["out_magnitude"]).sum())
        return c

    tot = _add_counts(_pool_map(chunk, T))
    n_o = T * h * len(G)
    assert tot["z_bad"] == 0 and tot["mask_bad"] == 0, tot
    assert tot["rstd_bad"] == 0 and tot["mean_bad"] == 0, tot
    assert tot["o_bad"] == 0, tot
    assert tot["o_floor_only"] <= compare.floor_only_bound(n_o), tot
    tot["elements"] = T * h
    return tot


def full_bwd_check(w, fwd_out, gamma, dy, dz_skip, out, dy_partials=None):
    """Every token of a backward against the oracle's per-token backward (on
    the GPU's own saved Z, mask and statistics): dResidual and every gathered
    dYpre copy within the bf16 bar with floor-only elements bounded, and the
    parameter gradients summed over all tokens in float64.  With
    ``dy_partials`` (the t full partial gradients of the backward entered
    through g) dY is the oracle's reduce-scatter of them, unrounded, and
    ``dy`` is unused.  Returns the counts."""
    from oracle import collectives as coll
    h, T = w.h, w.tokens
    if dy_partials is None:
        DY = _bits_rows(dy, h)
        dy_rows = lambda lo, hi: _val(DY[lo:hi])
    else:
        PD = [_full_bits(x, h) for x in dy_partials]

        def dy_rows(lo, hi):
            shards, _ = coll.reduce_scatter_seq([_val(P[lo:hi])[None] for P in PD])
            return np.concatenate([np.asarray(x).reshape(-1, h) for x in shards], axis=0)
    Z = _bits_rows(fwd_out["z"], h)
    M = _u8_rows(fwd_out["mask"], h)
    RS = _vec_rows(fwd_out["rstd"])
    MU = _vec_rows(fwd_out["mean"]) if w.norm == "layernorm" else None
    SK = None if dz_skip is None else _bits_rows(dz_skip, h)
    DR = _bits_rows(out["dres"], h)
    DG = [_full_bits(g, h) for g in out["dgat"]]
    g32 = f32(gamma)
    scale = float(ob.dropout_scale(w.p))
    names = ["dgamma", "dbias"] + (["dbeta"] if w.norm == "layernorm" else [])

    def chunk(lo):
        hi = min(T, lo + CHUNK)
        ref = ob.backward_rows(dy_rows(lo, hi), _val(Z[lo:hi]), M[lo:hi],
                               None if MU is None else MU[lo:hi], RS[lo:hi], g32,
                               None if SK is None else _val(SK[lo:hi]), p=w.p, norm=w.norm)
        c = {"dres_bad": int(compare.bf16_mismatch(DR[lo:hi], ref["dz"],
                                                   ref["dz_magnitude"]).sum()),
             "dres_floor_only": int(compare.bf16_floor_only(DR[lo:hi], ref["dz"],
                                                            ref["dz_magnitude"]).sum()),
             "dgat_bad": 0, "dgat_floor_only": 0}
        for g in DG:
            c["dgat_bad"] += int(compare.bf16_mismatch(g[lo:hi], ref["dypre_exact"],
                                                       ref["dz_magnitude"] * scale).sum())
            c["dgat_floor_only"] += int(compare.bf16_floor_only(
                g[lo:hi], ref["dypre_exact"], ref["dz_magnitude"] * scale).sum())
        sums = {n: (ref[n + "_terms"].sum(axis=0), (ref[n + "_terms"] ** 2).sum(axis=0))
                for n in names}
        return c, sums

    results = _pool_map(chunk, T)
    tot = _add_counts([c for c, _ in results])
    n = T * h
    assert tot["dres_bad"] == 0 and tot["dgat_bad"] == 0, tot
    assert tot["dres_floor_only"] <= compare.floor_only_bound(n), tot
    assert tot["dgat_floor_only"] <= compare.floor_only_bound(n * max(1, len(DG))), tot
    for name in names:   # chunk order is fixed, so the float64 sums are too
        acc = np.zeros(h)
        sq = np.zeros(h)
        for _, sums in results:
            acc += sums[name][0]
            sq += sums[name][1]
        got = out[name].cpu().numpy()
        bad = compare.colsum_mismatch(got, acc, np.sqrt(sq))
        assert not bad.any(), f"{name}: {bad.sum()} channels off"
    tot["elements"] = n
    return tot


def full_unfused_fwd_check(w, inp, y, o, out):
    """Every token of the unfused boundary: the reduce-scatter's bf16 shard
    rows equal the oracle's rank-ascending float32 sum rounded to bf16 (bit
    for bit); the shard step's Z and mask (bit for bit), statistics and O
    (bf16 bar) equal the oracle's token-wise forward of those rows; every
    gathered copy holds the shards' O bit for bit.  Returns the counts."""
    from oracle import bf16 as obf
    from oracle import collectives as oc
    h, T = w.h, w.tokens
    parts = [_full_bits(P, h) for P in inp["partials"]]
    R = _bits_rows(inp["residual"], h)
    Y = _bits_rows(y, h)
    Z = _bits_rows(out["z"], h)
    M = _u8_rows(out["mask"], h)
    RS = _vec_rows(out["rstd"])
    MU = _vec_rows(out["mean"]) if w.norm == "layernorm" else None
    O = _bits_rows(o, h)
    G = [_full_bits(g, h) for g in out["gathered"]]
    bias, gamma, beta = f32(inp["bias"]), f32(inp["gamma"]), f32(inp["beta"])

    def chunk(lo):
        hi = min(T, lo + CHUNK)
        shards, _ = oc.reduce_scatter_seq([_val(P[lo:hi])[None] for P in parts])
        y16 = obf.bf16_round(np.concatenate([np.asarray(x).reshape(-1, h) for x in shards]))
        ref = ob.forward_rows(y16[None], _val(R[lo:hi]), np.arange(lo, hi, dtype=np.int64),
                              bias, gamma, beta, eps=w.eps, p=w.p, seed=w.seed,
                              offset=w.offset, norm=w.norm)
        return {"y_bad": int((Y[lo:hi] != compare.bf16_bits(y16)).sum()),
                "z_bad": int((Z[lo:hi] != compare.bf16_bits(ref["z"])).sum()),
                "mask_bad": int((M[lo:hi] != ref["mask"]).sum()),
                "rstd_bad": int(compare.f32_rel_mismatch(RS[lo:hi], ref["rstd"]).sum()),
                "mean_bad": 0 if MU is None else
                int(compare.f32_rel_mismatch(MU[lo:hi], ref["mean"]).sum()),
                "o_bad": int(compare.bf16_mismatch(O[lo:hi], ref["out_exact"],
                                                   ref["out_magnitude"]).sum()),
                "o_floor_only": int(compare.bf16_floor_only(O[lo:hi], ref["out_exact"],
                                                            ref["out_magnitude"]).sum()),
                "gathered_bad": sum(int((g[lo:hi] != O[lo:hi]).sum()) for g in G)}

    tot = _add_counts(_pool_map(chunk, T))
    for key in ("y_bad", "z_bad", "mask_bad", "rstd_bad", "mean_bad", "o_bad", "gathered_bad"):
        assert tot[key] == 0, tot
    assert tot["o_floor_only"] <= compare.floor_only_bound(T * h), tot
    tot["elements"] = T * h
    return tot
