"""Seeded random shapes through every entry point, every element against the oracle.

Each case draws a shape the hand-picked variants may not combine: a rank count
t from 1 to 16, a width h from 8 to 16384 channels (any multiple of 8, so the
last chunk of a row is usually partial), dense batches of 1-3 rows or packed
sequences with random lengths (empty ones included, shards cut at floor(kT/t)
so they differ by a token), dropout p in {0, 0.1, 0.3, 0.9}, LayerNorm or
RMSNorm, 64-bit seeds and offsets, 0 to t gathered copies, with or without the
skip-path gradient.  Per case:

  - the fused forward: Z and the mask bit for bit, statistics at 1e-5, every
    gathered copy at the bf16 bar ("第 7 课：序列并行 SP" §2 and §3: the
    token-wise operators give the same result on whichever rank holds the
    token); and the same forward storing no mask, bit for bit the same;
  - the unfused forward (reduce-scatter, norm on the shards, all-gather) on the
    same inputs, against the oracle from its bf16 shard sums;
  - the backward from the shards with the stored mask, and the mask-free one
    from the forward that stored none, every dResidual / dYpre element and the
    parameter-gradient column sums; the forward and backward with the mask
    stored one bit per element, bit for bit the byte-mask pair (h a multiple
    of 32; other widths: the refusal);
  - the backward entered through g (t partial gradients reduce-scattered), or,
    for the shapes whose partial stages do not fit one SM's shared memory,
    the documented refusal with nothing written.

The case list is fixed by the seed, so a failure names a reproducible shape.
"""
import numpy as np
import pytest
import torch

from oracle import compare
from sp_boundary_norm_gb300 import workloads as wl

C = pytest.importorskip("_cases")

N_CASES = 24
ELEMS = 1 << 20          # tokens x h per case (the oracle finishes in about a second)


@pytest.fixture
def gpu(lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield


def draw_case(i):
    """Workload, skip flag and backward gathered-copy count of case i."""
    rng = np.random.default_rng(90_000 + i)
    t = int(rng.choice([1, 2, 3, 4, 5, 7, 8, 11, 13, 16]))
    h = 8 * int(np.clip(np.round(np.exp(rng.uniform(0.0, np.log(2048.0)))), 1, 2048))
    max_tokens = max(1, min(ELEMS // h, (8 * ELEMS) // (h * t), 4096))
    norm = "layernorm" if rng.random() < 0.6 else "rmsnorm"
    kw = dict(t=t, h=h, p=float(rng.choice([0.0, 0.1, 0.3, 0.9])), norm=norm,
              eps=1e-5 if norm == "layernorm" else 1e-6,
              seed=int(rng.integers(0, 2**63)), offset=int(rng.integers(0, 2**40)),
              draw_seed=1000 + i)
    if rng.random() < 0.4:   # packed sequences
        n_seqs = int(rng.integers(1, 9))
        lengths = [int(x) for x in rng.geometric(min(1.0, n_seqs / max_tokens), n_seqs)]
        lengths = [0 if rng.random() < 0.1 else min(x, max_tokens) for x in lengths]
        while sum(lengths) > max_tokens:
            j = int(np.argmax(lengths))
            lengths[j] //= 2
        if sum(lengths) == 0:
            lengths[0] = 1
        w = wl.Workload(f"rand{i}", b=1, s=sum(lengths), seqlens=tuple(lengths), **kw)
    else:
        b = int(rng.integers(1, 4))
        per = max(1, max_tokens // (b * t))
        w = wl.Workload(f"rand{i}", b=b, s=t * int(rng.integers(1, per + 1)), **kw)
    w = w.with_(n_gather=int(rng.choice([0, 1, 2, t])))
    return w, bool(rng.random() < 0.5), int(rng.choice([0, 1, 2]))


def test_case_list_spans_the_shape_space():
    """The drawn cases cover what they claim (checked without a GPU run)."""
    cases = [draw_case(i) for i in range(N_CASES)]
    ws = [c[0] for c in cases]
    assert {w.norm for w in ws} == {"layernorm", "rmsnorm"}
    assert any(w.ragged for w in ws) and any(not w.ragged for w in ws)
    assert any(w.h % 2048 != 0 for w in ws) and max(w.h for w in ws) >= 4096
    assert any(w.t >= 11 for w in ws) and any(w.t == 1 for w in ws)
    assert {w.p for w in ws} >= {0.0, 0.9}
    assert any(c[1] for c in cases) and any(not c[1] for c in cases)
    assert any(w.h % 32 == 0 for w in ws) and any(w.h % 32 for w in ws)   # bits, refusal
    for w in ws:
        assert w.h % 8 == 0 and 8 <= w.h <= 16384 and w.tokens * w.h <= ELEMS
        assert w.ragged or w.s % w.t == 0


def _cu(w):
    return torch.from_numpy(wl.cu_seqlens(w.seqlens)).to(C.DEV) if w.ragged else None


def _untouched(out, fill_bits):
    for x in out["dres"] + out["dgat"]:
        if x.numel() and not bool((x.view(torch.int16) == fill_bits).all()):
            return False
    return True


@pytest.mark.gpu
@pytest.mark.parametrize("i", range(N_CASES))
def test_random_shape_every_entry_point_every_element(gpu, i):
    w, with_skip, n_gather_bwd = draw_case(i)
    print(f"case {i}: t={w.t} b={w.b} s={w.s} h={w.h} p={w.p} {w.norm} "
          f"lengths={w.seqlens} n_gather={w.n_gather} skip={with_skip} bwd copies={n_gather_bwd}")
    cu = _cu(w)
    inp = wl.forward_inputs(w, C.DEV)

    # fused forward
    fwd = C.run_fwd(w, inp, cu_seqlens=cu)
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    C.fwd_compare_all(w, inp, fwd)

    # the same forward storing no mask: the same bits everywhere else
    nm = C.alloc_fwd(w, w.n_gather, fill=7.0)
    C.sp.sp_rs_norm_fwd(inp["partials"], inp["residual"], inp["bias"], inp["gamma"], inp["beta"],
                        eps=w.eps, p=w.p, seed=w.seed, offset=w.offset, norm=w.norm,
                        cu_seqlens=cu, z_out=nm["z"], mask_out=None, mean_out=nm["mean"],
                        rstd_out=nm["rstd"], gathered=nm["gathered"])
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    for key in ("z", "gathered", "rstd") + (("mean",) if w.norm == "layernorm" else ()):
        for a, b in zip(fwd[key], nm[key]):
            assert torch.equal(a.view(torch.int16 if a.dtype == torch.bfloat16 else torch.int32),
                               b.view(torch.int16 if b.dtype == torch.bfloat16 else torch.int32)), key

    # unfused forward: reduce-scatter, norm on the shards, all-gather
    y, o, un = C.run_unfused(w, inp, n_gather=max(1, w.n_gather))
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    C.full_unfused_fwd_check(w, inp, y, o, un)

    # backward from the shards: stored mask, then the mask drawn again
    bi = wl.backward_inputs(w, C.DEV, with_skip=with_skip)
    tokens = np.arange(w.tokens, dtype=np.int64)
    out = C.run_bwd(w, fwd, inp["gamma"], bi["dy"], bi["dz_skip"], n_gather=n_gather_bwd,
                    cu_seqlens=cu)
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    C.check_bwd_rows(w, fwd, inp["gamma"], bi["dy"], bi["dz_skip"], out, tokens)
    C.check_param_grads(w, fwd, inp["gamma"], bi["dy"], bi["dz_skip"], out)

    # the mask stored one bit per element (h a multiple of 32): the byte mask
    # packed, the rest bit for bit; other widths are refused
    if w.h % 32 == 0:
        fwd_k, bwd_k = C.run_bitmask_pair(w, inp, bi["dy"], bi["dz_skip"], w.n_gather,
                                          n_gather_bwd, cu_seqlens=cu)
        torch.cuda.synchronize()
        C.sp.check_device_status(C.DEV)
        C.assert_bitmask_pair_matches(w, fwd, out, fwd_k, bwd_k)
    else:
        with pytest.raises(C.sp.SpError):
            C.run_bitmask_pair(w, inp, bi["dy"], bi["dz_skip"], w.n_gather, n_gather_bwd,
                               cu_seqlens=cu)

    mf = C.alloc_bwd(w, n_gather_bwd)   # from the forward that stored no mask
    C.sp.sp_norm_bwd_philox(bi["dy"], nm["z"], nm["mean"], nm["rstd"], inp["gamma"],
                            bi["dz_skip"], s=w.s, p=w.p, seed=w.seed, offset=w.offset,
                            norm=w.norm, cu_seqlens=cu, dresidual=mf["dres"],
                            dgathered=mf["dgat"], dgamma=mf["dgamma"],
                            dbeta=mf["dbeta"] if w.norm == "layernorm" else None,
                            dbias=mf["dbias"], workspace=mf["ws"])
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    C.check_bwd_rows(w, fwd, inp["gamma"], bi["dy"], bi["dz_skip"], mf, tokens)
    C.check_param_grads(w, fwd, inp["gamma"], bi["dy"], bi["dz_skip"], mf)

    # backward entered through g
    gen = wl.make_generator(5000 + i, C.DEV)
    parts = [(torch.randn((w.b, w.s, w.h), generator=gen, device=C.DEV) * 0.5)
             .to(torch.bfloat16) for _ in range(w.t)]
    rs = C.alloc_bwd(w, n_gather_bwd)
    fill = -12345   # a bf16 bit pattern no result has here (a NaN payload)
    for x in rs["dres"] + rs["dgat"]:
        x.view(torch.int16).fill_(fill)
    try:
        C.sp.sp_rs_norm_bwd(parts, fwd["z"], fwd["mask"], fwd["mean"], fwd["rstd"],
                            inp["gamma"], bi["dz_skip"], p=w.p, norm=w.norm, cu_seqlens=cu,
                            dresidual=rs["dres"], dgathered=rs["dgat"], dgamma=rs["dgamma"],
                            dbeta=rs["dbeta"] if w.norm == "layernorm" else None,
                            dbias=rs["dbias"], workspace=rs["ws"])
    except C.sp.SpError as e:
        # refused before launch: only h above 8192, and h above 4096 with a
        # skip gradient and t >= 15 (the t partial stages and the row buffers
        # do not share one SM's shared memory)
        assert e.name == "SP_ERR_UNSUPPORTED", e
        assert w.h > 8192 or (with_skip and w.t >= 15 and w.h > 4096), (w.h, w.t, with_skip)
        torch.cuda.synchronize()
        assert _untouched(rs, fill)
        return
    torch.cuda.synchronize()
    C.sp.check_device_status(C.DEV)
    C.rs_bwd_check(w, fwd, inp, parts, bi["dz_skip"], rs)
    if w.h % 32 == 0:   # the same call reading the bit-packed mask: the same bits
        rk = C.run_rs_bwd_bitmask(w, fwd, inp, parts, bi["dz_skip"],
                                  C.oracle_mask_bits(fwd["mask"]), n_gather_bwd, cu_seqlens=cu)
        torch.cuda.synchronize()
        C.sp.check_device_status(C.DEV)
        C.assert_bwd_outputs_equal(w, rs, rk)
