"""Pins of the oracle's fused boundary, forward and backward (CPU only).

Each check ties the oracle to something other than itself: a textbook
library routine (torch's layer_norm / rms_norm / autograd, in float64), an
invariant the lesson "第 7 课：序列并行 SP" states (token-wise ops commute
with sequence sharding, §3; masks agree across ranks, answer to Q1), a closed
form (moments of a normalised row, §2), or brute force (finite differences).
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import boundary as ob
from oracle import collectives as coll
from oracle.bf16 import bf16_round
from sp_boundary_norm_gb300 import workloads as wl


def _np(x):
    return None if x is None else x.float().numpy()


def _inputs(w, seed=None):
    raw = wl.forward_inputs(w, "cpu", seed)
    return {"partials": [_np(x) for x in raw["partials"]],
            "residual": [_np(x) for x in raw["residual"]],
            "bias": _np(raw["bias"]), "gamma": _np(raw["gamma"]),
            "beta": _np(raw["beta"])}


def _fwd(w, inp, **kw):
    args = dict(eps=w.eps, p=w.p, seed=w.seed, offset=w.offset, norm=w.norm,
                n_gather=w.n_gather)
    args.update(kw)
    return ob.rs_norm_fwd(inp["partials"], inp["residual"], inp["bias"],
                          inp["gamma"], inp["beta"], **args)


SMALL = wl.Workload("small", t=4, b=2, s=12, h=64, draw_seed=11)


@pytest.mark.parametrize("norm", ["layernorm", "rmsnorm"])
def test_t1_p0_is_textbook_norm(norm):
    w = SMALL.with_(t=1, p=0.0, norm=norm, eps=1e-5 if norm == "layernorm" else 1e-6)
    inp = _inputs(w)
    res = _fwd(w, inp)
    P0 = torch.from_numpy(inp["partials"][0])
    R = torch.from_numpy(inp["residual"][0])
    bias = torch.from_numpy(inp["bias"])
    # fp32: (P0 + bias) + R, then bf16
    z = ((P0 + bias) + R).to(torch.bfloat16)
    assert np.array_equal(res["z"][0], z.float().numpy())
    assert res["mask"][0].all()
    z64 = z.double()
    g64 = torch.from_numpy(inp["gamma"]).double()
    if norm == "layernorm":
        ref = F.layer_norm(z64, (w.h,), g64, torch.from_numpy(inp["beta"]).double(), w.eps)
        var, mu = torch.var_mean(z64, dim=-1, unbiased=False)
        np.testing.assert_allclose(res["mean"][0], mu.float().numpy(), rtol=2e-7, atol=0)
    else:
        ref = F.rms_norm(z64, (w.h,), g64, w.eps)
        var = (z64 * z64).mean(-1)
    np.testing.assert_allclose(res["out_exact"][0], ref.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(res["out"][0], bf16_round(ref.numpy()))
    np.testing.assert_allclose(res["rstd"][0], (1 / torch.sqrt(var + w.eps)).float().numpy(),
                               rtol=2e-7, atol=0)


@pytest.mark.parametrize("t,s,b", [(2, 12, 2), (4, 12, 1), (8, 37, 1), (3, 10, 3)])
@pytest.mark.parametrize("norm", ["layernorm", "rmsnorm"])
def test_sharded_equals_unsharded_sliced_by_token(t, s, b, norm):
    w = SMALL.with_(t=t, s=s, b=b, norm=norm, n_gather=2)
    inp = _inputs(w)
    res = _fwd(w, inp)
    full_res = np.concatenate(inp["residual"], axis=1)
    un = ob.unsharded_fwd(inp["partials"], full_res, inp["bias"], inp["gamma"],
                          inp["beta"], eps=w.eps, p=w.p, seed=w.seed, norm=norm)
    offs = coll.shard_offsets(s, t)
    for k in range(t):
        sl = slice(offs[k], offs[k + 1])
        for key in ("z", "mask", "out"):
            assert np.array_equal(res[key][k], un[key][:, sl, :]), key
        assert np.array_equal(res["rstd"][k], un["rstd"][:, sl])
        if norm == "layernorm":
            assert np.array_equal(res["mean"][k], un["mean"][:, sl])
    for g in res["gathered"]:
        assert np.array_equal(g, un["out"])


def test_unit_gamma_zero_beta_moments():
    w = SMALL.with_(t=2, h=256)
    inp = _inputs(w)
    inp["gamma"] = np.ones(w.h, np.float32)
    inp["beta"] = np.zeros(w.h, np.float32)
    res = _fwd(w, inp)
    for k in range(w.t):
        o = res["out_exact"][k].reshape(-1, w.h)
        z = res["z"][k].reshape(-1, w.h).astype(np.float64)
        var = z.var(axis=-1)
        np.testing.assert_allclose(o.mean(-1), 0.0, atol=1e-12)
        np.testing.assert_allclose(o.var(-1), var / (var + w.eps), rtol=1e-12)
        ob16 = res["out"][k].reshape(-1, w.h).astype(np.float64)
        assert np.abs(ob16.mean(-1)).max() <= 1e-3
        assert np.abs(ob16.var(-1) - 1).max() <= 1e-2


def test_mask_independent_of_sharding_and_batch_position():
    base = wl.Workload("m", t=2, b=1, s=48, h=32, draw_seed=5)
    inp2 = _inputs(base)
    m2 = np.concatenate(_fwd(base, inp2)["mask"], axis=1)
    for t in (1, 3, 8):
        w = base.with_(t=t)
        inp = _inputs(w)
        mt = np.concatenate(_fwd(w, inp)["mask"], axis=1)
        assert np.array_equal(mt, m2)


def test_dropout_rate_scale_and_degenerate_p():
    w = wl.Workload("d", t=2, b=1, s=64, h=512, p=0.1, draw_seed=6)
    inp = _inputs(w)
    res = _fwd(w, inp)
    mask = np.concatenate(res["mask"], axis=1)
    n = mask.size
    drop = 1 - mask.mean()
    assert abs(drop - 0.1) < 5 * np.sqrt(0.1 * 0.9 / n)
    # dropped elements carry the residual only; kept ones the scaled sum
    y = (inp["partials"][0] + inp["partials"][1]).astype(np.float32) + inp["bias"]
    z = np.concatenate(res["z"], axis=1)
    r = np.concatenate(inp["residual"], axis=1)
    dropped = mask == 0
    assert np.array_equal(z[dropped], r[dropped])
    kept = ~dropped
    np.testing.assert_allclose((z - r)[kept], (y / 0.9)[kept], atol=2 ** -6)
    # inverted dropout keeps the expectation: E[mask * scale] == 1
    assert abs(mask.mean() * float(ob.dropout_scale(0.1)) - 1) < 5 * np.sqrt(0.1 / 0.9 / n)
    # p = 0: nothing dropped, scale exactly 1
    res0 = _fwd(w.with_(p=0.0), inp)
    assert all(m.all() for m in res0["mask"])
    assert ob.dropout_threshold(0.0) == 0 and ob.dropout_scale(0.0) == 1.0
    assert ob.dropout_threshold(0.1) == 429496729
    with pytest.raises(ValueError):
        ob.dropout_threshold(1.0)


def test_seed_and_offset_change_the_mask():
    w = wl.Workload("d", t=1, b=1, s=32, h=256, draw_seed=6)
    inp = _inputs(w)
    m = _fwd(w, inp)["mask"][0]
    assert not np.array_equal(m, _fwd(w.with_(seed=4321), inp)["mask"][0])
    assert not np.array_equal(m, _fwd(w.with_(offset=1), inp)["mask"][0])


def test_forward_rows_matches_full_forward():
    w = SMALL.with_(t=4, s=20, b=2)
    inp = _inputs(w)
    res = _fwd(w, inp)
    offs = coll.shard_offsets(w.s, w.t)
    tokens = np.array([0, 5, 19, 20, 33, 39])
    P = np.stack(inp["partials"])            # (t, b, s, h)
    for g in tokens:
        bi, si = divmod(int(g), w.s)
        k = max(j for j in range(w.t) if offs[j] <= si)
        row = ob.forward_rows(P[:, bi, si, :][:, None, :],
                              inp["residual"][k][bi, si - offs[k]][None, :],
                              np.array([g]), inp["bias"], inp["gamma"], inp["beta"],
                              eps=w.eps, p=w.p, seed=w.seed, norm=w.norm)
        assert np.array_equal(row["z"][0], res["z"][k][bi, si - offs[k]])
        assert np.array_equal(row["out"][0], res["out"][k][bi, si - offs[k]])
        assert np.array_equal(row["mask"][0], res["mask"][k][bi, si - offs[k]])


# ---------------------------------------------------------------- backward --

def _loss_and_grads_fd(w, inp, dy, dz_skip, which, idx, step=1e-6):
    """Central finite difference of L = sum_k <dY_k, O_k> + <dZskip_k, Z_k>."""
    def loss(inp_):
        r = _fwd(w, inp_, exact=True, n_gather=0)
        tot = 0.0
        for k in range(w.t):
            tot += float((dy[k] * r["out_exact"][k]).sum())
            if dz_skip is not None:
                tot += float((dz_skip[k] * r["z"][k]).sum())
        return tot

    def bumped(delta):
        cp = {k: ([a.astype(np.float64) for a in v] if isinstance(v, list) else
                  (None if v is None else v.astype(np.float64)))
              for k, v in inp.items()}
        arr = cp[which[0]] if len(which) == 1 else cp[which[0]][which[1]]
        arr[idx] += delta
        return cp

    return (loss(bumped(step)) - loss(bumped(-step))) / (2 * step)


@pytest.mark.parametrize("norm", ["layernorm", "rmsnorm"])
@pytest.mark.parametrize("with_skip", [False, True])
def test_backward_matches_finite_differences(norm, with_skip):
    w = wl.Workload("fd", t=2, b=1, s=8, h=16, p=0.25, norm=norm, draw_seed=9)
    inp = _inputs(w)
    rng = np.random.default_rng(0)
    sizes = w.shard_sizes()
    dy = [rng.standard_normal((1, sk, w.h)) for sk in sizes]
    skip = [rng.standard_normal((1, sk, w.h)) for sk in sizes] if with_skip else None
    fwd = _fwd(w, inp, exact=True, n_gather=0)
    bwd = ob.norm_bwd(dy, fwd["z"], fwd["mask"],
                      fwd["mean64"] if norm == "layernorm" else None,
                      fwd["rstd64"], inp["gamma"], skip, p=w.p, norm=norm, n_gather=w.t)
    # exact backward outputs (recompute unrounded from backward_rows)
    for k in range(w.t):
        one = ob.backward_rows(dy[k][0], fwd["z"][k][0], fwd["mask"][k][0],
                               None if norm != "layernorm" else fwd["mean64"][k][0],
                               fwd["rstd64"][k][0], inp["gamma"],
                               None if skip is None else skip[k][0], p=w.p, norm=norm)
        for j in (0, 3, 15):
            i = (0, 1, j)
            fd_r = _loss_and_grads_fd(w, inp, dy, skip, ("residual", k), i)
            assert one["dz"][1, j] == pytest.approx(fd_r, rel=1e-6, abs=1e-7)
            # every rank's partial receives the same gradient dYpre
            g = sum(sizes[:k]) + 1
            for r in range(w.t):
                fd_p = _loss_and_grads_fd(w, inp, dy, skip, ("partials", r), (0, g, j))
                assert one["dypre_exact"][1, j] == pytest.approx(fd_p, rel=1e-6, abs=1e-7)
    for name, key in (("dgamma", "gamma"), ("dbias", "bias"), ("dbeta", "beta")):
        if bwd[name] is None:
            assert norm == "rmsnorm" and name == "dbeta"
            continue
        for j in (0, 7, 15):
            fd = _loss_and_grads_fd(w, inp, dy, skip, (key,), j)
            assert bwd[name][j] == pytest.approx(fd, rel=1e-6, abs=1e-7), name


@pytest.mark.parametrize("norm", ["layernorm", "rmsnorm"])
def test_backward_matches_torch_autograd(norm):
    w = wl.Workload("ag", t=4, b=1, s=16, h=64, p=0.2, norm=norm, draw_seed=12)
    inp = _inputs(w)
    fwd = _fwd(w, inp, n_gather=0)
    rng = np.random.default_rng(1)
    dy = [rng.standard_normal(z.shape) for z in fwd["z"]]
    bwd = ob.norm_bwd(dy, fwd["z"], fwd["mask"], fwd["mean64"] if norm == "layernorm" else None,
                      fwd["rstd64"], inp["gamma"], None, p=w.p, norm=norm, n_gather=1)
    z = torch.from_numpy(np.concatenate(fwd["z"], axis=1)).double().requires_grad_()
    gamma = torch.from_numpy(inp["gamma"]).double().requires_grad_()
    if norm == "layernorm":
        beta = torch.from_numpy(inp["beta"]).double().requires_grad_()
        out = F.layer_norm(z, (w.h,), gamma, beta, w.eps)
    else:
        out = F.rms_norm(z, (w.h,), gamma, w.eps)
    out.backward(torch.from_numpy(np.concatenate(dy, axis=1)))
    dz = np.concatenate([r for r in bwd["dresidual"]], axis=1)
    np.testing.assert_array_equal(dz, bf16_round(z.grad.numpy()))
    np.testing.assert_allclose(bwd["dgamma"], gamma.grad.numpy(), rtol=1e-10, atol=1e-10)
    if norm == "layernorm":
        np.testing.assert_allclose(bwd["dbeta"], beta.grad.numpy(), rtol=1e-10, atol=1e-10)
    mask = np.concatenate(fwd["mask"], axis=1).astype(np.float64)
    want = bf16_round(z.grad.numpy() * mask * float(ob.dropout_scale(w.p)))
    assert np.array_equal(bwd["dgathered"][0], want)
    np.testing.assert_allclose(bwd["dbias"], (z.grad.numpy() * mask * float(ob.dropout_scale(w.p)))
                               .sum(axis=(0, 1)), rtol=1e-10, atol=1e-10)


# ------------------------------------------------------- unfused boundary --

def test_unfused_equals_fused_when_the_reduced_sum_is_bf16_exact():
    # partials with few significant bits and t = 2: the float32 sum is itself a
    # bf16 number, so rounding it (the unfused path) changes nothing
    w = wl.Workload("u", t=2, b=1, s=16, h=64, draw_seed=13)
    inp = _inputs(w)
    rng = np.random.default_rng(2)
    inp["partials"] = [(rng.integers(-8, 8, size=(1, 16, 64)) / 64).astype(np.float32)
                       for _ in range(2)]
    fused = _fwd(w, inp)
    un = ob.unfused_fwd(inp["partials"], inp["residual"], inp["bias"], inp["gamma"],
                        inp["beta"], eps=w.eps, p=w.p, seed=w.seed)
    for k in range(w.t):
        for key in ("z", "mask", "out"):
            assert np.array_equal(fused[key][k], un[key][k]), key
    assert np.array_equal(fused["gathered"][0], un["gathered"][0])


def test_unfused_differs_from_fused_only_by_rounding_the_sum():
    w = wl.Workload("u2", t=4, b=1, s=32, h=128, p=0.0, draw_seed=14)
    inp = _inputs(w)
    fused = _fwd(w, inp)
    un = ob.unfused_fwd(inp["partials"], inp["residual"], inp["bias"], inp["gamma"],
                        inp["beta"], eps=w.eps, p=w.p, seed=w.seed)
    for k in range(w.t):
        y32 = coll.reduce_scatter_seq(inp["partials"])[0][k]
        # the reduce-scatter output differs from its fp32 value by <= half a bf16 ulp
        assert np.all(np.abs(un["y_shards"][k] - y32) <= np.abs(y32) * 2.0 ** -8 + 1e-30)
        # ... and Z by at most that plus Z's own rounding (a few bf16 ulps of |Z|)
        dz = np.abs(fused["z"][k].astype(np.float64) - un["z"][k])
        assert np.all(dz <= 2.0 ** -7 * np.abs(fused["z"][k]) + 2.0 ** -8 * np.abs(y32) + 1e-30)


# ------------------------------------------- backward entering through g

def test_rs_norm_bwd_is_the_adjoint_of_gather_then_norm():
    """Finite differences: L = sum_r <W_r, gathered O> with each rank's
    column-linear partial gradient W_r; dL/dZ must equal the backward that
    first reduce-scatters the W_r (L7 §3.B: bwd of g is a reduce-scatter)."""
    w = wl.Workload("rb", t=3, b=1, s=9, h=16, p=0.3, draw_seed=15)
    inp = _inputs(w)
    rng = np.random.default_rng(4)
    W = [rng.standard_normal((1, w.s, w.h)) for _ in range(w.t)]

    def loss(res_):
        r = _fwd(w, res_, exact=True, n_gather=0)
        full = np.concatenate(r["out_exact"], axis=1)
        return float(sum((Wr * full).sum() for Wr in W))

    fwd = _fwd(w, inp, exact=True, n_gather=0)
    bwd = ob.rs_norm_bwd(W, fwd["z"], fwd["mask"], fwd["mean64"], fwd["rstd64"], inp["gamma"],
                         None, p=w.p, norm=w.norm, n_gather=1)
    offs = coll.shard_offsets(w.s, w.t)
    for k in range(w.t):
        for i in range(offs[k + 1] - offs[k]):
            for c in (0, 5, 15):
                cp = {kk: ([a.astype(np.float64) for a in v] if isinstance(v, list) else
                           (None if v is None else v.astype(np.float64))) for kk, v in inp.items()}
                cm = {kk: ([a.copy() for a in v] if isinstance(v, list) else
                           (None if v is None else v.copy())) for kk, v in cp.items()}
                cp["residual"][k][0, i, c] += 1e-6
                cm["residual"][k][0, i, c] -= 1e-6
                fd = (loss(cp) - loss(cm)) / 2e-6
                one = ob.backward_rows(bwd["dy_shards"][k][0], fwd["z"][k][0], fwd["mask"][k][0],
                                       fwd["mean64"][k][0], fwd["rstd64"][k][0], inp["gamma"],
                                       None, p=w.p, norm=w.norm)
                assert one["dz"][i, c] == pytest.approx(fd, rel=1e-6, abs=1e-7)


def test_rs_norm_bwd_equals_norm_bwd_on_the_reduced_gradient():
    w = wl.Workload("rb2", t=4, b=2, s=12, h=32, draw_seed=16)
    inp = _inputs(w)
    fwd = _fwd(w, inp, n_gather=0)
    rng = np.random.default_rng(5)
    W = [(np.round(rng.standard_normal((2, 12, 32)) * 64) / 64).astype(np.float32)
         for _ in range(w.t)]
    a = ob.rs_norm_bwd(W, fwd["z"], fwd["mask"], fwd["mean"], fwd["rstd"], inp["gamma"],
                       p=w.p, n_gather=1)
    shards, _ = coll.reduce_scatter_seq(W)
    b = ob.norm_bwd(shards, fwd["z"], fwd["mask"], fwd["mean"], fwd["rstd"], inp["gamma"],
                    p=w.p, n_gather=1)
    for k in range(w.t):
        assert np.array_equal(a["dresidual"][k], b["dresidual"][k])
    assert np.array_equal(a["dgamma"], b["dgamma"]) and np.array_equal(a["dbias"], b["dbias"])
    # (t-1) ranks x b rows x s/t tokens x h x 2 bytes
    assert a["rs_remote_bytes"] == [(w.t - 1) * 2 * (12 // 4) * 32 * 2] * w.t


def test_pack_mask_bits_worked_bytes():
    """Bytes worked out by hand from the layout's definition (channel 8j + e
    in bit e of byte j), then numpy's own bit packing in little-endian bit
    order as an independent routine, and the count of kept elements."""
    rows = np.array([[1, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 1],
                     [1, 1, 0, 1, 0, 0, 0, 0, 1, 1, 1, 1, 1, 1, 1, 1],
                     [0, 0, 0, 0, 0, 0, 0, 0, 0, 1, 0, 1, 0, 1, 0, 1]], dtype=np.uint8)
    got = ob.pack_mask_bits(rows)
    assert got.dtype == np.uint8 and got.shape == (3, 2)
    assert got.tolist() == [[0x01, 0x80], [0x0B, 0xFF], [0x00, 0xAA]]
    rng = np.random.default_rng(3)
    m = (rng.random((2, 5, 64)) < 0.7).astype(np.uint8)
    packed = ob.pack_mask_bits(m)
    assert np.array_equal(packed, np.packbits(m, axis=-1, bitorder="little"))
    assert int(np.unpackbits(packed, axis=-1, bitorder="little").sum()) == int(m.sum())
    with pytest.raises(ValueError):
        ob.pack_mask_bits(np.ones((2, 12), dtype=np.uint8))
