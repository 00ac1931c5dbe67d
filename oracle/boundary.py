"""The fused SP boundary, forward and backward, written out plainly (test only).

What one transformer-block boundary computes under tensor + sequence
parallelism with t ranks, following "第 7 课：序列并行 SP"
(hpc.payai.win/train/lesson07.html; cited below as L7):

forward, per rank k (L7 §3.A, the ``g*`` then ``g`` operators):
  1. ``g*`` reduce-scatter along s: Y = sum_r P_r on the tokens of shard k
     (float32, ranks in ascending order; L7 §3.A "一石二鸟").
  2. bias-add: Y += bias (the row-parallel linear's bias, added once after the
     sum; the pages are silent, this is the plainest reading).
  3. dropout: keep = (u >= floor(p * 2**32)) with u the Philox draw of the
     element's global index; D = keep ? Y * scale : 0, scale = f32(1/(1-p))
     (inverted dropout; L7 answer to Q1: one seed for all ranks, masks agree
     and cover the full tensor).  The mask is stored at 1 byte per element
     (L7 "具体演示与数值推演": dropout masks, 1 byte per element).
  4. residual-add: Z = bf16(D + R) in float32 then rounded (L7 §2: residual
     connections live in the non-TP region).
  5. token-wise norm over h of the bf16 values of Z (L7 §2 formula):
     LayerNorm  mu = mean(Z), var = mean((Z - mu)**2) (biased),
                rstd = 1/sqrt(var + eps), O = (Z - mu) * rstd * gamma + beta;
     RMSNorm    rstd = 1/sqrt(mean(Z**2) + eps), O = Z * rstd * gamma
                (L7 names RMSNorm as token-wise but prints no formula; this
                is the standard definition, no mean and no beta).
     Statistics in float64; O rounded once to bf16; mean/rstd stored as
     float32.
  6. ``g`` all-gather along s: every gathered copy holds O of every shard at
     the tokens' own sequence positions (L7 §3.A "前向转入 TP 区域").

backward (L7 §3.B: the adjoint of the forward; bwd(g*) is an all-gather):
  x_hat = (Z - mu) * rstd (LN) or Z * rstd (RMS), from the stored mean/rstd;
  dx_hat = dY * gamma;
  LN  dZ = rstd * (dx_hat - mean(dx_hat) - x_hat * mean(dx_hat * x_hat));
  RMS dZ = rstd * (dx_hat - x_hat * mean(dx_hat * x_hat));
  dZ_tot = dZ + dZ_skip (gradient reaching Z along the skip path, optional);
  dResidual = bf16(dZ_tot);  dYpre = dZ_tot * mask * scale;
  each rank's row-linear partial receives the full-sequence dYpre (bf16):
  the all-gather of the shards' dYpre;
  dgamma = sum_g dY * x_hat, dbeta = sum_g dY, dbias = sum_g dYpre, over all
  tokens of all shards (gamma, beta, bias are replicated on every rank).
"""
import math

import numpy as np

from . import bf16 as _bf16
from . import collectives as _coll
from . import philox as _philox

LAYERNORM = "layernorm"
RMSNORM = "rmsnorm"


def dropout_threshold(p):
    """Integer keep threshold: an element is kept when its draw u >= thr.

    thr = floor(p * 2**32) evaluated in double precision, so that the keep
    decision is an integer comparison with P(drop) = thr / 2**32 ~= p.
    """
    if not (0.0 <= p < 1.0):
        raise ValueError("dropout probability must lie in [0, 1)")
    return int(math.floor(p * 4294967296.0))


def pack_mask_bits(mask):
    """The mask stored one bit per element: (..., h) 0/1 bytes -> (..., h / 8)
    uint8, byte j holding channels [8j, 8j + 8) with channel 8j + e in bit e
    (value 2**e).  The pages keep one byte per element (L7 "具体演示与数值推演");
    this packed layout is one the implementation adds, with the same keep
    decisions, so it is written here from its own definition: the byte is the
    sum of its channels' bits, each shifted to its place.  Requires h % 8 == 0."""
    m = np.asarray(mask)
    h = m.shape[-1]
    if h % 8:
        raise ValueError("h must be a multiple of 8")
    groups = m.reshape(m.shape[:-1] + (h // 8, 8)).astype(np.uint32)
    packed = np.zeros(groups.shape[:-1], dtype=np.uint32)
    for e in range(8):
        packed += (groups[..., e] & 1) << e
    return packed.astype(np.uint8)


def dropout_scale(p):
    """Inverted-dropout scale 1/(1-p), computed in double, stored as float32."""
    return np.float32(1.0 / (1.0 - p))


def _norm_rows(z64, gamma, beta, eps, norm):
    """Token-wise LayerNorm / RMSNorm of rows z64 (n, h), float64 throughout.

    Returns (out, mean, rstd, magnitude) where magnitude = |x_hat * gamma| +
    |beta| is the size of the terms summed into each output (used only to
    bound the rounding error of a float32 evaluation in tests).
    """
    h = z64.shape[-1]
    g64 = np.asarray(gamma, dtype=np.float64)
    if norm == LAYERNORM:
        mu = z64.sum(axis=-1) / h
        centred = z64 - mu[:, None]
        var = (centred * centred).sum(axis=-1) / h
        rstd = 1.0 / np.sqrt(var + eps)
        scaled = centred * rstd[:, None] * g64
        b64 = np.asarray(beta, dtype=np.float64)
        return scaled + b64, mu, rstd, np.abs(scaled) + np.abs(b64)
    if norm == RMSNORM:
        ms = (z64 * z64).sum(axis=-1) / h
        rstd = 1.0 / np.sqrt(ms + eps)
        out = z64 * rstd[:, None] * g64
        return out, None, rstd, np.abs(out)
    raise ValueError(f"unknown norm {norm!r}")


def _after_reduce(y, r_rows, token_index, bias, gamma, beta, *, eps, p, seed,
                  offset, norm, exact):
    """Steps 2-5 on reduced rows y (n, h) of the tokens ``token_index``."""
    n, h = y.shape
    thr = dropout_threshold(p)
    scale = dropout_scale(p)
    elem = (np.asarray(token_index, dtype=np.int64)[:, None] * h
            + np.arange(h, dtype=np.int64)[None, :])
    u = _philox.element_uniforms(seed, offset, elem)
    keep = u.astype(np.int64) >= thr
    if exact:
        y = y + np.asarray(bias, dtype=np.float64)
        d = np.where(keep, y * np.float64(scale), 0.0)
        z = d + np.asarray(r_rows, dtype=np.float64)
        z64 = z
    else:
        y = (y + np.asarray(bias, dtype=np.float32)).astype(np.float32)
        d = np.where(keep, (y * scale).astype(np.float32), np.float32(0.0))
        zf = (d + np.asarray(r_rows, dtype=np.float32)).astype(np.float32)
        z = _bf16.bf16_round(zf)
        z64 = z.astype(np.float64)
    out64, mu, rstd, mag = _norm_rows(z64, gamma, beta, eps, norm)
    return {
        "out_magnitude": mag,
        "z": z,
        "mask": keep.astype(np.uint8),
        "mean": None if mu is None else mu.astype(np.float32),
        "rstd": rstd.astype(np.float32),
        "out": out64 if exact else _bf16.bf16_round(out64),
        "out_exact": out64,
        "mean64": mu,
        "rstd64": rstd,
    }


def forward_rows(partial_rows, residual_rows, token_index, bias, gamma, beta, *,
                 eps, p, seed, offset=0, norm=LAYERNORM, exact=False):
    """Forward of individual tokens, for spot checks at any size.

    partial_rows: (t, n, h) rows of the t partials at the tokens
    ``token_index`` (global index g = batch_row * s + position);
    residual_rows: (n, h).  The reduce is the same float32 rank-ascending sum
    as ``collectives.reduce_scatter_seq``.
    """
    pr = np.asarray(partial_rows)
    if exact:
        y = pr.astype(np.float64).sum(axis=0)
    else:
        y = pr[0].astype(np.float32).copy()
        for r in range(1, pr.shape[0]):
            y = (y + pr[r].astype(np.float32)).astype(np.float32)
    return _after_reduce(y, residual_rows, token_index, bias, gamma, beta,
                         eps=eps, p=p, seed=seed, offset=offset, norm=norm,
                         exact=exact)


def rs_norm_fwd(partials, residual, bias, gamma, beta, *, eps, p, seed,
                offset=0, norm=LAYERNORM, n_gather=1, exact=False):
    """The whole forward boundary over t emulated ranks.

    partials: t arrays (b, s, h); residual: t shard arrays (b, s_k, h).
    Returns per-shard lists z, mask, mean, rstd, out; ``gathered`` (n_gather
    full (b, s, h) copies of O); byte tallies ``rs_remote_bytes`` and
    ``ag_remote_bytes``.
    """
    t = len(partials)
    b, s, h = np.asarray(partials[0]).shape
    offs = _coll.shard_offsets(s, t)
    if exact:
        shards_y = [sum(np.asarray(P[:, offs[k]:offs[k + 1], :], dtype=np.float64)
                        for P in partials) for k in range(t)]
        rs_bytes = None
    else:
        shards_y, rs_bytes = _coll.reduce_scatter_seq(partials)
    res = {"z": [], "mask": [], "mean": [], "rstd": [], "out": [], "out_exact": [],
           "mean64": [], "rstd64": []}
    for k in range(t):
        sk = offs[k + 1] - offs[k]
        tok = (np.arange(b)[:, None] * s + offs[k] + np.arange(sk)[None, :]).reshape(-1)
        y = np.asarray(shards_y[k]).reshape(b * sk, h)
        r_rows = np.asarray(residual[k]).reshape(b * sk, h)
        one = _after_reduce(y, r_rows, tok, bias, gamma, beta, eps=eps, p=p,
                            seed=seed, offset=offset, norm=norm, exact=exact)
        for key in ("z", "mask", "out", "out_exact"):
            res[key].append(one[key].reshape(b, sk, h))
        res["mean"].append(None if one["mean"] is None else one["mean"].reshape(b, sk))
        res["rstd"].append(one["rstd"].reshape(b, sk))
        res["mean64"].append(None if one["mean64"] is None else one["mean64"].reshape(b, sk))
        res["rstd64"].append(one["rstd64"].reshape(b, sk))
    if n_gather > 0:
        gathered, ag_bytes = _coll.all_gather_seq(res["out"], n_gather)
    else:
        gathered, ag_bytes = [], []
    res["gathered"] = gathered
    res["rs_remote_bytes"] = rs_bytes
    res["ag_remote_bytes"] = ag_bytes
    return res


def shard_norm_fwd(y_shards, residual, bias, gamma, beta, *, s, eps, p, seed, offset=0,
                   norm=LAYERNORM):
    """Steps 2-5 on already reduced shards (the unfused boundary's middle step).

    y_shards: t arrays (b, s_k, h) holding each rank's reduce-scatter output
    as the collective delivered it (bf16 values).  Token indices, and hence
    dropout draws, are those of the full sequence.  Returns per-shard lists
    z, mask, mean, rstd, out (O of the shard) and out_exact.
    """
    t = len(y_shards)
    b = np.asarray(y_shards[0]).shape[0]
    h = np.asarray(y_shards[0]).shape[-1]
    offs = _coll.shard_offsets(s, t)
    res = {"z": [], "mask": [], "mean": [], "rstd": [], "out": [], "out_exact": []}
    for k in range(t):
        sk = offs[k + 1] - offs[k]
        tok = (np.arange(b)[:, None] * s + offs[k] + np.arange(sk)[None, :]).reshape(-1)
        one = _after_reduce(np.asarray(y_shards[k], dtype=np.float32).reshape(b * sk, h),
                            np.asarray(residual[k]).reshape(b * sk, h), tok, bias, gamma, beta,
                            eps=eps, p=p, seed=seed, offset=offset, norm=norm, exact=False)
        for key in ("z", "mask", "out", "out_exact"):
            res[key].append(one[key].reshape(b, sk, h))
        res["mean"].append(None if one["mean"] is None else one["mean"].reshape(b, sk))
        res["rstd"].append(one["rstd"].reshape(b, sk))
    return res


def unfused_fwd(partials, residual, bias, gamma, beta, *, eps, p, seed, offset=0,
                norm=LAYERNORM, n_gather=1):
    """The boundary as three separate steps: a bf16 reduce-scatter (the float32
    rank-ascending sum rounded to bf16, as a bf16 collective delivers it), the
    token-wise ops on each shard, then the all-gather of the shards' O."""
    shards_y, rs_bytes = _coll.reduce_scatter_seq(partials)
    y16 = [_bf16.bf16_round(y) for y in shards_y]
    s = np.asarray(partials[0]).shape[1]
    res = shard_norm_fwd(y16, residual, bias, gamma, beta, s=s, eps=eps, p=p, seed=seed,
                         offset=offset, norm=norm)
    res["y_shards"] = y16
    res["gathered"], res["ag_remote_bytes"] = (_coll.all_gather_seq(res["out"], n_gather)
                                               if n_gather > 0 else ([], []))
    res["rs_remote_bytes"] = rs_bytes
    return res


def unsharded_fwd(partials, residual_full, bias, gamma, beta, *, eps, p, seed,
                  offset=0, norm=LAYERNORM):
    """TP-only reference: all-reduce, then the token-wise ops on all tokens.

    This is the path sequence parallelism replaces (L7 §2: every TP rank keeps
    the full (b, s, h)); the sharded result must equal it sliced by token.
    """
    full = _coll.all_reduce(partials)[0]
    b, s, h = full.shape
    tok = np.arange(b * s)
    one = _after_reduce(full.reshape(b * s, h),
                        np.asarray(residual_full).reshape(b * s, h), tok, bias,
                        gamma, beta, eps=eps, p=p, seed=seed, offset=offset,
                        norm=norm, exact=False)
    return {k: (v.reshape(b, s, -1) if (v is not None and v.ndim == 2) else
                (v.reshape(b, s) if v is not None else None))
            for k, v in one.items()}


def backward_rows(dy, z, mask, mean, rstd, gamma, dz_skip=None, *, p,
                  norm=LAYERNORM):
    """Backward of the norm, residual-add and dropout on rows (n, h), float64.

    Inputs are the stored forward values (bf16 Z, uint8 mask, float32
    mean/rstd) and dY, the gradient of the normalised output O.  Returns the
    float64 total gradient of Z, the rounded stored gradients, and the
    per-token terms of the parameter gradients.
    """
    dy64 = np.asarray(dy, dtype=np.float64)
    z64 = np.asarray(z, dtype=np.float64)
    rs = np.asarray(rstd, dtype=np.float64)[:, None]
    g64 = np.asarray(gamma, dtype=np.float64)
    if norm == LAYERNORM:
        xhat = (z64 - np.asarray(mean, dtype=np.float64)[:, None]) * rs
    elif norm == RMSNORM:
        xhat = z64 * rs
    else:
        raise ValueError(f"unknown norm {norm!r}")
    dxhat = dy64 * g64
    h = z64.shape[-1]
    m2 = (dxhat * xhat).sum(axis=-1, keepdims=True) / h
    if norm == LAYERNORM:
        m1 = dxhat.sum(axis=-1, keepdims=True) / h
        dz = rs * (dxhat - m1 - xhat * m2)
        mag = rs * (np.abs(dxhat) + np.abs(m1) + np.abs(xhat * m2))
    else:
        dz = rs * (dxhat - xhat * m2)
        mag = rs * (np.abs(dxhat) + np.abs(xhat * m2))
    if dz_skip is not None:
        dz = dz + np.asarray(dz_skip, dtype=np.float64)
        mag = mag + np.abs(np.asarray(dz_skip, dtype=np.float64))
    scale = np.float64(dropout_scale(p))
    dypre = dz * np.asarray(mask, dtype=np.float64) * scale
    return {
        "dz_magnitude": mag,
        "dz": dz,
        "dresidual": _bf16.bf16_round(dz),
        "dypre_exact": dypre,
        "dypre": _bf16.bf16_round(dypre),
        "dgamma_terms": dy64 * xhat,
        "dbeta_terms": dy64 if norm == LAYERNORM else None,
        "dbias_terms": dypre,
    }


def norm_bwd(dy, z, mask, mean, rstd, gamma, dz_skip=None, *, p,
             norm=LAYERNORM, n_gather=1):
    """The whole backward boundary over t emulated ranks.

    dy, z, mask, rstd (and mean for LN; dz_skip optional): t shard arrays of
    shape (b, s_k, h) / (b, s_k).  Returns per-shard ``dresidual``, the
    gathered full-sequence ``dgathered`` copies (bwd of ``g*`` is an all-gather,
    L7 §3.B), and float64 ``dgamma``, ``dbeta`` (LN), ``dbias`` summed over
    every token of every shard, plus ``*_rss``: the root-sum-square of each
    sum's terms (the natural scale of a sum of mixed-sign terms, used to set
    test tolerances).
    """
    t = len(dy)
    h = np.asarray(dy[0]).shape[-1]
    dres, dypre = [], []
    acc = {"dgamma": np.zeros(h), "dbeta": np.zeros(h), "dbias": np.zeros(h)}
    sq = {"dgamma": np.zeros(h), "dbeta": np.zeros(h), "dbias": np.zeros(h)}
    for k in range(t):
        b, sk, _ = np.asarray(dy[k]).shape
        rows = lambda a: None if a is None else np.asarray(a).reshape(b * sk, -1)
        one = backward_rows(
            rows(dy[k]), rows(z[k]), rows(mask[k]),
            None if mean is None or mean[k] is None else np.asarray(mean[k]).reshape(-1),
            np.asarray(rstd[k]).reshape(-1), gamma,
            None if dz_skip is None or dz_skip[k] is None else rows(dz_skip[k]),
            p=p, norm=norm)
        dres.append(one["dresidual"].reshape(b, sk, h))
        dypre.append(one["dypre"].reshape(b, sk, h))
        for name in ("dgamma", "dbeta", "dbias"):
            terms = one[name + "_terms"]
            if terms is None:
                continue
            acc[name] += terms.sum(axis=0)
            sq[name] += (terms * terms).sum(axis=0)
    gathered, ag_bytes = (_coll.all_gather_seq(dypre, n_gather)
                          if n_gather > 0 else ([], []))
    out = {"dresidual": dres, "dypre": dypre, "dgathered": gathered,
           "ag_remote_bytes": ag_bytes}
    for name in ("dgamma", "dbeta", "dbias"):
        out[name] = None if (name == "dbeta" and norm != LAYERNORM) else acc[name]
        out[name + "_rss"] = np.sqrt(sq[name])
    return out


def rs_norm_bwd(dy_partials, z, mask, mean, rstd, gamma, dz_skip=None, *, p,
                norm=LAYERNORM, n_gather=1):
    """Backward entering through ``g``: the gradient of the all-gather is a
    reduce-scatter along s (L7 §3.B).  Each rank's column-parallel linear
    leaves a partial gradient of the full gathered input, (b, s, h); rank k's
    dY is the float32, rank-ascending sum of those partials on its tokens
    (not rounded: the fused boundary hands it to the norm backward directly),
    then the shard backward of ``norm_bwd`` runs on it."""
    dy_shards, rs_bytes = _coll.reduce_scatter_seq(dy_partials)
    b = np.asarray(dy_partials[0]).shape[0]
    out = norm_bwd([y.reshape(b, -1, y.shape[-1]) for y in dy_shards], z, mask, mean, rstd,
                   gamma, dz_skip, p=p, norm=norm, n_gather=n_gather)
    out["dy_shards"] = dy_shards
    out["rs_remote_bytes"] = rs_bytes
    return out
