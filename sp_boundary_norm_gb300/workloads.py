"""Seeded synthetic workloads for the SP boundary (shapes, distributions only).

This module draws inputs; it holds none of the boundary's arithmetic, so both
the CUDA path and the CPU oracle can be fed from it.  The shapes are the ones
the lesson works with ("第 7 课：序列并行 SP": the trace exercise at
s = h = 4096, t = 8; the 70B example at h = 8192, s = 16384, t = 8) plus a
small case and a packed, length-bucketed case of mixed sequence lengths (the
uneven per-rank token counts discussed in "分布式训练为什么一开 Sequence
Parallel 就开始省显存却抖吞吐").

Distributions (all drawn in float32, then rounded to bf16 by torch's
round-to-nearest-even cast): partials N(0, 0.02^2) each, residual N(0, 1),
bias N(0, 0.01^2), gamma 1 + N(0, 0.1^2), beta N(0, 0.1^2), upstream
gradient dY N(0, 1).
"""
from dataclasses import dataclass, field, replace

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    t: int
    b: int
    s: int                      # tokens per batch row (packed total when ragged)
    h: int
    eps: float = 1e-5
    p: float = 0.1
    seed: int = 1234            # dropout seed
    offset: int = 0             # dropout counter offset
    norm: str = "layernorm"
    n_gather: int = 1
    seqlens: tuple = field(default=())   # packed sequence lengths (b == 1)
    draw_seed: int = 0          # seed of the input draws

    @property
    def tokens(self):
        return self.b * self.s

    @property
    def ragged(self):
        return len(self.seqlens) > 0

    def shard_sizes(self):
        """Tokens per shard along s: o_k = floor(k*s/t)."""
        o = [(k * self.s) // self.t for k in range(self.t + 1)]
        return [o[k + 1] - o[k] for k in range(self.t)]

    def with_(self, **kw):
        return replace(self, **kw)


def ragged_lengths(n_seqs=8, median=4096, sigma=0.6, lo=512, hi=32768, seed=0):
    """Sequence lengths rint(lognormal(ln median, sigma)) clipped to [lo, hi]."""
    rng = np.random.default_rng(seed)
    raw = rng.lognormal(np.log(median), sigma, size=n_seqs)
    return tuple(int(x) for x in np.clip(np.rint(raw), lo, hi))


def cu_seqlens(lengths):
    """Prefix sums [0, l0, l0+l1, ...] as int32."""
    out = np.zeros(len(lengths) + 1, dtype=np.int64)
    out[1:] = np.cumsum(lengths)
    return out.astype(np.int32)


_RAGGED = ragged_lengths()

WORKLOADS = {
    "tiny": Workload("tiny", t=2, b=1, s=256, h=512, draw_seed=0),
    "trace4k": Workload("trace4k", t=8, b=1, s=4096, h=4096, draw_seed=1),
    "ragged": Workload("ragged", t=8, b=1, s=int(sum(_RAGGED)), h=5120,
                       seqlens=_RAGGED, draw_seed=2),
    "70b": Workload("70b", t=8, b=1, s=16384, h=8192, draw_seed=3),
    "bwd70b": Workload("bwd70b", t=8, b=1, s=16384, h=8192, draw_seed=4),
    "bwd70b_rms": Workload("bwd70b_rms", t=8, b=1, s=16384, h=8192, eps=1e-6,
                           norm="rmsnorm", draw_seed=4),
}


def _normal(shape, std, gen, device, mean=0.0):
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    if mean != 0.0:
        x.add_(mean)
    return x.to(torch.bfloat16)


def make_generator(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def forward_inputs(w, device="cpu", seed=None):
    """t partials (b, s, h); t residual shards (b, s_k, h); bias, gamma, beta (h)."""
    gen = make_generator(w.draw_seed if seed is None else seed, device)
    partials = [_normal((w.b, w.s, w.h), 0.02, gen, device) for _ in range(w.t)]
    residual = [_normal((w.b, sk, w.h), 1.0, gen, device) for sk in w.shard_sizes()]
    bias = _normal((w.h,), 0.01, gen, device)
    gamma = _normal((w.h,), 0.1, gen, device, mean=1.0)
    beta = _normal((w.h,), 0.1, gen, device)
    if w.norm == "rmsnorm":
        beta = None
    return {"partials": partials, "residual": residual, "bias": bias,
            "gamma": gamma, "beta": beta}


def backward_inputs(w, device="cpu", seed=None, with_skip=False):
    """dY on each shard (b, s_k, h) ~ N(0, 1); optional skip-path gradient."""
    gen = make_generator((w.draw_seed if seed is None else seed) + 1000, device)
    dy = [_normal((w.b, sk, w.h), 1.0, gen, device) for sk in w.shard_sizes()]
    skip = ([_normal((w.b, sk, w.h), 1.0, gen, device) for sk in w.shard_sizes()]
            if with_skip else None)
    return {"dy": dy, "dz_skip": skip}


def regroup_packed(w, order, lengths, partials, shards):
    """The sequences ``order`` of a packed workload (b = 1), laid out as a
    packed batch of their own: what a data loader hands the boundary after
    it has bucketed the batch by length.

    ``partials`` are the t full (1, T, h) partials; ``shards`` any number of
    sharded tensor lists (residual, dY, ...) of the original workload.
    Returns the regrouped workload (its s = the bucket's tokens, its
    ``seqlens`` = the sequences' lengths in bucket order), its t partials and
    each shard list re-cut at the new workload's shard offsets.  Values are
    moved, never computed."""
    if w.b != 1 or not w.ragged:
        raise ValueError("regrouping needs a packed workload (b == 1, seqlens)")
    cu = [0]
    for n in w.seqlens:
        cu.append(cu[-1] + int(n))
    for i, n in zip(order, lengths):
        if cu[i + 1] - cu[i] != int(n):
            raise ValueError(f"sequence {i} has {cu[i + 1] - cu[i]} tokens, not {n}")

    def pick(full):
        return torch.cat([full[:, cu[i]:cu[i + 1]] for i in order], dim=1).contiguous()

    wb = w.with_(s=int(sum(int(n) for n in lengths)), seqlens=tuple(int(n) for n in lengths))
    parts = [pick(P) for P in partials]
    out = []
    for lst in shards:
        full = pick(torch.cat(list(lst), dim=1))
        o = [(k * wb.s) // wb.t for k in range(wb.t + 1)]
        out.append([full[:, o[k]:o[k + 1]].contiguous() for k in range(wb.t)])
    return wb, parts, out
