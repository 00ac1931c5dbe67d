"""Length bucketing of packed sequences before the SP boundary (host side).

"分布式训练为什么一开 Sequence Parallel 就开始省显存却抖吞吐" (coreui.cn), section
on shape drift: when long and short samples share a bucket, the sequence
shards of a step carry uneven work and the short ranks wait for the long
ones; its recommended order is to tighten the length buckets first (its
pseudocode calls ``bucket_by_tokens(batch, max_cv=0.15)`` and checks the
bucket's ``length_cv``).  The page gives only the name, the bound and the
purpose; the procedure below is this library's reading:

* ``length_cv`` is the coefficient of variation of the sequence lengths
  (population standard deviation / mean; 0 for one sequence).
* ``bucket_by_tokens`` sorts the sequences by length and walks them in that
  order, closing the current bucket before a sequence that would push its
  length CV above ``max_cv`` or its token count above ``max_tokens``.  Every
  bucket is therefore a run of consecutive lengths in sorted order, each
  sequence lands in exactly one bucket, and a single sequence longer than
  ``max_tokens`` forms a bucket of its own.
* Each bucket carries the int32 ``cu_seqlens`` (prefix sums, leading 0) that
  the boundary's packed, padding-free entry points take, in the bucket's own
  order.
"""
from dataclasses import dataclass
from typing import List, Optional, Sequence

import numpy as np


def length_cv(lengths: Sequence[int]) -> float:
    """Population coefficient of variation of the lengths (0 for <= 1 length)."""
    a = np.asarray(lengths, dtype=np.float64)
    if a.size <= 1 or a.mean() == 0:
        return 0.0
    return float(a.std() / a.mean())


@dataclass(frozen=True)
class Bucket:
    indices: tuple          # positions of the sequences in the input batch
    lengths: tuple          # their lengths, in bucket order
    length_cv: float
    tokens: int

    @property
    def cu_seqlens(self) -> np.ndarray:
        out = np.zeros(len(self.lengths) + 1, dtype=np.int64)
        out[1:] = np.cumsum(self.lengths)
        return out.astype(np.int32)


def bucket_by_tokens(lengths: Sequence[int], max_cv: float = 0.15,
                     max_tokens: Optional[int] = None) -> List[Bucket]:
    """Group sequences into buckets of similar length (see module docstring)."""
    if max_cv < 0:
        raise ValueError("max_cv must be >= 0")
    if max_tokens is not None and max_tokens < 1:
        raise ValueError("max_tokens must be >= 1")
    lens = [int(x) for x in lengths]
    if any(x < 0 for x in lens):
        raise ValueError("lengths must be >= 0")
    order = sorted(range(len(lens)), key=lambda i: (lens[i], i))
    buckets: List[Bucket] = []
    cur: List[int] = []

    def close():
        if cur:
            ls = tuple(lens[i] for i in cur)
            buckets.append(Bucket(tuple(cur), ls, length_cv(ls), sum(ls)))

    for i in order:
        cand = cur + [i]
        ls = [lens[j] for j in cand]
        too_varied = length_cv(ls) > max_cv
        too_big = max_tokens is not None and sum(ls) > max_tokens
        if cur and (too_varied or too_big):
            close()
            cur = [i]
        else:
            cur = cand
    close()
    return buckets
