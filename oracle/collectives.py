"""Sequence-dimension collectives over emulated rank buffers (oracle; test only).

The t tensor-parallel ranks are a Python list of t arrays.  Each function
returns its result together with a tally of the bytes that cross from one
rank's buffer into another's, counted element by element as the data moves
(bf16: 2 bytes per element), so that the volume law of L7 §4 can be checked
against what the algorithm actually does rather than against a formula.

L7 = "第 7 课：序列并行 SP" (hpc.payai.win/train/lesson07.html).
"""
import numpy as np

BYTES_PER_ELEMENT = 2   # bf16 activations


def shard_offsets(n, t):
    """Token offsets o_0..o_t of the t sequence shards of an n-token axis.

    L7 §3 splits the sequence evenly into s/t tokens per rank; where t does
    not divide n (packed, mixed-length buckets as in P1's "形状漂移"
    paragraph) the reading is o_k = floor(k*n/t), so shard sizes differ by at
    most one token and no padding is added.
    """
    return [(k * n) // t for k in range(t + 1)]


def reduce_scatter_seq(partials):
    """``g*``: sum the t partials and keep shard k of the sum on rank k.

    L7 §3.A ("前向转出 TP 区域"): after the row-parallel linear every rank holds
    a partial sum of shape (b, s, h); the reduce-scatter along s both adds the
    partials and leaves (b, s/t, h) on each rank.

    The sum is float32, accumulated over ranks in ascending order
    (((P_0 + P_1) + P_2) + ...), the order the boundary's forward pins.

    Returns (shards, remote_bytes) with remote_bytes[k] = bytes rank k
    received from the other ranks.
    """
    t = len(partials)
    b, s, h = partials[0].shape
    offs = shard_offsets(s, t)
    shards, remote = [], []
    for k in range(t):
        lo, hi = offs[k], offs[k + 1]
        acc = None
        received = 0
        for r in range(t):
            piece = np.asarray(partials[r][:, lo:hi, :], dtype=np.float32)
            if r != k:
                received += piece.size * BYTES_PER_ELEMENT
            acc = piece.copy() if acc is None else (acc + piece).astype(np.float32)
        shards.append(acc)
        remote.append(received)
    return shards, remote


def all_gather_seq(shards, n_gather=None):
    """``g``: concatenate the t sequence shards into full (b, s, h) buffers.

    L7 §3.A ("前向转入 TP 区域"): (b, s/t, h) -> (b, s, h) before the
    column-parallel linear.  ``n_gather`` full copies are produced (rank j's
    copy for j < n_gather; default t).  Returns (copies, remote_bytes) with
    remote_bytes[j] = bytes written into copy j from shards k != j.
    """
    t = len(shards)
    n_gather = t if n_gather is None else n_gather
    copies, remote = [], []
    for j in range(n_gather):
        parts = []
        received = 0
        for k in range(t):
            parts.append(np.array(shards[k], copy=True))
            if k != j:
                received += np.asarray(shards[k]).size * BYTES_PER_ELEMENT
        copies.append(np.concatenate(parts, axis=1))
        remote.append(received)
    return copies, remote


def all_reduce(partials):
    """TP-only ``f*``: every rank ends with the full elementwise sum.

    By definition: each rank's result is the float32 sum over ranks in
    ascending order of the whole (b, s, h) partials (the same order as
    ``reduce_scatter_seq``).  Used only to check the ring identity of L7 §4,
    AllReduce(X) == AllGather(ReduceScatter(X)).
    """
    acc = np.asarray(partials[0], dtype=np.float32).copy()
    for r in range(1, len(partials)):
        acc = (acc + np.asarray(partials[r], dtype=np.float32)).astype(np.float32)
    return [acc.copy() for _ in partials]


def sum_seq_shards(full, t):
    """Transpose of ``all_gather_seq`` for the identity <AG x, y> = <x, RS y>.

    Given t full (b, s, h) arrays y_j, rank k's result is the float64 sum over
    j of y_j restricted to shard k (L7 §3.B: the backward of an all-gather
    along s is a reduce-scatter along s).
    """
    b, s, h = full[0].shape
    offs = shard_offsets(s, t)
    out = []
    for k in range(t):
        lo, hi = offs[k], offs[k + 1]
        acc = np.zeros((b, hi - lo, h), dtype=np.float64)
        for y in full:
            acc += np.asarray(y[:, lo:hi, :], dtype=np.float64)
        out.append(acc)
    return out
