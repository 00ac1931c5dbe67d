"""Shape trace and memory / communication arithmetic of the SP boundary (test only).

L7 = "第 7 课：序列并行 SP" (hpc.payai.win/train/lesson07.html).

* ``block_shape_trace`` restates the exercise of L7 ("代码填空题"): walk a
  block's regions layernorm -> col_linear -> gelu -> row_linear -> dropout
  and record the (s, h) activation shape after each, marking which entries
  are kept for the backward pass (resident) and which only live in
  communication / temporary buffers (transient).  Under TP+SP, ``g``
  (all-gather along s) precedes the column linear and the row linear's
  full-h output is cut back to s/t tokens by ``g*`` (reduce-scatter along s);
  those full tensors are transient.
* ``peak_resident_bytes`` is the largest resident entry, b*s*h*2 bytes.
* ``non_tp_activation_bytes`` is the part of the per-layer activation
  memory outside the tensor-parallel region, 10*s*b*h bytes (L7
  "具体演示与数值推演": two LayerNorm inputs 4sbh, QKV and MLP-in inputs
  4sbh, two 1-byte dropout masks 2sbh), divided by t under SP.
* ``volume_*`` are the per-rank byte counts of L7 §4 for a ring algorithm.
"""
from dataclasses import dataclass

BF16 = 2


@dataclass(frozen=True)
class TraceEntry:
    region: str
    s: int
    h: int
    resident: bool


def block_shape_trace(seq, hidden, tp, enable_sp):
    """Per-region (s, h) shapes of one block's forward, TP-only or TP+SP."""
    s, h = seq, hidden
    out = []
    # Non-TP region entering the block: TP-only keeps all s tokens; SP keeps
    # its own s/tp tokens (the LayerNorm input is sequence-sharded).
    if enable_sp:
        s = s // tp
    out.append(TraceEntry("layernorm", s, h, True))
    if enable_sp:
        s = s * tp                      # g: all-gather along s
        out.append(TraceEntry("g (all-gather seq)", s, h, False))
    h = h // tp                         # column-parallel linear splits h
    out.append(TraceEntry("col_linear", s, h, True))
    out.append(TraceEntry("gelu", s, h, True))   # element-wise
    h = h * tp                          # row-parallel linear restores h
    if enable_sp:
        # the full-h partial is consumed at once by g*: not resident
        out.append(TraceEntry("row_linear", s, h, False))
        out.append(TraceEntry("row_out (full h)", s, h, False))
        s = s // tp                     # g*: reduce-scatter along s
        out.append(TraceEntry("g* (reduce-scatter seq)", s, h, False))
    else:
        out.append(TraceEntry("row_linear", s, h, True))
    out.append(TraceEntry("dropout", s, h, True))
    return out


def peak_resident_bytes(trace, batch=1):
    """Largest activation kept for the backward pass, in bytes (bf16)."""
    return max(batch * e.s * e.h * BF16 for e in trace if e.resident)


def non_tp_activation_bytes(seq, batch, hidden, tp, sp):
    """Bytes of the per-layer activations outside the TP region.

    Breakdown in bytes: LayerNorm inputs 2 * (2 s b h) + QKV / MLP-in inputs
    2 * (2 s b h) + dropout masks 2 * (1 s b h) = 10 s b h.  Sequence
    parallelism keeps 1/tp of the tokens of each.
    """
    sbh = seq * batch * hidden
    total = 2 * (BF16 * sbh) + 2 * (BF16 * sbh) + 2 * (1 * sbh)
    return total // tp if sp else total


def volume_all_reduce(size_bytes, tp):
    """Per-rank bytes of a ring all-reduce: 2 (t-1)/t * Size (L7 §4)."""
    return 2 * (tp - 1) * size_bytes // tp


def volume_reduce_scatter(size_bytes, tp):
    """Per-rank bytes of a ring reduce-scatter: (t-1)/t * Size (L7 §4)."""
    return (tp - 1) * size_bytes // tp


def volume_all_gather(size_bytes, tp):
    """Per-rank bytes of a ring all-gather: (t-1)/t * Size (L7 §4)."""
    return (tp - 1) * size_bytes // tp


def volume_per_block(batch, seq, hidden, tp, sp):
    """Forward bytes per rank per block: 2 all-reduces (TP) or 2 all-gathers
    plus 2 reduce-scatters (TP+SP), Size = b*s*h*2 (L7 §4)."""
    size = batch * seq * hidden * BF16
    if sp:
        return 2 * (volume_all_gather(size, tp) + volume_reduce_scatter(size, tp))
    return 2 * volume_all_reduce(size, tp)
