"""CPU oracle for the TP+SP ``g*``/``g`` boundary — TEST INFRASTRUCTURE ONLY.

This package is a plain, slow, obviously-correct restatement of what the
sequence-parallel boundary of a transformer block computes.  It exists to be
compared against; it is never part of the product path.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py`` (its ``cpu_baseline`` leg and its
``--impl reference`` arm) may import it.  It shares no code with the CUDA
library: it imports numpy and the standard library only.

Sources (web pages, cited by title and section):

* L7 -- "第 7 课：序列并行 SP" (hpc.payai.win/train/lesson07.html):
  §2 LayerNorm formula; §3 token-wise operators and sequence sharding;
  §3.A the ``g`` (all-gather along s) and ``g*`` (reduce-scatter along s)
  operators; §3.B backward duality; §4 communication-volume theorem;
  "具体演示与数值推演" (70B activation arithmetic); the ``trace_block``
  exercise and its printed result; answers to Q1-Q3; figure 7-3.
* P1 -- "分布式训练为什么一开 Sequence Parallel 就开始省显存却抖吞吐"
  (coreui.cn/article/2565561): ``fused_shard_layernorm`` inside the shard,
  uneven per-rank token counts in mixed-length buckets.

Modules and what pins each one (tests under ``tests/test_oracle_*.py``):

* ``philox``      -- Philox4x32-10 (Salmon et al., SC'11).  Pinned by the
  published known-answer vectors.
* ``bf16``        -- IEEE round-to-nearest-even into bfloat16.  Pinned by
  torch's float32->bfloat16 cast and by brute force over all 65,536 values.
* ``collectives`` -- reduce-scatter / all-gather / all-reduce over rank
  buffers with a byte tally.  Pinned by AllReduce == AllGather(ReduceScatter)
  and by the volume law (t-1)/t * b*s*h*2 of L7 §4.
* ``boundary``    -- the fused forward (sum, bias, dropout, residual,
  LayerNorm/RMSNorm, gather) and its backward.  Pinned by: textbook
  layer_norm / rms_norm (torch, fp64) at t=1, p=0; sharded == unsharded
  sliced by token; gamma=1, beta=0 moments; mask independence of t; drop
  fraction; finite differences and torch autograd for the backward; the
  transpose identity <AG x, y> = <x, RS y>.
* ``accounting``  -- the block shape trace and the activation-memory law.
  Pinned by the printed numbers of L7 (33.6 MB / 4.2 MB; 1.34 GB / 167.8 MB).
* ``compare``     -- the parity checker's tolerance predicates.  Pinned by
  cases each predicate must reject (2 ulps either side and across zero, an
  error above the magnitude floor, 2e-5 on a statistic, a column sum with one
  term dropped, doubled or negated), by the oracle's magnitudes staying tight
  enough that the floor rarely exceeds one ulp, and by a float32 LayerNorm
  passing the bar with few elements accepted through the floor alone.

Parity unpinned: none of the functions above.  (Throughput has no page
figure to pin against; it is measured, not compared.)
"""
