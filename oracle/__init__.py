"""CPU oracle for one iteration-level batched decode step.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or
executes anything in this package.  The only permitted users are the tests
under ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py``.  The package shares no code with
the CUDA path (no kernels, headers, tables, constants or helpers); the two
meet only through seeded inputs generated elsewhere.

Modules
-------
model      fp64 forward pass of the decoder over contiguous per-sequence KV.
sampler    per-row penalty / temperature / top-k / top-p / inverse-CDF draw,
           and the decayed occurrence counters.
philox     Philox-4x32-10 counter-based generator (Salmon et al., SC'11).
sched_sim  the admission + step-composition policy, in plain Python.

Sources.  The pages describe the method, not the layer maths:
  * "20.3 服务、批处理与流式",
    section 20.3.2 批处理: step cost (W + B*A)/beta, iteration-level
    scheduling, paged KV pool, admission that reserves prompt blocks plus an
    answer budget, prefill chunks first then one row per decoding sequence,
    no eviction; the scaled illustration (4 slots, 4 positions per block,
    8-token chunks, 12 rows per step; Forma: 32 positions, 512-token chunks).
  * "0.8MB 跑通 Qwen 第 14-1 篇", sections 1-3:
    batched decode reads the weights once per step for the whole dynamic set,
    GQA + normalisation workers, and batching leaves outputs byte-identical.
  * "RWKV Runner Albatross 后端", sections
    "适配器" and "Worker 主循环": sampling defaults temperature 1.0,
    top_p 0.3, top_k 0, frequency penalty 1, penalty decay 0.996; batched
    penalty + sampling after the forward.
  The decoder itself (RMSNorm, rotate-half RoPE, GQA attention, SwiGLU, no
  biases, untied embeddings) is the model the benchmark configurations name;
  where the pages are silent the plainest reading is taken and each reading
  is listed in the repository's design notes.

Parity status.  model, sampler and sched_sim are pinned by tests that do
not re-derive them (brute force, closed forms, invariants, hand-worked
examples).  philox is pinned against cuRAND's host Philox-4x32-10 generator
where that library is present; see ``philox`` for the exact claim.
"""
