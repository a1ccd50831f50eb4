/*
 * cbd.h -- C ABI of libcbd: one iteration-level ("continuous") batched step
 * of a decoder-only GQA transformer on one GB300 (sm_103a).
 *
 * The method, as the pages state it:
 *   - "20.3 服务、批处理与流式",
 *     section 20.3.2 批处理: a decode step reads every weight once for the
 *     whole batch, costing about (W + B*A)/beta; scheduling is per model
 *     iteration, so requests join and leave every step; KV lives in a pool
 *     of fixed-size blocks shared by all slots (Forma: 32 positions per
 *     block, 512-token prefill chunks); admission reserves blocks for the
 *     prompt plus part of the answer, because admitting on a free slot alone
 *     can exhaust the pool with no sequence able to finish; each step runs
 *     prefill chunks first, then one row per decoding sequence, and rows
 *     that do not fit wait instead of being evicted; the Scheduler (what to
 *     run) is kept apart from the Batch (running it).
 *   - "0.8MB 跑通 Qwen 第 14-1 篇", sections 1-3: the
 *     rows of one step form a dynamic set whose KV is indexed per request,
 *     computed by batched GQA / normalisation workers; batched and serial
 *     runs gave byte-identical greedy outputs (near ties aside).
 *   - "RWKV Runner Albatross 后端", sections
 *     "适配器" and "Worker 主循环": per-slot sampling parameters held on the
 *     device (temperature, top_p, top_k, presence / frequency penalty with
 *     decay 0.996), applied to every row of the batch after the forward.
 *
 * Conventions for every function:
 *   - Returns a cbd_status (int32): CBD_OK == 0, negative on failure.  On
 *     failure cbd_last_error() returns a message for the calling thread.
 *   - No function aborts the process, throws across the ABI or traps the GPU.
 *   - "host" pointers are ordinary CPU memory, read during the call only;
 *     "device" pointers are CUDA global memory of the engine's device.
 *   - Calls that take a `stream` (a cudaStream_t passed as void*, NULL for
 *     the legacy default stream) are stream-ordered: they enqueue work and
 *     return; outputs are valid once the stream reaches that point.
 *   - An engine, its pools and its batches belong to one device and must be
 *     used from one host thread at a time.
 *   - Everything libcbd allocates it frees in the matching _destroy call.
 */
#ifndef CBD_H
#define CBD_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------ status */
#define CBD_OK 0
#define CBD_EINVAL (-1)        /* an argument or an input row is invalid      */
#define CBD_ENOMEM (-2)        /* device or host allocation failed            */
#define CBD_ECUDA (-3)         /* a CUDA runtime/driver call failed           */
#define CBD_EPOOL (-4)         /* request can never fit the KV pool           */
#define CBD_EUNSUPPORTED (-5)  /* shape or device not supported               */
#define CBD_EDEVICE (-6)       /* a kernel flagged an error (cbd_engine_check) */
#define CBD_EDEADLOCK (-7)     /* scheduler: no running sequence can progress */
#define CBD_ESTATE (-8)        /* call out of order (e.g. commit w/o plan)    */
#define CBD_EBUSY (-9)         /* admission queue full: retry later (HTTP 429) */

typedef int32_t cbd_status;

/* Message of the last failing call on this thread ("" if none).  The
 * pointer stays valid until the thread's next libcbd call. */
const char* cbd_last_error(void);

/* Library version string, e.g. "cbd 0.1 sm_103a". */
const char* cbd_version(void);

/* ------------------------------------------------------------ model */
/* Shape of the decoder.  Block size is fixed at 32 positions (Forma's
 * constant, "20.3 服务、批处理与流式" section 20.3.2). */
typedef struct cbd_config {
  int32_t n_layers;           /* L                                          */
  int32_t d_model;            /* d, multiple of 64                          */
  int32_t n_heads;            /* H_q                                        */
  int32_t n_kv_heads;         /* H_kv, divides H_q                          */
  int32_t head_dim;           /* hd, 64 or 128                              */
  int32_t ffn_dim;            /* F, multiple of 64                          */
  int32_t vocab;              /* V, <= 65536                                */
  float rope_base;            /* RoPE base (10000)                          */
  float rms_eps;              /* RMSNorm epsilon (1e-6)                     */
  int32_t block_size;         /* must be 32                                 */
  int32_t max_rows;           /* rows per step (decode + prefill), <= 4096  */
  int32_t max_slots;          /* sequence slots (penalty counters per slot) */
  int32_t max_blocks_per_seq; /* block-table width; max positions / 32      */
  int32_t kv_fp8;             /* 0: bf16 K/V; 1: FP8 E4M3 K/V ("大模型推理为什么需要
                               * Continuous Batching" section 6), rounded to
                               * nearest even and saturated at +-448, no
                               * scale; half the pool bytes per position.
                               * Needs attention path 0. */
  int32_t weights_int8;       /* 0: the streamed weights stay bf16; 1: int8
                               * weights ("RWKV Runner Albatross 后端",
                               * 边界与后续路线: int8-quantised weights as
                               * follow-up work).  Every matrix the step
                               * streams (q, k, v, o, gate, up, down, LM head)
                               * is quantised per output row when the engine
                               * is created: s = fp32(max|w| / 127), q =
                               * nearest integer to w / s (ties to even; the
                               * quotient in fp64), clamped to +-127; the step
                               * computes s * sum(q * a), fp32 accumulation.
                               * The embedding and the norm gains stay as
                               * given.  Half the weight bytes per step.  Needs
                               * gemm path 0 or 2 (tensor cores). */
} cbd_config;

/* Weights of one layer: bf16, row-major [out][in], no biases. */
typedef struct cbd_layer_weights {
  const void* attn_norm;  /* [d]                  RMSNorm gain before attention */
  const void* wq;         /* [H_q*hd][d]                                        */
  const void* wk;         /* [H_kv*hd][d]                                       */
  const void* wv;         /* [H_kv*hd][d]                                       */
  const void* wo;         /* [d][H_q*hd]                                        */
  const void* ffn_norm;   /* [d]                  RMSNorm gain before the FFN   */
  const void* w_gate;     /* [F][d]                                             */
  const void* w_up;       /* [F][d]                                             */
  const void* w_down;     /* [d][F]                                             */
} cbd_layer_weights;

typedef struct cbd_weights {
  int32_t on_device;                 /* 1: pointers are device memory; 0: host */
  const void* embed;                 /* [V][d] bf16 (untied from lm_head)      */
  const void* final_norm;            /* [d] bf16                               */
  const void* lm_head;               /* [V][d] bf16                            */
  const cbd_layer_weights* layers;   /* host array of n_layers structs         */
} cbd_weights;

typedef struct cbd_engine cbd_engine;
typedef struct cbd_kv_pool cbd_kv_pool;
typedef struct cbd_batch cbd_batch;

/* Create an engine on the current CUDA device: the weights that every step
 * reads once for all of its rows ("20.3 服务、批处理与流式" section 20.3.2: a
 * decode step costs (W + B*A)/beta, W being streamed once per step whatever
 * B is; "0.8MB 跑通 Qwen 第 14-1 篇" section 1: the weights are read once per
 * step for the whole batch), the Batch executor's state that is separate
 * from the Scheduler (same section of the Forma page), and the per-slot
 * device state of the Albatross worker ("RWKV Runner Albatross 后端",
 * section 连续批处理：Worker 主循环: occurrence counters for the penalties,
 * one row per slot).  The weights are copied and repacked into an
 * engine-owned device arena (row orders chosen for the kernels'
 * epilogues); the caller may free its buffers when this returns.  Also
 * allocates the step's activations, workspaces and the per-slot penalty
 * counters ([max_slots][V] fp32, zero).  Every later call on the engine,
 * its pools and batches runs on this device, whichever device is current
 * in the calling thread.  Errors: CBD_EINVAL (shape), CBD_EUNSUPPORTED (not
 * an sm_103 device, or a shape the kernels do not cover), CBD_ENOMEM,
 * CBD_ECUDA.  *out is NULL on failure. */
cbd_status cbd_engine_create(const cbd_config* cfg, const cbd_weights* w, cbd_engine** out);
cbd_status cbd_engine_destroy(cbd_engine* e);

/* Synchronise the device and report a kernel-detected error: CBD_OK, or
 * CBD_EDEVICE with the recorded code (a bounded wait that ran out, an index
 * a kernel refused) in the message; the error word is then cleared. */
cbd_status cbd_engine_check(cbd_engine* e);

/* Failure path of the step's kernels, exercised on purpose: every pipeline
 * wait in them (TMA stages, MMA completion, accumulator hand-over) is an
 * mbarrier wait that gives up after about 2^31 SM cycles, records
 * kDevWaitTimeout (code 3) in the engine's error word and lets its kernel
 * wind down instead of hanging the device.  This call launches one
 * single-warp kernel on `stream` that runs that same wait, with a limit of
 * limit_cycles (1 .. 2^31), on a shared-memory barrier that nothing
 * completes -- no copy in flight, no tensor memory, no other CTA involved --
 * so the wait runs out and the kernel returns.  cbd_engine_check then
 * reports CBD_EDEVICE with code 3 and clears the word; the engine stays
 * usable.  For tests of the failure path.  CBD_EINVAL for a limit outside
 * the range. */
cbd_status cbd_engine_test_wait_timeout(cbd_engine* e, int64_t limit_cycles, void* stream);

/* Choose how the step's weight contractions run: path 0 = automatic (the
 * CUDA-core GEMV for up to gemv_max_rows rows, tcgen05 tensor cores above),
 * 1 = always the CUDA-core GEMV, 2 = always tcgen05.  Both paths compute
 * the same sums (fp32 accumulation of bf16 weights times hi + lo bf16
 * activations); they differ only in summation order.  Default: 0 and 0
 * (tcgen05 from one row: it streams a 7B step's weights in 3.47 ms at
 * B = 1, the GEMV in 8.67 ms). */
cbd_status cbd_engine_set_gemm_path(cbd_engine* e, int32_t path, int32_t gemv_max_rows);

/* Attention of prefill runs (at least 16 rows of one slot at consecutive
 * positions, wherever they sit in the step's row array: a prompt chunk,
 * "20.3 服务、批处理与流式" section 20.3.2) on a kernel that takes blocks of
 * consecutive query positions and streams each K/V block once per block of
 * queries, instead of once per row.  Applies to attention path 0, bf16 or
 * FP8 K/V; the other rows keep the streaming kernel.  Same arithmetic (q and
 * P split into hi + lo halves: bf16, or f16 over E4M3 K/V), summed in
 * another order.  enable != 0: on (the default). */
cbd_status cbd_engine_set_prefill_attention(cbd_engine* e, int32_t enable);

/* On the tcgen05 path, steps of at least min_rows rows (prefill chunks,
 * "20.3 服务、批处理与流式" section 20.3.2) may run their weight
 * contractions on a persistent kernel with 128-row activation tiles: each
 * weight tile feeds 128 rows per pass instead of 64, and two TMEM
 * accumulators overlap one tile's epilogue with the next tile's mainloop;
 * such a step runs the RMSNorm as its own kernel.  With
 * force == 0 a GEMM takes this kernel only where its weights are tiled 128
 * rows wide and its units fill at least 0.6 of the last wave of resident
 * CTAs (else the 64-row-tile kernel, which takes two row tiles per CTA,
 * splits K and, past 128 rows, pairs 128-row weight tiles into 256-wide
 * units: 16.04 ms at 544 rows, where this kernel's 80 units fill 0.53 of
 * the GPU, against 17.66 ms with it); with force != 0 every GEMM of the
 * step takes it.  Same sums as
 * the other paths, in another order.  min_rows 0 = never.  Default 256
 * (7B shape on GB300, both kernels copying one activation box per 64 rows:
 * 12.37 vs 12.45 ms at 288 rows and 17.59 vs 18.58 ms at 544 rows against
 * the 64-row-tile kernel with the fused RMSNorm; 9.11 vs 8.96 ms the other
 * way at 160 rows; 42.82 vs 48.11 ms at 2080 rows against the 64-row-tile
 * kernel everywhere), force 0.  CBD_EINVAL if min_rows < 0. */
cbd_status cbd_engine_set_rows_gemm(cbd_engine* e, int32_t min_rows, int32_t force);

/* Choose the attention kernel: 0 = persistent streaming kernel (each warp
 * pipelines its chunks' K/V tiles through a TMA ring; mma.sync; default),
 * 1 = CUDA cores, 2 = one CTA per chunk with mma.sync.  All use the same
 * 128-position chunks and the same merge order. */
cbd_status cbd_engine_set_attention_path(cbd_engine* e, int32_t path);

/* Forbidden tokens (the Albatross worker masks them before the penalties,
 * "RWKV Runner Albatross 后端", section 连续批处理：Worker 主循环, step 6):
 * token ids that the sampler of cbd_step, cbd_batch_run and cbd_sample
 * never draws -- as if their logits were -inf before the penalty, so they
 * carry no probability mass and greedy rows skip them.  The returned logits
 * stay raw.  ids: host [n], 0 <= id < vocab, copied; n == 0 clears the mask;
 * at least one id must stay allowed.  Waits for the device to be idle, so
 * every step launched afterwards sees the new mask.  cbd_sample_static does
 * not apply it. */
cbd_status cbd_engine_set_forbidden(cbd_engine* e, const int32_t* ids, int32_t n);

/* RMSNorm fused into the weight contractions (default on): on the tcgen05
 * path the embedding and the residual epilogues write the next norm's input
 * x * g (hi + lo bf16) and per-row partial sums of x^2, and the QKV and
 * gate/up contractions multiply their sums by 1/sqrt(mean(x^2) + eps),
 * which is RMSNorm(x) W^T with no separate normalisation launch.  Off (0),
 * or on the CUDA-core GEMV path, a normalisation kernel runs before each of
 * those contractions.  The two agree to rounding (they round the
 * activations at different points).  Errors: CBD_EINVAL for a NULL engine. */
cbd_status cbd_engine_set_fused_norm(cbd_engine* e, int32_t enable);

/* Decode steps as persistent contraction chains (default off): on the
 * tcgen05 path with the fused RMSNorm, bf16 weights and at most 64 rows,
 * each layer's O, gate/up and down contractions and the next layer's QKV
 * run as the phases of one launch, separated by grid-wide barriers instead
 * of kernel boundaries, so each phase's first weight tiles stream while the
 * previous phase's epilogue runs ("20.3 服务、批处理与流式", 20.3.2: a decode
 * step costs (W + B*A)/beta, the time between weight streams is overhead).
 * Every phase keeps the per-launch kernel's tiles, K split and epilogue:
 * results are bit-identical with the setting on or off.  Shapes the chain
 * does not cover (another tile width or K split, more CTAs than fit on the
 * GPU at once) take the per-launch kernels.  enable != 0: on.  Off by
 * default: on GB300 (7B shape, 32 rows) the chained step measured 5.43 ms
 * against 4.73 ms launch by launch -- each phase boundary still costs ~10 us
 * (the slowest CTA's tail, the exchange of partial sums and the grid
 * barrier), and CTAs held to the end of the chain keep the next attention
 * launch from starting early on their SMs.  cbd_engine_set_l2_prefetch also
 * applies inside the chain (each phase's weights beyond the staged tiles).
 * Errors: CBD_EINVAL for a NULL engine. */
cbd_status cbd_engine_set_gemm_chain(cbd_engine* e, int32_t enable);

/* L2 prefetch across kernel boundaries: once a kernel of the step has issued
 * its last load, it asks L2 to fetch the first k-blocks of the next weight
 * contraction's work units, up to `bytes` in all, so HBM could keep
 * streaming while one launch drains and the next starts ("20.3 服务、批处理
 * 与流式", 20.3.2: a decode step costs (W + B*A)/beta).  Default 0 (off):
 * on GB300 the prefetched lines were largely not found by the next kernel's
 * copies, so the prefetch added DRAM reads and slowed the 7B step (5.11 ms
 * off, 5.20 ms at 16 MiB, 5.33 ms at 48 MiB).  A prefetch is a cache hint
 * only: results are identical with any setting.
 * Errors: CBD_EINVAL for a NULL engine or more than 1 GiB. */
cbd_status cbd_engine_set_l2_prefetch(cbd_engine* e, uint64_t bytes);

/* The engine's copy of one streamed weight matrix, for inspection and
 * tests: which = 0 (q, k and v rows as the QKV contraction holds them: per
 * head of q and then of k, output dims in the order 0, hd/2, 1, hd/2+1, ...,
 * so each RoPE pair is adjacent; then v in its own order), 1 (o), 2 (gate
 * and up interleaved: gate row i, up row i, gate row i+1, ...), 3 (down),
 * 4 (LM head; layer ignored).  dst (host): the matrix row-major in that row
 * order, [M][K] -- bf16 for a bf16 engine, int8 for an int8 engine; scales
 * (host, nullable): [M] fp32 per-row scales of an int8 engine.  Synchronous.
 * CBD_EINVAL for a bad index. */
cbd_status cbd_engine_read_weight(cbd_engine* e, int32_t which, int32_t layer, void* dst, float* scales);

/* Device pointer of the per-slot occurrence counters, [max_slots][V] fp32,
 * owned by the engine (for inspection and for seeding tests). */
cbd_status cbd_engine_counters(cbd_engine* e, float** counters);

/* Per-kernel timing.  cbd_engine_profile(e, 1) clears the record and makes
 * every later launch of this engine bracket itself with CUDA events on its
 * own stream; cbd_engine_profile(e, 0) stops recording.  cbd_engine_profile_read
 * synchronises the device and writes up to `cap` per-kernel-class totals
 * (name, launches, summed event time) to `out`, *n = classes recorded.
 * Profiling serialises nothing but adds one event pair per launch. */
typedef struct cbd_kernel_stat {
  char name[32];
  int64_t launches;
  double total_ms;
} cbd_kernel_stat;
cbd_status cbd_engine_profile(cbd_engine* e, int32_t enable);
cbd_status cbd_engine_profile_read(cbd_engine* e, cbd_kernel_stat* out, int32_t cap, int32_t* n);

/* Zero slot `slot`'s occurrence counters and its last sampled token
 * (CBD_TOKEN_LAST): a request was admitted to the slot, and its penalty
 * state starts empty ("RWKV Runner Albatross 后端", section 连续批处理：Worker
 * 主循环: the per-slot penalty state belongs to the request occupying the
 * slot; "20.3 服务、批处理与流式" section 20.3.2: sequences join the batch at
 * any iteration).  Stream-ordered on `stream`; CBD_EINVAL for a slot outside
 * [0, max_slots). */
cbd_status cbd_slot_reset(cbd_engine* e, int32_t slot, void* stream);

/* ------------------------------------------------------------ KV pool */
/* Paged KV pool ("20.3 服务、批处理与流式" section 20.3.2: fixed-size blocks
 * allocated on demand; Forma: 32 positions per block).  Layout, bf16:
 *     pool[L][n_blocks][H_kv][2][tile]     (index 0 = K, 1 = V)
 * where a tile holds 32 positions x hd dims in 128-byte-swizzled order:
 * element (position r, dim d) sits at
 *     (d / 64) * 2048 + r * 64 + (((d % 64) / 8) XOR (r % 8)) * 8 + d % 8.
 * So K and V of one (layer, block, KV head) are one contiguous
 * 2 * 32 * hd * 2-byte run.  The pool is owned by libcbd; its contents
 * start undefined. */
cbd_status cbd_kv_pool_create(cbd_engine* e, int32_t n_blocks, cbd_kv_pool** out);
cbd_status cbd_kv_pool_destroy(cbd_kv_pool* p);

/* Base device pointer and size in bytes of the pool (layout above). */
cbd_status cbd_kv_pool_data(cbd_kv_pool* p, void** base, uint64_t* bytes, int32_t* n_blocks);

/* ------------------------------------------------------------ step */
/* One row of a step.  A decode row feeds the request's last token at
 * position pos = number of cached positions; a prefill row feeds prompt
 * token `token` at position pos.  Every row writes its K/V at (slot, pos)
 * and attends causally over positions 0..pos of its slot, so a prefill row
 * sees the earlier rows of its own chunk.  sample != 0 marks rows whose
 * logits are produced and sampled (every decode row; the last row of a
 * prefill chunk that completes its prompt). */
/* cbd_row.token of a decode row may be CBD_TOKEN_LAST: the token that this
 * engine's sampler last drew for the row's slot (cbd_step, cbd_batch_run or
 * cbd_sample, in stream order; 0 after engine creation or cbd_slot_reset),
 * read on the device.  A decode loop can then enqueue step k + 1 before step
 * k's tokens reach the host ("20.3 服务、批处理与流式" 20.3.2: the next
 * iteration's inputs are the previous iteration's outputs), reading each
 * step's tokens back asynchronously.  Not allowed on prefill rows. */
#define CBD_TOKEN_LAST (-1)

typedef struct cbd_row {
  int32_t slot;
  int32_t token;
  int32_t pos;
  int32_t is_prefill;
  int32_t sample;
} cbd_row;

/* Per sampled row.  Order (Albatross "Worker 主循环" lists the parameters;
 * the order is this library's reading): penalty
 *   l' = (l - presence*[cnt>0]) - frequency*cnt   (fp32, no fused multiply-add)
 * then greedy argmax (ties to the lowest id) if temperature == 0 or
 * top_k == 1; else z = l'/temperature, top-k (k > 0) by (z desc, id asc),
 * top-p: shortest prefix by (p desc, id asc) with mass >= top_p, then the
 * first id in ascending order whose cumulative kept mass exceeds u * total.
 * Afterwards cnt[slot][:] *= penalty_decay; cnt[slot][token] += 1.
 * u = (Philox4x32-10(ctr=(token_index, request_id lo, request_id hi, 0),
 *                    key=(seed lo, seed hi)).x >> 8) * 2^-24. */
typedef struct cbd_sampling {
  float temperature;
  float top_p;
  int32_t top_k;
  float presence_penalty;
  float frequency_penalty;
  float penalty_decay;
  uint64_t seed;
  uint64_t request_id;
  uint32_t token_index;   /* index of the token being generated in its request */
  uint32_t reserved;      /* must be 0 */
} cbd_sampling;

/* Run one batched step on `stream`: one model iteration over the step's
 * row set -- the Batch executing what the Scheduler decided ("20.3 服务、批
 * 处理与流式" section 20.3.2: iteration-level scheduling, requests join and
 * leave between iterations; every row reads its own KV through its slot's
 * block table in the shared pool; prefill chunks and decode rows in one
 * step), with every weight read once for all rows and per-row attention
 * over each request's own KV ("0.8MB 跑通 Qwen 第 14-1 篇" sections 1-2),
 * then the per-row penalties and batched sampling ("RWKV Runner Albatross
 * 后端", section 连续批处理：Worker 主循环).
 *   rows [n_rows] (host): the step's row set, any order, 1 <= n_rows <= max_rows.
 *   block_tables (host): [table_slots][max_blocks_per_seq] int32, row s maps
 *     slot s's logical block b to a physical pool block; entries past
 *     n_blocks_per_slot[s] are ignored.  Every row's slot must be < table_slots.
 *   n_blocks_per_slot (host): [table_slots].
 *   sampling (host): one entry per row with sample != 0, in row order (m of them).
 *   uniforms (host, nullable): m values in [0,1) that replace the Philox draw.
 *   out_tokens (device): [m] int32 sampled token ids.
 *   out_logits (device, nullable, 16-byte aligned): [m][V] fp32 raw logits
 *     (before penalty).
 * Host-side validation (CBD_EINVAL, nothing enqueued): slot/token/pos ranges,
 * pos < n_blocks_per_slot[slot]*32 <= max_blocks_per_seq*32, physical block
 * ids inside the pool and not shared between slots used by the step, distinct
 * positions per slot forming one contiguous run, at most one sampled row per
 * slot, m <= max_slots, sampling parameters finite (temperature >= 0,
 * 0 <= top_p <= 1, 0 <= top_k <= V).  The arrays are copied into pinned
 * staging before return; the caller may reuse them immediately. */
cbd_status cbd_step(cbd_engine* e, cbd_kv_pool* pool,
                    const cbd_row* rows, int32_t n_rows,
                    const int32_t* block_tables, int32_t table_slots,
                    const int32_t* n_blocks_per_slot,
                    const cbd_sampling* sampling, const float* uniforms,
                    int32_t* out_tokens, float* out_logits, void* stream);

/* A Batch: the same inputs as cbd_step, validated once and kept resident in
 * device memory, so the step can be re-run (timing, CUDA-graph capture)
 * without host->device traffic.  Running a batch twice re-writes the same
 * K/V values and updates the counters again.  cbd_batch_create enqueues the
 * upload on `stream`.  The batch may outlive neither the engine nor the pool. */
cbd_status cbd_batch_create(cbd_engine* e, cbd_kv_pool* pool,
                            const cbd_row* rows, int32_t n_rows,
                            const int32_t* block_tables, int32_t table_slots,
                            const int32_t* n_blocks_per_slot,
                            const cbd_sampling* sampling, const float* uniforms,
                            cbd_batch** out, void* stream);
cbd_status cbd_batch_run(cbd_engine* e, cbd_kv_pool* pool, cbd_batch* b,
                         int32_t* out_tokens, float* out_logits, void* stream);
cbd_status cbd_batch_destroy(cbd_batch* b);

/* Number of kernel launches one run of this batch enqueues. */
cbd_status cbd_batch_launches(cbd_batch* b, int32_t* n_launches);

/* CUDA Graph replay of the batch's launch sequence (the CUDA-graph decode
 * step that "RWKV Runner Albatross 后端" lists as follow-up work).  With
 * enable != 0 the next cbd_batch_run captures the step's launches (stream
 * capture on an engine-owned stream; nothing executes while capturing),
 * instantiates them as one graph and launches it into `stream`; later runs
 * with the same pool and output pointers and no engine setting changed since
 * (GEMM or attention path, fused norm, L2 prefetch, forbidden tokens) launch
 * the graph again, and any such change captures a new one.  The kernels and
 * their programmatic-dependency edges are the same as without the graph, so
 * results are bit-identical; the host enqueues one launch per step instead
 * of one per kernel.  enable == 0 drops the graph.  Runs with per-launch
 * profiling on (cbd_engine_profile) do not use the graph. */
cbd_status cbd_batch_set_graph(cbd_batch* b, int32_t enable);
/* How many graphs this batch has captured so far. */
cbd_status cbd_batch_captures(cbd_batch* b, int32_t* n);

/* cbd_step through CUDA graphs: with enable != 0 each cbd_step still
 * validates its inputs and lays out its staging image on the host, then
 * launches one graph that uploads the image and runs the step's kernels.
 * Graphs are cached per staging buffer (up to 8 each, least recently used
 * dropped), keyed by the step's shape (rows, sampled rows, attention work
 * items, table slots, longest chunk list, image size), the pool, the output
 * pointers and the engine settings; a new key captures a new graph (about
 * the cost of one launch-by-launch step).  Results are bit-identical to the
 * launch-by-launch step.  enable == 0 frees the cached graphs (waits for
 * the device).  Not used while per-launch profiling is on. */
cbd_status cbd_engine_set_step_graph(cbd_engine* e, int32_t enable);
/* Graphs captured so far by cbd_step (all keys, all staging buffers). */
cbd_status cbd_engine_step_graph_captures(cbd_engine* e, int32_t* n);

/* Sample m rows of given logits with the same kernel cbd_step uses.
 *   logits (device) [m][V] fp32 (raw); slots (host) [m], distinct;
 *   sampling (host) [m]; uniforms (host, nullable) [m]; out_tokens (device) [m].
 * Updates the slots' counters exactly as a step does. */
cbd_status cbd_sample(cbd_engine* e, const float* logits, int32_t m,
                      const int32_t* slots, const cbd_sampling* sampling,
                      const float* uniforms, int32_t* out_tokens, void* stream);

/* Allocation-free sampler.  The paper has no counterpart to this entry
 * point; it exists for callers that cannot call cudaMalloc -- for example a
 * host framework whose caching allocator already holds the device memory
 * budget, or a serving loop that forbids allocation after warm-up because an
 * allocation can synchronise the device.  It runs the same sampler kernel as
 * cbd_sample on caller-owned buffers, with its scratch (one fp32 row per
 * sampled row plus the rows' parameters) in a fixed-size device array inside
 * libcbd instead of engine memory:
 *   logits (device) [m][vocab] fp32; counters (device) [counter_rows][vocab]
 *   fp32, updated in place exactly as a step updates the engine's counters;
 *   slots (host) [m], distinct, < counter_rows; sampling (host) [m];
 *   uniforms (host, nullable) [m]; out_tokens (device) [m].
 * Limits: 1 <= m <= CBD_SAMPLE_STATIC_MAX_ROWS, 1 <= vocab <=
 * CBD_SAMPLE_STATIC_MAX_VOCAB; larger sizes return CBD_EINVAL with a message.
 * The array (4 MB + 1.3 KB) is held by every GPU that loads libcbd until the
 * process exits.  The first call on a device looks up the array's device
 * address; make that first call before any stream capture.  All calls on a
 * device share the array and it keeps the last call's contents (each call
 * writes what it reads); calls that overlap on the GPU race.  A row for
 * which no token can be drawn (every logit -inf or NaN after the penalty)
 * gets token 0 and sets an error word in the array, which stays set until
 * cbd_sample_static_check reads it.  Calls no cudaMalloc, cudaFree or other
 * allocating routine. */
#define CBD_SAMPLE_STATIC_MAX_ROWS 16
#define CBD_SAMPLE_STATIC_MAX_VOCAB 65536
cbd_status cbd_sample_static(const float* logits, int32_t m, int32_t vocab, float* counters,
                             int32_t counter_rows, const int32_t* slots, const cbd_sampling* sampling,
                             const float* uniforms, int32_t* out_tokens, void* stream);
/* Error status of the cbd_sample_static calls on the current device since
 * the last check: waits for `stream`, reads the array's error word and
 * clears it.  CBD_OK, or CBD_EDEVICE with the code in the message (a row had
 * no token to draw).  Make sure every call to check has reached `stream`
 * (or the device) before it.  Allocates nothing. */
cbd_status cbd_sample_static_check(void* stream);

/* ------------------------------------------------------------ scheduler */
/* Host-side scheduler ("20.3 服务、批处理与流式" section 20.3.2 and 20.3.4):
 * first-come first-served admission that reserves blocks for the prompt
 * plus min(max_tokens, answer_budget) positions, lowest free slot, blocks
 * handed out lowest id first; each plan puts prefill chunks (admission
 * order, at most `chunk` rows each) before one decode row per decoding
 * sequence (longest-waiting first, then admission order) within max_rows;
 * rows that do not fit wait, nothing is evicted.  Growth beyond a
 * reservation takes an unreserved free block or waits, and admission
 * freezes while a row waits for a block.  If every running sequence is
 * stuck, the youngest is stopped (reason CBD_FINISH_FALLBACK) unless
 * stall_fallback == 0, in which case cbd_sched_plan returns CBD_EDEADLOCK.
 * No EOS: a request finishes after max_tokens generated tokens.
 * reserve_answer == 0 gives the free-slot-only admission the page warns
 * about (for tests). */
typedef struct cbd_sched_config {
  int32_t n_blocks;
  int32_t block_size;          /* positions per block (32 in the engine)  */
  int32_t max_slots;
  int32_t max_rows;
  int32_t chunk;               /* prefill rows per sequence per step (512) */
  int32_t answer_budget;       /* reserved answer positions (128)          */
  int32_t max_blocks_per_seq;
  int32_t reserve_answer;      /* 1: reservation policy; 0: free slot only */
  int32_t stall_fallback;      /* 1: stop the youngest when all are stuck  */
  /* Overload and backpressure ("20.3 服务、批处理与流式" section 20.3.4;
   * 0 disables each; the page's defaults are 8, 30000 and a small buffer): */
  int32_t queue_per_slot;      /* waiting requests allowed per slot; submit
                                * beyond max_slots * queue_per_slot waiters
                                * returns CBD_EBUSY                         */
  int32_t queue_timeout_ms;    /* a request still waiting this long after
                                * submit finishes CBD_FINISH_TIMEOUT        */
  int32_t out_buffer;          /* undelivered tokens a request may hold; a
                                * token that finds its buffer full cancels
                                * the request (CBD_FINISH_LAGGING)           */
  /* Composition policy.  CBD_POLICY_FORMA (0): the rules above.
   * CBD_POLICY_ALBATROSS (1), after the Albatross worker loop ("RWKV Runner
   * Albatross 后端", section 连续批处理：Worker 主循环): at most max_prefill
   * requests prefill at a time (admission waits for one to finish); a
   * prompt shorter than short_prompt tokens is fed one token per step, like
   * a decode row; longer prompts advance by one chunk only in "sequence
   * steps", one after every prefill_every steps that carried decode rows
   * (at once when nothing decodes).  The block reservation is kept.  0 in a
   * field takes the page's value: max(floor(0.125 max_slots), 1), 5, 10. */
  int32_t policy;
  int32_t max_prefill;
  int32_t prefill_every;
  int32_t short_prompt;
} cbd_sched_config;

#define CBD_POLICY_FORMA 0
#define CBD_POLICY_ALBATROSS 1

typedef struct cbd_request {
  uint64_t id;                 /* unique per scheduler                     */
  const int32_t* prompt;       /* host [prompt_len], copied on submit      */
  int32_t prompt_len;          /* >= 1                                     */
  int32_t max_tokens;          /* >= 1                                     */
  cbd_sampling sampling;       /* token_index is filled in by the plan     */
} cbd_request;

/* A plan: the rows of the next step and everything cbd_step needs.  All
 * pointers are owned by the scheduler and stay valid until the next
 * cbd_sched_plan / cbd_sched_commit / cbd_sched_destroy. */
typedef struct cbd_plan {
  int32_t n_rows;
  const cbd_row* rows;                 /* prefill rows first, then decode rows */
  int32_t n_sampled;
  const cbd_sampling* sampling;        /* [n_sampled], row order               */
  const uint64_t* sampled_ids;         /* [n_sampled] request id per sampled row */
  int32_t table_slots;                 /* = max_slots                          */
  const int32_t* block_tables;         /* [max_slots][max_blocks_per_seq], -1 pad */
  const int32_t* n_blocks_per_slot;    /* [max_slots]                          */
  int32_t n_resets;
  const int32_t* reset_slots;          /* slots admitted by this plan: zero their counters */
  int32_t n_stopped;
  const uint64_t* stopped_ids;         /* requests stopped by the stall fallback */
} cbd_plan;

#define CBD_FINISH_LENGTH 1
#define CBD_FINISH_FALLBACK 2
#define CBD_FINISH_ABORTED 3          /* cbd_sched_abort: client went away (HTTP 499) */
#define CBD_FINISH_TIMEOUT 4          /* waited longer than queue_timeout_ms (HTTP 429) */
#define CBD_FINISH_LAGGING 5          /* delivery buffer full: slow client cancelled    */

typedef struct cbd_finished {
  uint64_t id;
  int32_t reason;                      /* CBD_FINISH_*                          */
  int32_t n_tokens;                    /* generated tokens                      */
} cbd_finished;

typedef struct cbd_sched_stats {
  int32_t running, waiting, free_blocks, allocated, reserved, outstanding;
  int64_t steps, rows_prefill, rows_decode, fallback_stops, stalled_rows;
  int64_t rejected_busy, timed_out, aborted, lagging;
} cbd_sched_stats;

typedef struct cbd_sched cbd_sched;

cbd_status cbd_sched_create(const cbd_sched_config* cfg, cbd_sched** out);
cbd_status cbd_sched_destroy(cbd_sched* s);
/* Queue a request.  CBD_EPOOL if blocks(prompt + min(max_tokens, budget))
 * exceeds the pool, or prompt + max_tokens - 1 positions exceed
 * max_blocks_per_seq blocks; CBD_EINVAL for an empty prompt, max_tokens < 1
 * or a duplicate id. */
cbd_status cbd_sched_submit(cbd_sched* s, const cbd_request* r);
/* Admit and compose the next step.  n_rows == 0 only when nothing runs. */
cbd_status cbd_sched_plan(cbd_sched* s, cbd_plan* out);
/* Feed back the step's sampled tokens (host [m], row order of the last
 * plan).  Writes up to `cap` finished records to `finished` and their count
 * to *n_finished.  CBD_ESTATE without a preceding plan. */
cbd_status cbd_sched_commit(cbd_sched* s, const int32_t* tokens, int32_t m,
                            cbd_finished* finished, int32_t cap, int32_t* n_finished);
/* Copy up to `cap` generated tokens of a finished request; *n = its count.
 * CBD_EINVAL if the id has not finished. */
cbd_status cbd_sched_output(cbd_sched* s, uint64_t id, int32_t* tokens, int32_t cap, int32_t* n);
/* Cancel a request because its client went away (section 20.3.4: stop
 * generating at once and return the KV blocks).  A waiting request leaves
 * the queue; a running one frees its slot and blocks now, or, if the last
 * plan (not yet committed) has rows of it, at that commit, which drops its
 * token.  It finishes CBD_FINISH_ABORTED (reported by the commit or by
 * cbd_sched_finished).  CBD_EINVAL for an unknown or finished id. */
cbd_status cbd_sched_abort(cbd_sched* s, uint64_t id);
/* The scheduler's clock in milliseconds (caller-driven, so runs replay):
 * submit stamps a request's arrival with it, and cbd_sched_plan expires
 * waiters older than queue_timeout_ms.  Must not go backwards. */
cbd_status cbd_sched_set_time(cbd_sched* s, int64_t now_ms);
/* The client side of a request's delivery buffer: move up to `cap` of its
 * undelivered tokens (oldest first) to `tokens`; *n = how many.  Works for
 * running and finished requests (a finished request keeps its undelivered
 * tokens).  With out_buffer == 0 nothing is buffered and *n = 0. */
cbd_status cbd_sched_read(cbd_sched* s, uint64_t id, int32_t* tokens, int32_t cap, int32_t* n);
/* Requests finished outside a commit (abort of a request not in flight,
 * queue timeouts at plan time) since the last call: up to `cap` records,
 * *n = how many were written; the rest stay for the next call. */
cbd_status cbd_sched_finished(cbd_sched* s, cbd_finished* out, int32_t cap, int32_t* n);
cbd_status cbd_sched_stats_get(cbd_sched* s, cbd_sched_stats* out);

#ifdef __cplusplus
}
#endif
#endif /* CBD_H */
