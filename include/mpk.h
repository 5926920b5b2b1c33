/*
 * mpk.h -- C ABI of the GB300 (sm_103a) mega-kernel decode runtime.
 *
 * One LLM decode step is compiled into a task/event graph (tGraph) and run
 * inside one persistent kernel: "MPK: A Compiler and Runtime for
 * Mega-Kernelizing Tensor Programs" (§2 Q2, §4, Table 1).  Two calls carry
 * the method: mpk_build_tgraph (model shape + tile sizes -> tGraph) and
 * mpk_decode_step (graph + tokens + paged KV cache + stream -> one step).
 *
 * Conventions for every call:
 *   - All tensors are row-major.  bf16 tensors are IEEE bfloat16 bit
 *     patterns (uint16).  Pointers named d_* and every pointer inside
 *     mpk_weights / mpk_kv_cache are CUDA device pointers on the device that
 *     is current when mpk_bind_weights is called; all other pointers are host
 *     pointers.
 *   - Ownership: the caller owns weights, KV pools, page tables, seq_lens,
 *     tokens, logits and next-token buffers, and keeps them alive while the
 *     graph uses them (pointers are borrowed, never copied or freed).  The
 *     library owns the graph, its device encoding (descriptors, queues,
 *     counters) and the activation workspace, all released by
 *     mpk_destroy_tgraph.
 *   - Errors: host-detectable errors are returned synchronously and leave
 *     the graph unchanged.  Errors detected inside the kernel (a bounded wait
 *     that ran out, an unmapped KV page, a full queue) are latched in a
 *     device status word that mpk_get_status reads; the kernel then exits
 *     cleanly and the graph needs mpk_reset before the next step.
 *   - Threading: no global state.  One graph is used by one host thread and
 *     one stream at a time; distinct graphs are independent.
 */
#ifndef MPK_H_
#define MPK_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MPK_OK = 0,
  MPK_ERR_INVALID_ARG = 1,     /* a null pointer, a non-positive size, ... */
  MPK_ERR_UNSUPPORTED = 2,     /* a shape the task bodies do not handle    */
  MPK_ERR_CUDA = 3,            /* a CUDA runtime/driver call failed         */
  MPK_ERR_OOM = 4,             /* device or host allocation failed          */
  MPK_ERR_NOT_CORESIDENT = 5,  /* workers + schedulers exceed the SMs, or
                                  the persistent grid cannot be co-resident */
  MPK_ERR_TIMEOUT = 6,         /* a bounded device wait ran out             */
  MPK_ERR_KV_PAGE = 7,         /* page_table holds -1 where a token lives   */
  MPK_ERR_QUEUE_OVERFLOW = 8,  /* a device queue could not take an entry    */
  MPK_ERR_GRAPH_INVALID = 9,   /* the built graph failed its invariants     */
  MPK_ERR_NOT_BOUND = 10       /* decode before mpk_bind_weights            */
} mpk_status;

/* Model shape.  Decoder mode: n_layers >= 1, chain_ffn == 0.  Chained-linear
 * mode: n_layers == 0 and chain_ffn > 0; the step is then
 * x = embed[token]; n = RMSNorm(x, final_norm); y = silu(n W1^T);
 * z = y W2^T; logits = z lm_head^T (no KV cache, no attention). */
typedef struct {
  int n_layers;
  int hidden;
  int n_q_heads;
  int n_kv_heads;
  int head_dim;          /* even, <= 128                                   */
  int ffn;               /* SwiGLU intermediate size                        */
  int vocab;
  float rms_eps;
  float rope_theta;
  int qk_norm;           /* 1: per-head RMSNorm of q and k before RoPE      */
  int chain_ffn;         /* > 0 selects the chained-linear mode             */
  int page_size;         /* KV tokens per page                              */
  int max_pages_per_seq; /* columns of the page table                       */
} mpk_model_shape;

/* Tile sizes and runtime geometry; 0 selects the default. */
typedef struct {
  int num_workers;        /* W worker SMs.  0: the SM count of the current
                             device minus num_sched_sms (needs a GPU)       */
  int gemv_rows_per_task; /* MatMul output rows per task at batch < 8 (a
                             multiple of 8).  0: T = W * ceil(ceil(N/cap)/W)
                             tiles (at most ceil(N/8)) of multiples of 8
                             rows (single rows at batch 1).  cap at batch 1:
                             2560 / p rows, p = the partial sums a row's dot
                             product is split into (1 when a 32 KB page
                             holds r = max(1, 16384 / K) >= 8 rows, else
                             8 / r); 64 at batch 2..7; a gate/up row counts
                             twice; rounded down to a multiple of 8        */
  int mma_rows_per_task;  /* the same for batch >= 8, where MatMul tiles run
                             on tensor cores; 0: as above with cap = 128    */
  int attn_chunks;        /* split-KV chunks per (sequence, KV head).  0:
                             max(1, min(ceil(max_ctx/128),
                             ceil(4W/(batch*n_kv_heads))))                  */
  int num_sched_sms;      /* SMs running scheduler warps.  0: 4 (Table 1)
                             when the graph has JIT tasks, none when every
                             task is AOT (no dispatch: all SMs are workers) */
  int sched_warps_per_sm; /* 0: 4 (Table 1)                                 */
  int smem_pages;         /* weight pages per worker (batch 1: 32 KB of
                             whole rows; batch > 1: 8 rows x 2048 columns,
                             32 KB + row skew). 0: as many as fit, <= 6    */
  int coarse_events;      /* 1: every task of an operator waits for every
                             task of the operators it reads (the
                             operator-level graph of Figure 4c, an
                             ablation); 0: region-overlap events           */
} mpk_tile_sizes;

/* Task kinds (one per operator of the decode step). */
enum {
  MPK_TASK_EMPTY = 0,     /* normalisation glue: waits, then triggers      */
  MPK_TASK_QKV = 1,       /* MatMul tile of W_qkv; prologue: residual add
                             (layer 0: embedding gather) + RMSNorm          */
  MPK_TASK_ATTN = 2,      /* one KV chunk of one (sequence, KV head): q/k
                             RMSNorm (optional) + RoPE + KV append, paged
                             attention over the chunk, and the log-sum-exp
                             merge of all chunks by the last to finish     */
  MPK_TASK_O = 3,         /* MatMul tile of W_o                             */
  MPK_TASK_GATEUP = 4,    /* MatMul tile of W_gate and W_up; prologue:
                             residual add + RMSNorm; epilogue: SwiGLU       */
  MPK_TASK_DOWN = 5,      /* MatMul tile of W_down                          */
  MPK_TASK_LM_HEAD = 6,   /* MatMul tile of lm_head (prologue: final norm),
                             fp32 logits + tile argmax                      */
  MPK_TASK_ARGMAX = 7,    /* argmax over tile maxima; seq_lens += 1         */
  MPK_TASK_CHAIN_UP = 8,  /* MatMul tile of W1 (prologue: RMSNorm) + SiLU   */
  MPK_TASK_CHAIN_DOWN = 9,
  MPK_TASK_NKINDS = 10
};

/* Launch classes (hybrid JIT/AOT, MPK summary §2 Q2 and "Design space"). */
enum {
  MPK_LAUNCH_AOT = 0,     /* statically placed on one worker's queue        */
  MPK_LAUNCH_JIT = 1,     /* placed by a scheduler warp when its event fires*/
  MPK_LAUNCH_INLINE = 2   /* empty task, run by whoever fires its event     */
};

/* Execution modes of mpk_decode_step. */
enum {
  MPK_MODE_MEGAKERNEL = 0,  /* one persistent launch per step (default)     */
  MPK_MODE_KPO = 1,         /* one launch per operator, same task bodies    */
  MPK_MODE_KPO_GRAPH = 2    /* the KPO launches replayed from a CUDA Graph  */
};

/* Per-layer weight tensors, in the order of mpk_weights.layers. */
enum {
  MPK_W_LN1 = 0,     /* bf16 [hidden]                                       */
  MPK_W_QKV = 1,     /* bf16 [(Hq + 2 Hkv) d][hidden]: q heads, k heads, v  */
  MPK_W_QNORM = 2,   /* bf16 [d] (qk_norm only, else ignored)               */
  MPK_W_KNORM = 3,   /* bf16 [d] (qk_norm only, else ignored)               */
  MPK_W_O = 4,       /* bf16 [hidden][Hq d]                                 */
  MPK_W_LN2 = 5,     /* bf16 [hidden]                                       */
  MPK_W_GATEUP = 6,  /* bf16 [2 ffn][hidden]: rows [0,ffn) gate, then up    */
  MPK_W_DOWN = 7,    /* bf16 [hidden][ffn]                                  */
  MPK_LAYER_NTENSORS = 8
};

typedef struct mpk_graph mpk_graph; /* opaque, library-owned */

/* Device weight pointers (borrowed).  Every bf16 tensor must be 16-byte
 * aligned.  `layers` is a HOST array of n_layers * MPK_LAYER_NTENSORS device
 * pointers, read during the call only. */
typedef struct {
  const void* embed;           /* bf16 [vocab][hidden]                       */
  const void* final_norm;      /* bf16 [hidden]                              */
  const void* lm_head;         /* bf16 [vocab][hidden]                       */
  const void* const* layers;   /* decoder mode                               */
  const void* chain_w1;        /* chained mode: bf16 [chain_ffn][hidden]     */
  const void* chain_w2;        /* chained mode: bf16 [hidden][chain_ffn]     */
} mpk_weights;

/* Paged KV cache (caller-owned device memory).  Token t of sequence b lives
 * in page page_table[b][t / page_size] at slot t % page_size. */
typedef struct {
  void* k_pool;                /* bf16 [n_layers][num_pages][Hkv][page_size][d] */
  void* v_pool;                /* same layout                                */
  const int32_t* page_table;   /* int32 [batch][max_pages_per_seq], -1 = none */
  int32_t* seq_lens;           /* int32 [batch]: tokens already cached       */
  int num_pages;
} mpk_kv_cache;

/* Host arrays describing a built graph, owned by the graph (valid until
 * mpk_destroy_tgraph).  Tasks and events are in linearised order. */
typedef struct {
  int n_tasks, n_events, n_ops, n_empty, n_workers, attn_chunks;
  const int32_t* task_kind;    /* MPK_TASK_*                                 */
  const int32_t* task_op;      /* operator index, -1 for empty tasks         */
  const int32_t* task_layer;   /* layer (n_layers for the final operators)   */
  const int32_t* task_tile;    /* tile index within its operator             */
  const int32_t* task_row0;    /* MatMul: output rows [row0, row1)           */
  const int32_t* task_row1;
  const int32_t* task_b;       /* attention family: sequence, KV head, chunk */
  const int32_t* task_g;
  const int32_t* task_c;
  const int32_t* task_dep;     /* the one event the task waits on            */
  const int32_t* task_trig;    /* the one event the task triggers            */
  const int32_t* task_launch;  /* MPK_LAUNCH_*                               */
  const int32_t* task_worker;  /* AOT worker, -1 otherwise                   */
  const int32_t* task_pre_id;  /* id before linearisation (program order)    */
  const int32_t* event_count;  /* triggers needed to activate the event      */
  const int32_t* event_first;  /* dependent tasks are [first, last]          */
  const int32_t* event_last;
  const int32_t* op_kind;      /* per operator, in program order             */
  const int32_t* op_layer;
  const int32_t* op_n_tasks;
  int64_t n_raw_events;        /* events before fusion                       */
  int64_t n_fused_events;      /* events after fusion, before normalisation  */
  int n_sched_sms;             /* scheduler SMs of the launch (0: all-AOT)   */
  int sched_warps_per_sm;
} mpk_graph_export;

/* Decompose one decode step of `shape` at `batch` sequences into per-tile
 * tasks, derive events from overlapping output/input regions, fuse them
 * (Defs 4.1 and 4.2), normalise (<= 1 dependent and <= 1 triggering event
 * per task) and BFS-linearise (each event's fan-out is [first, last]).
 * MPK summary §2 Q2 and §4 "6 minimum checks".  Host only: touches no GPU
 * unless tiles->num_workers == 0.  On success *out owns a new graph. */
mpk_status mpk_build_tgraph(const mpk_model_shape* shape,
                            const mpk_tile_sizes* tiles, int batch,
                            mpk_graph** out);

/* Copy the graph's device encoding to the current device, allocate the
 * activation workspace and bind the weights (pointers borrowed).  May be
 * called again to rebind other weights of the same shape. */
mpk_status mpk_bind_weights(mpk_graph* g, const mpk_weights* w);

/* Enqueue one decode step on `cuda_stream` (a cudaStream_t, 0 = legacy
 * default stream): d_tokens int32 [batch] in; d_logits fp32 [batch][vocab]
 * and d_next_tokens int32 [batch] (greedy, lowest index on ties) out.  Reads
 * kv->seq_lens[b] as the position of the new token, writes its K/V there,
 * and on success increments seq_lens in the kernel.  Asynchronous: returns
 * after the launch(es) are enqueued.  In megakernel mode this is one
 * cooperative launch of a persistent grid (MPK summary, Figure 1: "a
 * single launch").  d_tokens may alias the previous step's d_next_tokens. */
mpk_status mpk_decode_step(mpk_graph* g, const int32_t* d_tokens,
                           const mpk_kv_cache* kv, float* d_logits,
                           int32_t* d_next_tokens, void* cuda_stream);

/* Several greedy steps in ONE launch (MPK summary, Figure 1: the whole
 * decode loop inside a single launch).  Step i (0 <= i < n_steps) embeds
 * d_tokens for i = 0, else the tokens step i - 1 wrote; it writes its own to
 * d_next_tokens + i * batch (device int32 [n_steps][batch]).  d_logits
 * receives the last step's logits.  kv and seq_lens advance by n_steps.
 * Inside the kernel every worker walks its task queue once per step: the
 * first tasks of step i + 1 wait for step i's end event, while the
 * producers already stream step i + 1's weights during step i's last tasks
 * (cached K/V pages only after that end event).  In the kernel-per-operator
 * modes the steps are enqueued one after another.  Same errors and
 * asynchrony as mpk_decode_step; n_steps < 1 is MPK_ERR_INVALID_ARG. */
mpk_status mpk_decode_steps(mpk_graph* g, const int32_t* d_tokens,
                            const mpk_kv_cache* kv, float* d_logits,
                            int32_t* d_next_tokens, int n_steps,
                            void* cuda_stream);

/* Read the device status word of the last step.  Synchronises the device.
 * MPK_OK, or the first error the kernel latched. */
mpk_status mpk_get_status(mpk_graph* g);

/* Select MPK_MODE_MEGAKERNEL, MPK_MODE_KPO or MPK_MODE_KPO_GRAPH. */
mpk_status mpk_set_mode(mpk_graph* g, int mode);

/* Fill *out with host arrays of the built graph (for parity checks). */
mpk_status mpk_export_tgraph(const mpk_graph* g, mpk_graph_export* out);

/* Clear the device status, abort flag, event counters and queues after an
 * error (synchronises the device).  The KV cache is the caller's to fix. */
mpk_status mpk_reset(mpk_graph* g);

/* Free everything the graph owns.  Null is ignored. */
void mpk_destroy_tgraph(mpk_graph* g);

const char* mpk_status_string(mpk_status s);

/* Test hooks.  mpk_debug_set_wait_timeout_ms bounds every device wait of
 * later steps (default 2000 ms).  mpk_debug_add_event_count adds `delta` to
 * the trigger count of linearised event `event` in the device encoding, so a
 * test can make a wait that never completes and check MPK_ERR_TIMEOUT. */
mpk_status mpk_debug_set_wait_timeout_ms(mpk_graph* g, int ms);
mpk_status mpk_debug_add_event_count(mpk_graph* g, int event, int delta);

/* Tracing (megakernel mode).  mpk_debug_set_trace(g, capacity) allocates
 * room for `capacity` task records (0 disables).  Each executed task adds one
 * record of eight uint64: task id | (worker << 32), then the %globaltimer
 * nanoseconds at which the worker's leader started looking for it, found it
 * ready, had its operands staged (batch-1 MatMul tiles; else 0), had
 * consumed its last weight page (batch-1 MatMul tiles; else 0), finished its
 * body, and finished its trigger; the eighth word is 0.
 * mpk_debug_read_trace copies up to `capacity` records into host_records,
 * stores the count, and clears the trace for the next steps (synchronises
 * the device). */
mpk_status mpk_debug_set_trace(mpk_graph* g, int capacity);
mpk_status mpk_debug_read_trace(mpk_graph* g, uint64_t* host_records,
                                int capacity, int* n_records);

/* Copy the residual stream entering decoder layer `layer` of the last step
 * (0 <= layer <= n_layers; n_layers is the input of the final RMSNorm) into
 * host_out, bf16 [batch][hidden] (synchronises the device).  The first
 * MatMul tile of each layer (and of lm_head) stores it as a by-product of
 * its RMSNorm prologue.  Decoder mode only. */
mpk_status mpk_debug_read_hidden(mpk_graph* g, int layer, uint16_t* host_out);

/* CPU model of the runtime protocol (no GPU needed).  Runs `steps` steps
 * of g's own device encoding with one host thread per worker leader and per
 * scheduler warp: epoch counters, AOT queues in linear order (with the
 * cached fan-outs of the AOT records), JIT dispatch through scheduler and
 * worker rings, and empty tasks run inline by the activating trigger, as
 * the kernel does (MPK summary, §2 Q2 runtime; Figure 8).  Task bodies
 * are replaced by random delays of 0..max_delay_us microseconds (seeded).
 * Reports, in *report: executions, executions that started before some
 * task triggering their event had finished in the same step, duplicate and
 * missing executions per completed step, and whether a step failed to
 * finish within timeout_ms (a deadlock).  Returns MPK_ERR_INVALID_ARG for
 * bad arguments; the verdict is in the report. */
typedef struct {
  int64_t tasks_run;
  int64_t order_violations;
  int64_t duplicate_runs;
  int64_t missing_runs;
  int32_t deadlocked;
  int32_t steps_completed;
  double seconds;
} mpk_sim_report;
mpk_status mpk_debug_simulate(const mpk_graph* g, int steps, uint32_t seed,
                              int max_delay_us, int timeout_ms,
                              mpk_sim_report* report);

/* Allocation-free decode step.  (The paper has no counterpart: this is a
 * convenience for callers of the library.)
 *
 * For callers that cannot call cudaMalloc while they run: a serving process
 * whose device memory is reserved up front by its own caching allocator, a
 * latency-critical loop that may not take the device-wide synchronisation
 * cudaMalloc/cudaFree imply, or a plugin whose host owns every allocation.
 * The call runs the kernel-per-operator form of the step (the same task
 * bodies as mpk_decode_step) and keeps all of its scratch -- task
 * descriptors, the layer pointer table, the RoPE table, the attention merge
 * counters, the activation workspace and the status words -- in one static
 * device array of MPK_NOALLOC_SCRATCH_BYTES that every
 * GPU loading the library holds until the process exits.  It calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *
 * g comes from mpk_build_tgraph (mpk_bind_weights is not needed); w, d_tokens,
 * kv, d_logits and d_next_tokens are as for mpk_bind_weights and
 * mpk_decode_step, on the current device.  d_status (nullable, device
 * uint32) receives the step's mpk_status once the step has run.
 * Returns MPK_ERR_UNSUPPORTED, before touching the device, when the graph
 * needs more scratch than MPK_NOALLOC_SCRATCH_BYTES (8 MiB: e.g. the tiny,
 * ~1B-parameter and chained-linear shapes fit, the 36-layer 8B shape does
 * not).  The first call on a device looks up the array's device address,
 * so make that first call before any stream capture.  All calls share the
 * one array, which keeps the last call's contents: calls that overlap on
 * the GPU (other streams, or other host threads) race and must not be
 * issued.  Asynchronous on cuda_stream. */
#define MPK_NOALLOC_SCRATCH_BYTES (8u << 20)
mpk_status mpk_decode_step_noalloc(const mpk_graph* g, const mpk_weights* w,
                                   const int32_t* d_tokens,
                                   const mpk_kv_cache* kv, float* d_logits,
                                   int32_t* d_next_tokens, uint32_t* d_status,
                                   void* cuda_stream);

#ifdef __cplusplus
}
#endif
#endif /* MPK_H_ */
