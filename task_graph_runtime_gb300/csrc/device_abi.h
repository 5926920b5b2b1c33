// Plain-old-data structures shared by the host encoder and the sm_103a
// kernels: the compact device encoding of a linearised tGraph (fixed-size
// task descriptors, events as {count, first, last}) and the launch
// parameters.  MPK: A Compiler and Runtime for Mega-Kernelizing Tensor
// Programs, §2 Q2 ("compact device-memory structure") and "关键实现细节" 2
// (fixed-size task descriptors, prefetched into shared memory).
#pragma once

#include <stdint.h>

namespace mpk {

// 32-byte task descriptor, in linear order.
struct TaskDesc {
  int16_t kind;     // MPK_TASK_*
  uint8_t launch;   // MPK_LAUNCH_*
  uint8_t flags;    // TASK_F_*
  int16_t layer;
  int16_t b;        // attention: sequence
  int32_t dep;      // the one event this task waits on
  int32_t trig;     // the one event this task triggers
  int32_t row0;     // MatMul: output rows [row0, row1)
  int32_t row1;
  int16_t g;        // attention: KV head
  int16_t c;        // attention: KV chunk
  int32_t tile;     // tile index within the operator
};
static_assert(sizeof(TaskDesc) == 32, "task descriptor must stay 32 bytes");

// Tile 0 of a MatMul whose prologue forms a residual sum also stores it.
enum : uint8_t { TASK_F_RESIDUAL = 1u };

// Event flags.  Empty (inline) tasks get the highest ids and BFS appends
// an event's dependent tasks in ascending id, so an event's inline tasks are
// the last n of [first, last]; n is stored in bits 8..31.
enum : uint32_t { EV_HAS_JIT = 1u, EV_HAS_INLINE = 2u, EV_FAN_CACHED = 4u };
constexpr int kEvInlineShift = 8;

// 16-byte event descriptor: activated when its counter reaches
// epoch * count; its dependent tasks are [first, last].
struct EventDesc {
  uint32_t count;
  int32_t first;
  int32_t last;
  uint32_t flags;   // EV_HAS_*
};
static_assert(sizeof(EventDesc) == 16, "event descriptor must stay 16 bytes");

// One entry of a worker's AOT queue with everything its leader needs about
// the task: the descriptor, the count its dependent event reaches per step,
// and its triggering event.  Fetched asynchronously while the task before
// it runs, so dispatch and trigger make no dependent global loads.
// When every dependent task of the triggering event is an empty (inline)
// task, there are at most two of them and each triggers an event with no
// JIT or inline work of its own, trig_ev.flags carries EV_FAN_CACHED and
// fan[] holds those events: the trigger then fires them without reading the
// graph (and, for an event with one trigger, without touching its counter,
// which nothing else reads).
struct AotRec {
  TaskDesc desc;
  uint32_t dep_count;
  int32_t id;          // linear task id
  int32_t fan[2];
  EventDesc trig_ev;
};
static_assert(sizeof(AotRec) == 64, "AOT record must stay 64 bytes");

// Multi-producer single-consumer ring in global memory.  Slot value:
// (ticket << 32) | payload, ticket = position + 1.  Head and tail live on
// separate 128-byte lines.
struct RingHdr {
  uint32_t tail;
  uint32_t pad0[31];
  uint32_t head;
  uint32_t pad1[31];
};

// Weight pages.
// Batch 1: the rows [i, i + n) of a tile are n * K contiguous elements, so a
// page is b1_rows_per_page(K) whole rows (at most 32 KB) in one bulk copy.
// With 8 or more rows a page, consumer warp w dots rows w, w + 8, ...; with
// fewer, each row is split over b1_warps_per_row(K) warps into equal column
// parts, and warp w always takes part w % b1_warps_per_row(K), one partial
// sum each.
// Batch > 1: 8 matrix rows x up to 2048 columns, each row one bulk copy,
// rows kPagePitch bytes apart (16 bytes of skew per row keep ldmatrix reads
// of 8 rows free of bank conflicts).
constexpr int kContigPageBytes = 32768;
constexpr int kPageRows = 8;
constexpr int kSegCols = 2048;
constexpr int kPagePitch = kSegCols * 2 + 16;          // 4112
constexpr int kPageBytes = kPageRows * kPagePitch;     // 32896
constexpr int kAttnMaxTokens = 128;                    // per prefetched chunk
constexpr int kB1Partials = 2560;   // batch-1 row partial sums per tile

#if defined(__CUDACC__)
#define MPK_HD __host__ __device__
#else
#define MPK_HD
#endif
MPK_HD inline int b1_rows_per_page(int K) {
  const int r = (kContigPageBytes / 2) / K;
  return r < 1 ? 1 : r;
}
MPK_HD inline int b1_warps_per_row(int K) {
  const int r = b1_rows_per_page(K);
  return r >= 8 ? 1 : 8 / r;
}

// Byte offsets of the regions of a worker CTA's dynamic shared memory.
struct SmemLayout {
  int n_pages;      // ring slots
  int page_bytes;   // slot size: kContigPageBytes (batch 1) or kPageBytes
  int xs;           // activation staging / attention scratch
  int xs_bytes;
  int res;          // MatMul row results (fp32)
  int res_floats;
  int bars;         // full[n_pages], empty[n_pages] mbarriers
  int ctrl;         // control words + staged task descriptors
  int scratch;      // small reductions (512 bytes)
  int total;
};

// Shape and geometry the kernels need.
struct Dims {
  int L, h, Hq, Hkv, d, F, V, chain_ffn, qk_norm;
  float eps;
  float attn_scale;  // 1/sqrt(d), rounded once from double on the host
  int B;             // batch
  int C;             // split-KV chunks per (sequence, KV head)
  int page_size, max_pages;
  int n_lm_tiles;
  int max_ctx;       // rows of the RoPE table
  int kmax;          // longest MatMul reduction (x staging at batch 1)
};

// Activation workspace: one block per layer (identical layout), plus a
// block of step-global tensors.  Offsets in bytes.
struct ActLayout {
  char* base;
  int64_t layer_stride;
  int64_t o_h, o_qkv, o_opart, o_attn, o_o, o_hmid, o_act, o_dout;
  int64_t g_z, g_amax;         // offsets from the global block
  int64_t global_block;        // offset of the global block from base
};

struct DevGraph {
  const TaskDesc* tasks;
  const EventDesc* events;
  int n_tasks, n_events;
  int root, end;
  const int32_t* aot_list;     // per worker, linear task ids in order
  const int32_t* aot_off;      // [W + 1]
  const AotRec* aot_rec;       // parallel to aot_list
  const int32_t* op_tasks;     // per operator, linear ids in tile order
  uint32_t* counters;          // [n_events]
  uint32_t* merge_cnt;         // [L][B][Hkv] attention chunk arrivals
  RingHdr* jit_hdr;            // [W]
  unsigned long long* jit_cost;  // JIT work dealt so far (tokens + fixed
                                 // part per task), over all steps
  uint64_t* jit_slots;         // [W][jit_cap]
  RingHdr* sched_hdr;          // [S]
  uint64_t* sched_slots;       // [S][sched_cap]
  uint32_t jit_cap, sched_cap;
  uint32_t* status;            // latched mpk_status
  uint32_t* abort_flag;
  uint64_t* trace;             // nullable: 8 words per executed task
  uint32_t* trace_count;
  uint32_t trace_cap;          // records
  int W;                       // worker CTAs
  int has_jit;                 // any JIT task (else workers never poll
                               // their JIT rings)
  int S;                       // scheduler warps in total
  int sched_warps_per_sm;
};

struct WeightPtrs {
  const uint16_t* embed;
  const uint16_t* final_norm;
  const uint16_t* lm_head;
  const uint16_t* chain_w1;
  const uint16_t* chain_w2;
  const uint16_t* const* layers;   // device array [L][MPK_LAYER_NTENSORS]
  const float* rope_cs;            // [max_ctx][d/2][2] (cos, sin)
};

struct StepArgs {
  const int32_t* tokens;
  uint16_t* k_pool;
  uint16_t* v_pool;
  const int32_t* page_table;
  int32_t* seq_lens;
  int num_pages;
  float* logits;
  int32_t* next_tokens;
  uint32_t epoch;               // first step's number since the last reset
  int n_steps;                  // greedy steps run by this launch (>= 1):
                                // step i embeds the tokens step i - 1 wrote
                                // to next_tokens + (i - 1) * B and writes its
                                // own to next_tokens + i * B
  uint64_t timeout_ns;
};

struct KernelParams {
  Dims dims;
  SmemLayout sm;
  DevGraph graph;
  WeightPtrs w;
  ActLayout act;
  StepArgs step;
};

}  // namespace mpk
