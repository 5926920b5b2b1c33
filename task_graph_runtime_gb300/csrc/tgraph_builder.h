// Host tGraph builder: operators -> per-tile tasks -> overlap events ->
// fused events -> normalised graph -> BFS-linearised graph.
//
// MPK: A Compiler and Runtime for Mega-Kernelizing Tensor Programs,
// §2 Q2 (decomposition, dependency analysis, fusion, normalisation,
// linearisation into a compact device structure) and §4 (Defs 4.1/4.2,
// "6 minimum checks" items 1-4).
#pragma once

#include <cstdint>
#include <string>
#include <vector>

#include "mpk.h"

namespace mpk {

struct Region {
  int tensor;            // interned (tensor kind, layer)
  int r0, r1, c0, c1;    // half-open rectangle over a 2-D view
};

struct BTask {
  int kind = MPK_TASK_EMPTY;
  int op = -1;
  int layer = -1;
  int tile = 0;
  int row0 = 0, row1 = 0;
  int b = 0, g = 0, c = 0;
  std::vector<Region> reads, writes;
};

struct BOp {
  int kind, layer, first, n;
};

struct BuildConfig {
  mpk_model_shape shape;
  int batch;
  int num_workers;
  int gemv_rows_per_task;  // batch < 8 (0: default)
  int mma_rows_per_task;   // batch >= 8 (0: default)
  int attn_chunks;         // resolved (> 0 for decoder mode)
  int coarse_events;       // 1: operator-level events (Figure 4c ablation)
};

struct BuiltGraph {
  BuildConfig cfg;
  std::vector<BOp> ops;
  std::vector<BTask> tasks;      // pre-linearisation ids; empties appended
  int n_real = 0;
  int64_t n_raw = 0, n_fused = 0;
  // linearised (index = linear position / linear event id)
  std::vector<int32_t> order, dep, trig, launch, worker;
  std::vector<int32_t> ev_count, ev_first, ev_last;
  int root_lin = 0, end_lin = 0;   // linear ids of the root and end events
};

// Most output rows one MatMul tile with reduction length K may hold.  Batch
// 1: its row partial sums (rows x warps per row, twice for a gate/up tile)
// fit the 2560-float result buffer; batch 2..7: 64 weight rows, batch >= 8:
// 128 weight rows (per-thread accumulators); a gate/up tile streams two
// weight rows per output row.  Rounded down to a multiple of 8.
int tile_row_cap(int batch, bool dual, int K);

// Row tiling of an N-row MatMul in units of `unit` rows (1 at batch 1, 8
// otherwise): explicit size (at most the cap), or T = W * ceil(T0 / W)
// tiles (at most U = ceil(N/unit)) with T0 = ceil(U / (cap/unit)),
// boundaries at unit * floor(i*U/T) rows.
std::vector<std::pair<int, int>> row_tiles(int n_rows, int rows_per_task,
                                           int num_workers, int cap_rows,
                                           int unit);

// Attention chunks are AOT (their KV prefetched into the ring) at batch 1
// when no chunk can exceed 128 tokens, JIT otherwise.
bool attn_is_aot(int batch, int max_ctx, int chunks);

int default_attn_chunks(int batch, int n_kv_heads, int max_ctx,
                        int num_workers);

// Validates the shape (the task bodies' limits) and builds the graph.
// Returns MPK_OK or an error with a message in *err.
mpk_status build_tgraph(const BuildConfig& cfg, BuiltGraph* out,
                        std::string* err);

// Re-checks the invariants of a linearised graph (<=1/<=1 by construction,
// contiguous fan-outs, counts, topological order).
bool validate(const BuiltGraph& g, std::string* err);

}  // namespace mpk
