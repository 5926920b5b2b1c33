// Host-side geometry of a built graph, shared by the translation units that
// launch it (capi.cpp and noalloc.cu): the worker CTA's shared-memory
// regions, the kernels' shape parameters and the activation workspace.
#pragma once

#include <cstdint>

#include "device_abi.h"
#include "tgraph_builder.h"

namespace mpk {

// Shared-memory layout for `pages_req` ring pages (0: as many as fit, at
// most 6), shrunk until it fits `limit` bytes.  False if even two pages do
// not fit.
bool smem_layout(const BuiltGraph& bg, int pages_req, int limit,
                 SmemLayout* out);

// Number of lm_head tiles (the argmax task's fan-in).
int lm_head_tiles(const BuiltGraph& bg);

// Kernel shape parameters.
Dims make_dims(const BuiltGraph& bg);

// Activation workspace offsets (A->base left null); returns its size in
// bytes.  256-byte aligned blocks: one per layer plus one per step.
int64_t act_layout(const BuiltGraph& bg, ActLayout* A);

// Size of the merge-counter array ([L][batch][Hkv] u32).
int64_t merge_counters(const BuiltGraph& bg);

// Host table of (cos, sin) of p * theta^(-2i/d) evaluated in double and
// rounded once to fp32, [max_ctx][d/2][2].
void rope_table(const mpk_model_shape& s, float* out);
int64_t rope_table_floats(const mpk_model_shape& s);

// Task flags the kernels read (TASK_F_*).
uint8_t task_flags(const BuiltGraph& bg, int kind, int tile);

}  // namespace mpk
