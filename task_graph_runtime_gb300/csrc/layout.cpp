// Host-side geometry of a built graph; see layout.h.
#include "layout.h"

#include <algorithm>
#include <cmath>

namespace mpk {

namespace {
int round_up(int x, int a) { return (x + a - 1) / a * a; }
int64_t round_up64(int64_t x, int64_t a) { return (x + a - 1) / a * a; }
}  // namespace

bool smem_layout(const BuiltGraph& bg, int pages_req, int limit,
                 SmemLayout* out) {
  const mpk_model_shape& s = bg.cfg.shape;
  const int B = bg.cfg.batch;
  const bool chain = s.chain_ffn > 0;
  const int kmax = chain ? std::max(s.hidden, s.chain_ffn)
                         : std::max({s.hidden, s.n_q_heads * s.head_dim,
                                     s.ffn});
  // bf16 x at batch 1; at batch > 1 one 2048-column segment of every
  // sequence plus a 512-column scratch row per sequence for the staging
  int xs = B == 1 ? round_up(kmax * 2, 16) : B * kPagePitch + B * 64 * 16;
  // batch >= 8: the MatMul tile's 8 per-warp partial sums (fp32, up to 128
  // rows of every sequence) are added through this buffer at the tile's end
  if (B >= 8) xs = std::max(xs, 8 * B * 128 * 4);
  if (!chain) {
    const int grp = s.n_q_heads / s.n_kv_heads, d = s.head_dim;
    // query rows + 8 warp records (+ the new K/V rows)
    int attn = (grp * d + 8 * grp * (2 + d)) * 4 + 2 * d * 2;
    const int max_ctx = s.max_pages_per_seq * s.page_size;
    if (!attn_is_aot(B, max_ctx, bg.cfg.attn_chunks))
      attn += 2 * 64 * d * 2 * 2;   // two K/V stages of 64 tokens (JIT)
    xs = std::max(xs, round_up(attn, 16));
  }
  const int res_floats = B == 1 ? kB1Partials : B * (B < 8 ? 64 : 128);
  const int page_bytes = B == 1 ? kContigPageBytes : kPageBytes;
  // default ring depth: 4 pages at batch 1 (measured faster than 5 or 6 on
  // the 8B shape: fewer bulk copies in flight keep the L2 and HBM queues,
  // and so the latency of every operator boundary, shorter), else as many as
  // fit up to 6
  int pages = pages_req > 0 ? std::min(pages_req, 8) : (B == 1 ? 4 : 6);
  for (; pages >= 2; --pages) {
    SmemLayout L{};
    L.n_pages = pages;
    L.page_bytes = page_bytes;
    int off = pages * page_bytes;
    L.xs = off;
    L.xs_bytes = xs;
    off = round_up(off + xs, 128);
    L.res = off;
    L.res_floats = res_floats;
    off = round_up(off + res_floats * 4, 128);
    L.bars = off;
    off = round_up(off + 16 * pages, 128);
    L.ctrl = off;
    off += 448;   // control words, staged descriptors and records, times,
                  // attention positions per ring slot
    L.scratch = off;
    off += 384;   // reductions: <= 96 floats
    L.total = off;
    if (off <= limit) {
      *out = L;
      return true;
    }
  }
  return false;
}

int lm_head_tiles(const BuiltGraph& bg) {
  for (const BOp& o : bg.ops)
    if (o.kind == MPK_TASK_LM_HEAD) return o.n;
  return 0;
}

Dims make_dims(const BuiltGraph& bg) {
  const mpk_model_shape& s = bg.cfg.shape;
  const bool chain = s.chain_ffn > 0;
  Dims D{};
  D.L = s.n_layers;
  D.h = s.hidden;
  D.Hq = s.n_q_heads;
  D.Hkv = s.n_kv_heads;
  D.d = s.head_dim;
  D.F = s.ffn;
  D.V = s.vocab;
  D.chain_ffn = s.chain_ffn;
  D.qk_norm = s.qk_norm;
  D.eps = s.rms_eps;
  D.attn_scale = chain ? 1.0f : (float)(1.0 / std::sqrt((double)s.head_dim));
  D.B = bg.cfg.batch;
  D.C = chain ? 0 : bg.cfg.attn_chunks;
  D.page_size = s.page_size;
  D.max_pages = s.max_pages_per_seq;
  D.n_lm_tiles = lm_head_tiles(bg);
  D.max_ctx = chain ? 1 : s.max_pages_per_seq * s.page_size;
  D.kmax = chain ? std::max(s.hidden, s.chain_ffn)
                 : std::max({s.hidden, s.n_q_heads * s.head_dim, s.ffn});
  return D;
}

int64_t act_layout(const BuiltGraph& bg, ActLayout* A) {
  const mpk_model_shape& s = bg.cfg.shape;
  const bool chain = s.chain_ffn > 0;
  const int64_t B = bg.cfg.batch, h = s.hidden, d = s.head_dim;
  const int64_t Hq = s.n_q_heads, Hkv = s.n_kv_heads;
  const int64_t grp = chain ? 1 : Hq / Hkv;
  const int64_t C = chain ? 0 : bg.cfg.attn_chunks;
  const int64_t Nqkv = chain ? 0 : (Hq + 2 * Hkv) * d;
  const int64_t Fa = std::max(s.ffn, s.chain_ffn);
  *A = ActLayout{};
  int64_t off = 0;
  auto take = [&](int64_t bytes) {
    const int64_t o = off;
    off += round_up64(bytes, 256);
    return o;
  };
  A->o_h = take(B * h * 2);
  A->o_qkv = take(B * Nqkv * 2);
  A->o_opart = take(B * Hkv * C * grp * (d + 2) * 4);
  A->o_attn = take(B * Hq * d * 2);
  A->o_o = take(B * h * 2);
  A->o_hmid = take(B * h * 2);
  A->o_act = take(B * Fa * 2);
  A->o_dout = take(B * h * 2);
  A->layer_stride = off;
  const int64_t nblocks = std::max(s.n_layers, 1) + 1;
  A->global_block = A->layer_stride * nblocks;
  int64_t goff = 0;
  A->g_z = goff;
  goff += round_up64(B * h * 2, 256);
  A->g_amax = goff;
  goff += round_up64(B * lm_head_tiles(bg) * 8, 256);
  return A->global_block + goff;
}

int64_t merge_counters(const BuiltGraph& bg) {
  const mpk_model_shape& s = bg.cfg.shape;
  if (s.chain_ffn > 0) return 1;
  return (int64_t)s.n_layers * bg.cfg.batch * s.n_kv_heads;
}

int64_t rope_table_floats(const mpk_model_shape& s) {
  if (s.chain_ffn > 0) return 0;
  return (int64_t)s.max_pages_per_seq * s.page_size * (s.head_dim / 2) * 2;
}

void rope_table(const mpk_model_shape& s, float* cs) {
  const int max_ctx = s.max_pages_per_seq * s.page_size, d = s.head_dim;
  for (int p = 0; p < max_ctx; ++p)
    for (int i = 0; i < d / 2; ++i) {
      const double inv = std::pow((double)s.rope_theta, -2.0 * i / d);
      const double ang = (double)p * inv;
      cs[((size_t)p * (d / 2) + i) * 2] = (float)std::cos(ang);
      cs[((size_t)p * (d / 2) + i) * 2 + 1] = (float)std::sin(ang);
    }
}

uint8_t task_flags(const BuiltGraph& bg, int kind, int tile) {
  if (tile != 0) return 0;
  if (kind == MPK_TASK_QKV || kind == MPK_TASK_GATEUP) return TASK_F_RESIDUAL;
  if (kind == MPK_TASK_LM_HEAD && bg.cfg.shape.chain_ffn == 0)
    return TASK_F_RESIDUAL;
  return 0;
}

}  // namespace mpk
