"""Oracle decode step: plain NumPy, fp32 math on bf16-rounded tensors.
TEST INFRASTRUCTURE ONLY (see the package docstring).

What the step computes is the standard decoder step; MPK only schedules it
differently and is semantics-equivalent by construction (MPK summary,
§5 "Numerical considerations").  The precision contract is bf16 inputs and
outputs with an FP32 accumulator and round-to-nearest-even (MPK summary, §3
"Target operation, shapes & precision contract").  Every tensor that crosses
an operator boundary is rounded to bf16; logits stay fp32.

Readings taken where the pages are silent:
  * RMSNorm rounds once, after the multiply by the gain;
  * RoPE is the rotate-half form, pair (i, i + d/2), angle pos * theta^(-2i/d);
    the angle and its cos/sin are evaluated in float64, the rotation in fp32;
  * Qwen3-style per-head RMSNorm of q and k (``qk_norm``) precedes RoPE;
  * query head j reads KV head j // (Hq / Hkv) (grouped-query attention);
  * the new token's K/V are written at position seq_len[b] before attention,
    which then covers positions 0 .. seq_len[b] inclusive;
  * SwiGLU: a = silu(g) * u with g, u each rounded to bf16 first;
  * greedy argmax takes the lowest index among equal maxima.

Arrays: bf16 tensors are numpy ``uint16`` bit patterns.
"""
from __future__ import annotations

import math
from typing import Dict, Optional

import numpy as np

F32 = np.float32


# ------------------------------------------------------------------ bf16 I/O
def bf16_to_f32(u: np.ndarray) -> np.ndarray:
    """Widen bf16 bits to float32 (exact)."""
    return (np.asarray(u, dtype=np.uint16).astype(np.uint32) << 16).view(F32)


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 bits, round-to-nearest-even (MPK summary, §3
    precision contract "RNE").  NaN stays NaN (quiet)."""
    x = np.ascontiguousarray(x, dtype=F32)
    u = x.view(np.uint32)
    lsb = (u >> 16) & np.uint32(1)
    r = ((u + np.uint32(0x7FFF) + lsb) >> 16).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        r = np.where(nan, ((u >> 16) | np.uint32(0x40)).astype(np.uint16), r)
    return r


def round_bf16(x: np.ndarray) -> np.ndarray:
    """float32 -> nearest bf16 value, returned as float32."""
    return bf16_to_f32(f32_to_bf16(x))


# -------------------------------------------------------------- elementwise
def rmsnorm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm over the last axis: x * (mean(x^2) + eps)^-1/2 * w, fp32 from
    bf16 inputs, one rounding to bf16 at the end.  (The elementwise "E"
    tasks of MPK summary, Figure 1.)  x, w: bf16 bits; returns bf16 bits."""
    xf = bf16_to_f32(x)
    wf = bf16_to_f32(w)
    ms = np.mean(xf * xf, axis=-1, keepdims=True, dtype=F32)
    r = F32(1.0) / np.sqrt(ms + F32(eps), dtype=F32)
    return f32_to_bf16((xf * r) * wf)


def silu(z: np.ndarray) -> np.ndarray:
    """silu(z) = z / (1 + e^-z), fp32."""
    z = np.asarray(z, dtype=F32)
    with np.errstate(over="ignore"):
        return z / (F32(1.0) + np.exp(-z, dtype=F32))


def swiglu(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    """a = silu(g) * u on bf16 g, u; fp32 math, bf16 result."""
    return f32_to_bf16(silu(bf16_to_f32(g)) * bf16_to_f32(u))


def residual_add(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """bf16 + bf16 in fp32, rounded to bf16."""
    return f32_to_bf16(bf16_to_f32(a) + bf16_to_f32(b))


# ------------------------------------------------------------------- linear
# Accumulator of every MatMul: float32 (the pages' contract) by default.
# ``set_accumulator(np.float64)`` selects an exact-in-practice accumulator;
# the two variants differ only in rounding order and are used to measure the
# rounding-order noise of the whole bf16 pipeline.
_ACC = np.float32


def set_accumulator(dtype) -> None:
    global _ACC
    _ACC = np.dtype(dtype).type


def linear(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """y = x . W^T with bf16 operands and an FP32 accumulator (MPK summary,
    §3: MatMul task, "bf16 input/output, FP32 accumulator").  x: [B, K] bf16
    bits, W: [N, K] bf16 bits (row-major, one output per row).  Returns the
    unrounded fp32 [B, N]; callers round where the tensor crosses a
    boundary."""
    xf = bf16_to_f32(x)
    wf = bf16_to_f32(w)
    if _ACC is not F32:
        xf = xf.astype(_ACC)
        wf = wf.astype(_ACC)
    return np.matmul(xf, wf.T).astype(F32)


# ----------------------------------------------------------------- position
def rope(x: np.ndarray, pos, theta: float) -> np.ndarray:
    """Rotate-half rotary embedding on the last axis (size d).
    x: fp32 [..., d]; pos: int or int array broadcastable to x[..., 0].
    For i < d/2: (x_i, x_{i+d/2}) -> (x_i c - x_{i+d/2} s, x_{i+d/2} c + x_i s)
    with c, s = cos, sin(pos * theta^(-2i/d)).  Returns fp32."""
    x = np.asarray(x, dtype=F32)
    d = x.shape[-1]
    half = d // 2
    inv = theta ** (-2.0 * np.arange(half, dtype=np.float64) / d)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * inv
    c = np.cos(ang).astype(F32)
    s = np.sin(ang).astype(F32)
    x1 = x[..., :half]
    x2 = x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


# ---------------------------------------------------------------- attention
def gather_kv(pool: np.ndarray, page_table_row: np.ndarray, layer: int,
              kv_head: int, n: int) -> np.ndarray:
    """Tokens 0..n-1 of one sequence and KV head from the paged pool
    [L][pages][Hkv][page_size][d]; token t lives in page
    page_table[t // page_size] at slot t % page_size.  Returns bf16 [n, d]."""
    P = pool.shape[3]
    t = np.arange(n)
    pages = page_table_row[t // P]
    if n and (pages < 0).any():
        raise ValueError("unmapped KV page")
    return pool[layer, pages, kv_head, t % P, :]


def attention_decode(q: np.ndarray, k: np.ndarray, v: np.ndarray
                     ) -> np.ndarray:
    """Single-query attention, naive softmax (every score materialised).
    q: bf16 [Hg, d] (the query heads that share one KV head); k, v: bf16
    [n, d].  s = q.k / sqrt(d), p = exp(s - max s) / sum, o = sum p v, all
    fp32.  Returns fp32 [Hg, d] (unrounded) -- paged-attention decode
    (MPK summary, §3: Attention task)."""
    qf = bf16_to_f32(q)
    kf = bf16_to_f32(k)
    vf = bf16_to_f32(v)
    d = qf.shape[-1]
    s = np.matmul(qf, kf.T).astype(F32) * F32(1.0 / math.sqrt(d))
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m, dtype=F32)
    p = e / np.sum(e, axis=-1, keepdims=True, dtype=F32)
    return np.matmul(p, vf).astype(F32)


def attention_probs(q: np.ndarray, k: np.ndarray) -> np.ndarray:
    """The softmax rows of ``attention_decode`` (for the row-sum check)."""
    qf = bf16_to_f32(q)
    kf = bf16_to_f32(k)
    s = np.matmul(qf, kf.T).astype(F32) * F32(1.0 / math.sqrt(qf.shape[-1]))
    e = np.exp(s - np.max(s, axis=-1, keepdims=True), dtype=F32)
    return e / np.sum(e, axis=-1, keepdims=True, dtype=F32)


# ------------------------------------------------------------------ argmax
def argmax_lowest(logits: np.ndarray) -> np.ndarray:
    """Greedy next token per row: the lowest index among equal maxima."""
    return np.argmax(logits, axis=-1).astype(np.int32)


# --------------------------------------------------------------- the step
def _split_qkv(qkv: np.ndarray, shape):
    B = qkv.shape[0]
    Hq, Hkv, d = shape.n_q_heads, shape.n_kv_heads, shape.head_dim
    q = qkv[:, :Hq * d].reshape(B, Hq, d)
    k = qkv[:, Hq * d:(Hq + Hkv) * d].reshape(B, Hkv, d)
    v = qkv[:, (Hq + Hkv) * d:].reshape(B, Hkv, d)
    return q, k, v


def layer_step(shape, W: Dict[str, np.ndarray], l: int, x: np.ndarray,
               k_pool: np.ndarray, v_pool: np.ndarray,
               page_table: np.ndarray, seq_lens: np.ndarray) -> np.ndarray:
    """One decoder layer for a batch of single-token rows.  x: bf16 [B, h].
    Writes this token's K/V into the pools (in place).  Returns bf16 [B, h].
    """
    Hq, Hkv, d = shape.n_q_heads, shape.n_kv_heads, shape.head_dim
    grp = Hq // Hkv
    P = k_pool.shape[3]
    n1 = rmsnorm(x, W[f"layer{l}.ln1"], shape.rms_eps)
    qkv = f32_to_bf16(linear(n1, W[f"layer{l}.wqkv"]))
    q, k, v = _split_qkv(qkv, shape)
    if shape.qk_norm:
        q = rmsnorm(q, W[f"layer{l}.q_norm"], shape.rms_eps)
        k = rmsnorm(k, W[f"layer{l}.k_norm"], shape.rms_eps)
    pos = seq_lens.astype(np.int64)
    q = f32_to_bf16(rope(bf16_to_f32(q), pos[:, None], shape.rope_theta))
    k = f32_to_bf16(rope(bf16_to_f32(k), pos[:, None], shape.rope_theta))
    B = x.shape[0]
    attn = np.empty((B, Hq * d), dtype=np.uint16)
    for b in range(B):
        p = int(pos[b])
        page = page_table[b, p // P]
        if page < 0:
            raise ValueError("unmapped KV page for the new token")
        k_pool[l, page, :, p % P, :] = k[b]
        v_pool[l, page, :, p % P, :] = v[b]
        for g in range(Hkv):
            kk = gather_kv(k_pool, page_table[b], l, g, p + 1)
            vv = gather_kv(v_pool, page_table[b], l, g, p + 1)
            o = attention_decode(q[b, g * grp:(g + 1) * grp], kk, vv)
            attn[b, g * grp * d:(g + 1) * grp * d] = f32_to_bf16(o).reshape(-1)
    o = f32_to_bf16(linear(attn, W[f"layer{l}.wo"]))
    h = residual_add(x, o)
    n2 = rmsnorm(h, W[f"layer{l}.ln2"], shape.rms_eps)
    F = shape.ffn
    wgu = W[f"layer{l}.wgu"]
    g_ = f32_to_bf16(linear(n2, wgu[:F]))
    u_ = f32_to_bf16(linear(n2, wgu[F:]))
    a = swiglu(g_, u_)
    dn = f32_to_bf16(linear(a, W[f"layer{l}.wd"]))
    return residual_add(h, dn)


def decode_step(shape, W: Dict[str, np.ndarray], tokens: np.ndarray,
                k_pool: Optional[np.ndarray], v_pool: Optional[np.ndarray],
                page_table: Optional[np.ndarray],
                seq_lens: Optional[np.ndarray],
                layers: Optional[range] = None) -> Dict[str, np.ndarray]:
    """One greedy decode step (MPK summary, Q1: "tiny batch (1-16), 1 token
    per step").  Updates k_pool, v_pool and seq_lens in place (seq_lens += 1)
    and returns {"hidden": [per-layer bf16 outputs], "logits": fp32 [B, V],
    "next_tokens": int32 [B]}.

    ``layers`` restricts the layer loop (used only to time a bounded sample);
    the default runs every layer."""
    x = W["embed"][np.asarray(tokens, dtype=np.int64)]
    hidden = []
    if shape.is_chain:
        n = rmsnorm(x, W["final_norm"], shape.rms_eps)
        h1 = f32_to_bf16(linear(n, W["chain_w1"]))
        y = f32_to_bf16(silu(bf16_to_f32(h1)))
        z = f32_to_bf16(linear(y, W["chain_w2"]))
        hidden = [n, y, z]
        logits = linear(z, W["lm_head"])
    else:
        for l in (layers if layers is not None else range(shape.n_layers)):
            x = layer_step(shape, W, l, x, k_pool, v_pool, page_table,
                           seq_lens)
            hidden.append(x)
        nf = rmsnorm(x, W["final_norm"], shape.rms_eps)
        hidden.append(nf)
        logits = linear(nf, W["lm_head"])
        seq_lens += 1
    return {"hidden": hidden, "logits": logits,
            "next_tokens": argmax_lowest(logits)}


# ------------------------------------------- full-sequence (prefill) forward
def forward_sequence(shape, W: Dict[str, np.ndarray], token_ids: np.ndarray
                     ) -> Dict[str, np.ndarray]:
    """Causal forward over a whole sequence (one batch row), contiguous K/V,
    no paging.  Row t attends to positions 0..t and is rotated at position
    t.  Returns the fp32 logits [n, V] and the bf16 K/V per layer
    ([L][n][Hkv][d]).  Used to check that a decode step equals the last row
    of the full-sequence forward."""
    Hq, Hkv, d = shape.n_q_heads, shape.n_kv_heads, shape.head_dim
    grp = Hq // Hkv
    x = W["embed"][np.asarray(token_ids, dtype=np.int64)]
    n = x.shape[0]
    pos = np.arange(n)
    ks, vs = [], []
    for l in range(shape.n_layers):
        n1 = rmsnorm(x, W[f"layer{l}.ln1"], shape.rms_eps)
        qkv = f32_to_bf16(linear(n1, W[f"layer{l}.wqkv"]))
        q, k, v = _split_qkv(qkv, shape)
        if shape.qk_norm:
            q = rmsnorm(q, W[f"layer{l}.q_norm"], shape.rms_eps)
            k = rmsnorm(k, W[f"layer{l}.k_norm"], shape.rms_eps)
        q = f32_to_bf16(rope(bf16_to_f32(q), pos[:, None], shape.rope_theta))
        k = f32_to_bf16(rope(bf16_to_f32(k), pos[:, None], shape.rope_theta))
        ks.append(k)
        vs.append(v)
        attn = np.empty((n, Hq * d), dtype=np.uint16)
        for t in range(n):
            for g in range(Hkv):
                o = attention_decode(q[t, g * grp:(g + 1) * grp],
                                     k[:t + 1, g], v[:t + 1, g])
                attn[t, g * grp * d:(g + 1) * grp * d] = \
                    f32_to_bf16(o).reshape(-1)
        o = f32_to_bf16(linear(attn, W[f"layer{l}.wo"]))
        h = residual_add(x, o)
        n2 = rmsnorm(h, W[f"layer{l}.ln2"], shape.rms_eps)
        F = shape.ffn
        g_ = f32_to_bf16(linear(n2, W[f"layer{l}.wgu"][:F]))
        u_ = f32_to_bf16(linear(n2, W[f"layer{l}.wgu"][F:]))
        dn = f32_to_bf16(linear(swiglu(g_, u_), W[f"layer{l}.wd"]))
        x = residual_add(h, dn)
    nf = rmsnorm(x, W["final_norm"], shape.rms_eps)
    return {"logits": linear(nf, W["lm_head"]), "k": ks, "v": vs}


# ------------------------------------------------------ attention partials
def attention_partial(q: np.ndarray, k: np.ndarray, v: np.ndarray):
    """Un-normalised attention over one slice of the keys: returns
    (m, l, acc) with m = max score, l = sum exp(s - m), acc = sum exp(s-m) v,
    fp32.  A split of the keys followed by ``merge_partials`` equals
    ``attention_decode`` (the split-KV reading of the paged-attention task
    taken for decode with few KV heads)."""
    qf = bf16_to_f32(q)
    kf = bf16_to_f32(k)
    vf = bf16_to_f32(v)
    s = np.matmul(qf, kf.T).astype(F32) * F32(1.0 / math.sqrt(qf.shape[-1]))
    if s.shape[-1] == 0:
        return (np.full(qf.shape[0], -np.inf, F32), np.zeros(qf.shape[0], F32),
                np.zeros_like(qf))
    m = np.max(s, axis=-1)
    e = np.exp(s - m[:, None], dtype=F32)
    return m, np.sum(e, axis=-1, dtype=F32), np.matmul(e, vf).astype(F32)


def merge_partials(parts):
    """Log-sum-exp merge of (m, l, acc) partials: M = max m_c,
    L = sum l_c e^(m_c - M), o = sum acc_c e^(m_c - M) / L."""
    ms = np.stack([p[0] for p in parts])
    M = np.max(ms, axis=0)
    wts = [np.where(np.isfinite(p[0]), np.exp(p[0] - M, dtype=F32), F32(0))
           for p in parts]
    L = sum(w * p[1] for w, p in zip(wts, parts))
    acc = sum(w[:, None] * p[2] for w, p in zip(wts, parts))
    return (acc / L[:, None]).astype(F32)
