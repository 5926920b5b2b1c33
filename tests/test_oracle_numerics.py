"""Pins for the oracle's decode-step numerics (CPU only).

Each check ties the oracle to something other than itself: a library routine
(torch in float64), a closed form, an invariant or a special case.  Sizes are
small so the whole file runs in seconds."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as Fn

from oracle import numerics as nx
from task_graph_runtime_gb300 import synth

RNG = np.random.default_rng(1234)


def bits_to_torch64(u):
    return torch.from_numpy(np.ascontiguousarray(u).view(np.int16)).view(
        torch.bfloat16).to(torch.float64)


def rand_bf16(shape, std=1.0):
    return nx.f32_to_bf16((RNG.standard_normal(shape) * std).astype(np.float32))


# ------------------------------------------------------------------ bf16
def test_bf16_rne_matches_torch_conversion():
    x = np.concatenate([
        RNG.standard_normal(100000).astype(np.float32) * 10,
        # exact ties: 1 + 2^-8 and 1 + 3*2^-8 lie halfway between bf16 values
        np.array([1 + 2**-8, 1 + 3 * 2**-8, -(1 + 2**-8), 2**-130, 3e38,
                  np.inf, -np.inf, 0.0, -0.0], dtype=np.float32)])
    ours = nx.f32_to_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy() \
        .view(np.uint16)
    assert np.array_equal(ours, ref)
    # ties go to the even mantissa
    assert nx.bf16_to_f32(nx.f32_to_bf16(np.float32(1 + 2**-8))) == 1.0
    assert nx.bf16_to_f32(nx.f32_to_bf16(np.float32(1 + 3 * 2**-8))) == \
        np.float32(1 + 2**-6)
    assert np.isnan(nx.bf16_to_f32(nx.f32_to_bf16(np.float32(np.nan))))


def test_bf16_widen_is_exact():
    u = np.arange(0, 65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(u.view(np.int16)).view(torch.bfloat16).to(
        torch.float32).numpy()
    ours = nx.bf16_to_f32(u)
    same = (ours == ref) | (np.isnan(ours) & np.isnan(ref))
    assert same.all()


# ---------------------------------------------------------------- RMSNorm
def test_rmsnorm_matches_torch_rms_norm():
    x = rand_bf16((8, 512))
    w = nx.f32_to_bf16(1 + 0.02 * RNG.standard_normal(512).astype(np.float32))
    ours = nx.bf16_to_f32(nx.rmsnorm(x, w, 1e-6)).astype(np.float64)
    ref = Fn.rms_norm(bits_to_torch64(x), (512,), weight=bits_to_torch64(w),
                      eps=1e-6).numpy()
    # one bf16 rounding: at most one ulp (2^-8 relative) apart
    assert np.all(np.abs(ours - ref) <= 2**-8 * np.abs(ref) + 1e-30)


def test_rmsnorm_constant_vector_gives_gain():
    for c in (0.5, -3.0, 7.25):
        x = nx.f32_to_bf16(np.full((1, 256), c, dtype=np.float32))
        w = rand_bf16((256,))
        y = nx.bf16_to_f32(nx.rmsnorm(x, w, 0.0))
        assert np.array_equal(y, np.sign(c) * nx.bf16_to_f32(w)[None])


def test_rmsnorm_scale_invariant():
    x = rand_bf16((4, 256))
    w = rand_bf16((256,))
    x2 = nx.f32_to_bf16(nx.bf16_to_f32(x) * np.float32(4.0))  # exact in bf16
    assert np.array_equal(nx.rmsnorm(x, w, 0.0), nx.rmsnorm(x2, w, 0.0))


# ----------------------------------------------------------------- linear
def test_linear_matches_float64_within_fp32_bound():
    K, N = 1000, 37
    x = rand_bf16((3, K))
    W = rand_bf16((N, K), 0.02)
    ours = nx.linear(x, W).astype(np.float64)
    ref = Fn.linear(bits_to_torch64(x), bits_to_torch64(W)).numpy()
    absdot = np.abs(nx.bf16_to_f32(x)).astype(np.float64) @ \
        np.abs(nx.bf16_to_f32(W)).astype(np.float64).T
    bound = K * 2.0**-24 * absdot           # gamma_K for fp32 accumulation
    assert np.all(np.abs(ours - ref) <= bound)


def test_linear_basis_vector_selects_column():
    K, N = 64, 24                   # non-square: a transposed W would fail
    W = rand_bf16((N, K))
    for k in (0, 5, 63):
        x = np.zeros((1, K), dtype=np.float32)
        x[0, k] = 1.0
        y = nx.linear(nx.f32_to_bf16(x), W)
        assert np.array_equal(y[0], nx.bf16_to_f32(W[:, k]))


# ------------------------------------------------------------------- RoPE
def test_rope_equals_complex_rotation():
    d = 64
    x = RNG.standard_normal((5, d)).astype(np.float32)
    pos = np.array([0, 1, 17, 2048, 4100])
    theta = 1e6
    ours = nx.rope(x, pos, theta).astype(np.float64)
    z = x[:, :d // 2].astype(np.float64) + 1j * x[:, d // 2:]
    freq = theta ** (-np.arange(0, d, 2, dtype=np.float64) / d)
    zr = z * np.exp(1j * pos[:, None] * freq[None])
    ref = np.concatenate([zr.real, zr.imag], axis=1)
    assert np.allclose(ours, ref, rtol=0, atol=4e-6 * np.abs(ref).max())


def test_rope_position_zero_is_identity_and_norms_preserved():
    x = RNG.standard_normal((3, 128)).astype(np.float32)
    assert np.array_equal(nx.rope(x, 0, 1e4), x)
    y = nx.rope(x, 1234, 1e4)
    pair_in = x[:, :64] ** 2 + x[:, 64:] ** 2
    pair_out = y[:, :64] ** 2 + y[:, 64:] ** 2
    assert np.allclose(pair_in, pair_out, rtol=1e-5, atol=1e-6)


def test_rope_scores_depend_on_relative_position_only():
    q = RNG.standard_normal(64).astype(np.float32)
    k = RNG.standard_normal(64).astype(np.float32)
    a = np.dot(nx.rope(q, 10, 1e4), nx.rope(k, 3, 1e4))
    b = np.dot(nx.rope(q, 1010, 1e4), nx.rope(k, 1003, 1e4))
    assert abs(a - b) < 1e-3


# -------------------------------------------------------------- attention
def test_attention_matches_torch_sdpa_gqa():
    Hq, Hkv, d, n = 8, 2, 64, 77
    q = rand_bf16((Hq, d))
    k = rand_bf16((n, Hkv, d))
    v = rand_bf16((n, Hkv, d))
    grp = Hq // Hkv
    ours = np.concatenate([nx.attention_decode(q[g * grp:(g + 1) * grp],
                                               k[:, g], v[:, g])
                           for g in range(Hkv)])
    Q = bits_to_torch64(q)[None, :, None, :]          # [1, Hq, 1, d]
    Kt = bits_to_torch64(k).permute(1, 0, 2)[None]    # [1, Hkv, n, d]
    Vt = bits_to_torch64(v).permute(1, 0, 2)[None]
    ref = Fn.scaled_dot_product_attention(Q, Kt, Vt, enable_gqa=True)[0, :, 0]
    assert np.allclose(ours, ref.numpy(), rtol=0, atol=2e-5)


def test_attention_softmax_rows_sum_to_one():
    q = rand_bf16((4, 128))
    k = rand_bf16((300, 128), 3.0)
    p = nx.attention_probs(q, k)
    assert np.allclose(p.sum(-1), 1.0, atol=1e-5)
    assert (p >= 0).all()


def test_attention_single_token_returns_v():
    q = rand_bf16((4, 64))
    k = rand_bf16((1, 64))
    v = rand_bf16((1, 64))
    o = nx.attention_decode(q, k, v)
    assert np.array_equal(o, np.repeat(nx.bf16_to_f32(v), 4, axis=0))


def test_attention_equal_keys_average_values():
    q = rand_bf16((2, 64))
    k = np.repeat(rand_bf16((1, 64)), 40, axis=0)
    v = rand_bf16((40, 64))
    o = nx.attention_decode(q, k, v)
    ref = nx.bf16_to_f32(v).astype(np.float64).mean(0)
    assert np.allclose(o, np.repeat(ref[None], 2, 0), atol=1e-5)


def test_paged_gather_equals_contiguous_under_permutation():
    L, Hkv, P, d, n = 2, 3, 16, 32, 70
    pages = -(-n // P)
    contig = rand_bf16((L, n, Hkv, d))
    perm = RNG.permutation(pages + 5)[:pages]
    pool = np.zeros((L, pages + 5, Hkv, P, d), dtype=np.uint16)
    for t in range(n):
        pool[:, perm[t // P], :, t % P] = contig[:, t]
    table = np.full(pages + 2, -1, dtype=np.int32)
    table[:pages] = perm
    for l in range(L):
        for g in range(Hkv):
            assert np.array_equal(nx.gather_kv(pool, table, l, g, n),
                                  contig[l, :, g])
    with pytest.raises(ValueError):
        nx.gather_kv(pool, table, 0, 0, (pages + 1) * P)


def test_split_kv_merge_equals_naive_softmax():
    q = rand_bf16((4, 128))
    k = rand_bf16((513, 128), 2.0)
    v = rand_bf16((513, 128))
    full = nx.attention_decode(q, k, v)
    for cuts in ([0, 513], [0, 100, 513], [0, 1, 2, 300, 512, 513],
                 [0, 0, 200, 513]):
        parts = [nx.attention_partial(q, k[a:b], v[a:b])
                 for a, b in zip(cuts[:-1], cuts[1:])]
        assert np.allclose(nx.merge_partials(parts), full, atol=2e-6)


# ---------------------------------------------------------- SiLU, argmax
def test_silu_matches_torch():
    z = (RNG.standard_normal(10000) * 8).astype(np.float32)
    ref = Fn.silu(torch.from_numpy(z).double()).numpy()
    assert np.allclose(nx.silu(z), ref, rtol=2e-6, atol=1e-30)
    assert nx.silu(np.float32(0.0)) == 0.0
    assert nx.silu(np.float32(-200.0)) == 0.0


def test_argmax_lowest_index_on_ties():
    x = np.array([[1.0, 3.0, 3.0, 2.0], [5.0, 5.0, 5.0, 5.0]], np.float32)
    assert nx.argmax_lowest(x).tolist() == [1, 0]


# ------------------------------------------------------ whole decode step
SMALL = synth.ModelShape(2, 128, 4, 2, 32, 192, 256, 1e-6, 1e4, True)


def _paged_from_contiguous(ks, vs, n, page, extra_pages, seed):
    L = len(ks)
    Hkv, d = ks[0].shape[1], ks[0].shape[2]
    pages = -(-(n + 1) // page)
    rng = np.random.default_rng(seed)
    perm = rng.permutation(pages + extra_pages)[:pages].astype(np.int32)
    kp = np.zeros((L, pages + extra_pages, Hkv, page, d), np.uint16)
    vp = np.zeros_like(kp)
    for l in range(L):
        for t in range(n):
            kp[l, perm[t // page], :, t % page] = ks[l][t]
            vp[l, perm[t // page], :, t % page] = vs[l][t]
    return kp, vp, perm[None]


@pytest.mark.parametrize("shape", [SMALL, synth.TINY])
def test_decode_step_equals_last_row_of_full_forward(shape):
    """A decode step with the KV cache of the first n-1 tokens equals the
    last row of the causal full-sequence forward (contiguous, unpaged)."""
    W = synth.model_weights(shape, base_seed=7)
    n = 21
    toks = np.random.default_rng(3).integers(0, shape.vocab, n).astype(
        np.int32)
    full = nx.forward_sequence(shape, W, toks)
    prefix = nx.forward_sequence(shape, W, toks[:-1])
    kp, vp, table = _paged_from_contiguous(prefix["k"], prefix["v"], n - 1, 8,
                                           3, 11)
    seq = np.array([n - 1], np.int32)
    out = nx.decode_step(shape, W, toks[-1:], kp, vp, table, seq)
    ref = full["logits"][-1]
    got = out["logits"][0]
    assert np.abs(got - ref).max() <= 2e-2 * np.abs(ref).max() + 1e-3
    assert seq[0] == n
    # the new token's K/V landed in the slot the page table names
    for l in range(shape.n_layers):
        assert np.array_equal(kp[l, table[0, (n - 1) // 8], :, (n - 1) % 8],
                              full["k"][l][n - 1])


def _torch_reference_logits(shape, W, tokens, ks, vs):
    """float64 torch model from library ops: embedding, rms_norm, linear,
    SDPA with grouped-query heads, SiLU; RoPE as complex multiplication."""
    T = lambda a: bits_to_torch64(a)
    Hq, Hkv, d = shape.n_q_heads, shape.n_kv_heads, shape.head_dim
    eps = shape.rms_eps
    x = Fn.embedding(torch.from_numpy(tokens.astype(np.int64)), T(W["embed"]))
    n = x.shape[0]
    freq = shape.rope_theta ** (-torch.arange(0, d, 2, dtype=torch.float64) / d)
    ang = torch.arange(n, dtype=torch.float64)[:, None] * freq[None]
    rot = torch.polar(torch.ones_like(ang), ang)          # [n, d/2]

    def rope(t):                                          # [n, H, d]
        z = torch.complex(t[..., :d // 2], t[..., d // 2:]) * rot[:, None]
        return torch.cat([z.real, z.imag], -1)

    for l in range(shape.n_layers):
        h1 = Fn.rms_norm(x, (shape.hidden,), T(W[f"layer{l}.ln1"]), eps)
        qkv = Fn.linear(h1, T(W[f"layer{l}.wqkv"]))
        q = qkv[:, :Hq * d].reshape(n, Hq, d)
        k = qkv[:, Hq * d:(Hq + Hkv) * d].reshape(n, Hkv, d)
        v = qkv[:, (Hq + Hkv) * d:].reshape(n, Hkv, d)
        if shape.qk_norm:
            q = Fn.rms_norm(q, (d,), T(W[f"layer{l}.q_norm"]), eps)
            k = Fn.rms_norm(k, (d,), T(W[f"layer{l}.k_norm"]), eps)
        q, k = rope(q), rope(k)
        a = Fn.scaled_dot_product_attention(
            q.permute(1, 0, 2)[None], k.permute(1, 0, 2)[None],
            v.permute(1, 0, 2)[None], is_causal=True, enable_gqa=True)
        a = a[0].permute(1, 0, 2).reshape(n, Hq * d)
        x = x + Fn.linear(a, T(W[f"layer{l}.wo"]))
        h2 = Fn.rms_norm(x, (shape.hidden,), T(W[f"layer{l}.ln2"]), eps)
        F = shape.ffn
        gu = Fn.linear(h2, T(W[f"layer{l}.wgu"]))
        x = x + Fn.linear(Fn.silu(gu[:, :F]) * gu[:, F:], T(W[f"layer{l}.wd"]))
    hf = Fn.rms_norm(x, (shape.hidden,), T(W["final_norm"]), eps)
    return Fn.linear(hf, T(W["lm_head"])).numpy()


@pytest.mark.parametrize("shape", [SMALL, synth.TINY])
def test_full_forward_matches_torch_float64_model(shape):
    W = synth.model_weights(shape, base_seed=5)
    toks = np.random.default_rng(9).integers(0, shape.vocab, 12).astype(
        np.int32)
    ours = nx.forward_sequence(shape, W, toks)["logits"]
    ref = _torch_reference_logits(shape, W, toks, None, None)
    assert np.abs(ours - ref).max() <= 2e-2 * np.abs(ref).max() + 1e-3


def test_chain_step_matches_torch_float64():
    shape = synth.ModelShape(0, 128, 1, 1, 32, 0, 300, chain_ffn=256)
    W = synth.model_weights(shape, base_seed=2)
    toks = np.array([3, 77, 299], np.int32)
    out = nx.decode_step(shape, W, toks, None, None, None, None)
    T = bits_to_torch64
    x = Fn.embedding(torch.from_numpy(toks.astype(np.int64)), T(W["embed"]))
    x = Fn.rms_norm(x, (128,), T(W["final_norm"]), shape.rms_eps)
    y = Fn.silu(Fn.linear(x, T(W["chain_w1"])))
    ref = Fn.linear(Fn.linear(y, T(W["chain_w2"])), T(W["lm_head"])).numpy()
    assert np.abs(out["logits"] - ref).max() <= 2e-2 * np.abs(ref).max() + 1e-3


def test_float64_accumulator_is_closer_to_exact():
    """The float64 accumulator variant agrees with torch float64 to fp64
    rounding, and the default (float32) stays within its gamma_K bound."""
    K = 4096
    x = rand_bf16((2, K))
    W = rand_bf16((16, K), 0.02)
    ref = Fn.linear(bits_to_torch64(x), bits_to_torch64(W)).numpy()
    try:
        nx.set_accumulator(np.float64)
        y64 = nx.linear(x, W).astype(np.float64)
    finally:
        nx.set_accumulator(np.float32)
    assert np.all(np.abs(y64 - ref) <= 2**-24 * np.abs(ref) + 1e-30)
