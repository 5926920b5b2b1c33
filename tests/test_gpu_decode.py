"""Decode-step parity on the GPU: the C-ABI library (megakernel and
kernel-per-operator modes) against the oracle, on the same seeded inputs.

Bound (hidden states and logits): |gpu - ref| <= 2e-2 * max|ref| + 1e-3.
Greedy tokens must match except where the oracle's top-2 logit gap is
below 1e-2.  Megakernel and kernel-per-operator run the same task bodies
with fixed reduction orders, so their outputs must agree bit for bit."""
import dataclasses

import numpy as np
import pytest
import torch

from oracle import numerics as nx
from task_graph_runtime_gb300 import mpk, synth

from gpu_util import (bf16_to_f32, dev_kv, dev_weights, to_dev,
                      tokens_agree, within_bound)

pytestmark = pytest.mark.gpu


def _graph(wl, batch=None, **kw):
    return mpk.Graph(wl.shape, batch or wl.batch, page_size=wl.page_size,
                     max_pages_per_seq=max(1, wl.max_pages_per_seq), **kw)


def _outputs(B, V):
    return (torch.empty(B, V, dtype=torch.float32, device="cuda"),
            torch.empty(B, dtype=torch.int32, device="cuda"))


def run_gpu(wl, W_dev, kv_host, tokens, steps=1, mode=mpk.MODE_MEGAKERNEL,
            **kw):
    """Run `steps` greedy steps; returns per-step (logits, tokens) and the
    final device KV cache."""
    g = _graph(wl, **kw)
    g.bind(W_dev)
    g.set_mode(mode)
    kv = dev_kv(kv_host) if kv_host is not None else None
    tok = torch.from_numpy(np.asarray(tokens, np.int32)).cuda()
    out = []
    for _ in range(steps):
        logits, nxt = _outputs(wl.batch, wl.shape.vocab)
        g.decode_step(tok, kv, logits, nxt)
        torch.cuda.synchronize()
        assert g.status() == mpk.MPK_OK, mpk.STATUS_NAMES[g.status()]
        out.append((logits.cpu().numpy(), nxt.cpu().numpy()))
        tok = nxt
    g.close()
    return out, kv


def run_oracle(wl, W, kv_host, tokens, steps=1):
    k = kv_host.k_pool.copy() if kv_host is not None else None
    v = kv_host.v_pool.copy() if kv_host is not None else None
    seq = kv_host.seq_lens.copy() if kv_host is not None else None
    pt = kv_host.page_table if kv_host is not None else None
    tok = np.asarray(tokens, np.int32)
    out = []
    for _ in range(steps):
        r = nx.decode_step(wl.shape, W, tok, k, v, pt, seq)
        out.append((r["logits"], r["next_tokens"]))
        tok = r["next_tokens"]
    return out, (k, v, seq)


def check_steps(gpu, ref):
    for s, ((gl, gt), (rl, rt)) in enumerate(zip(gpu, ref)):
        ok, err, lim = within_bound(gl, rl)
        assert ok, f"step {s}: logits err {err:.3e} > {lim:.3e}"
        assert tokens_agree(gt, rl), f"step {s}: tokens {gt} vs {rt}"
        if not np.array_equal(gt, rt):
            break      # a near-tie picked another token: sequences diverge


def _inputs(wl, seed=0):
    W = synth.model_weights(wl.shape, seed)
    kv = synth.kv_inputs(wl, seed) if not wl.shape.is_chain else None
    return W, kv, synth.tokens(wl, seed)


# ----------------------------------------------------------------- tiny
@pytest.fixture(scope="module")
def tiny():
    wl = synth.WORKLOADS["tiny"]
    W, kv, tok = _inputs(wl)
    return wl, W, dev_weights(W, wl.shape), kv, tok


def test_tiny_one_step_matches_oracle(tiny):
    wl, W, Wd, kv, tok = tiny
    gpu, kvd = run_gpu(wl, Wd, kv, tok)
    ref, (k_ref, v_ref, seq_ref) = run_oracle(wl, W, kv, tok)
    check_steps(gpu, ref)
    assert np.array_equal(kvd.seq_lens.cpu().numpy(), seq_ref)
    # the new token's K/V in every layer, at the slot the page table names
    pos = int(kv.seq_lens[0])
    page = kv.page_table[0, pos // wl.page_size]
    kg = bf16_to_f32(kvd.k_pool)[:, page, :, pos % wl.page_size]
    vg = bf16_to_f32(kvd.v_pool)[:, page, :, pos % wl.page_size]
    kr = nx.bf16_to_f32(k_ref[:, page, :, pos % wl.page_size])
    vr = nx.bf16_to_f32(v_ref[:, page, :, pos % wl.page_size])
    assert within_bound(kg, kr)[0] and within_bound(vg, vr)[0]
    # nothing else in the pools changed
    kk = bf16_to_f32(kvd.k_pool)
    kk[:, page, :, pos % wl.page_size] = 0
    k0 = nx.bf16_to_f32(kv.k_pool).copy()
    k0[:, page, :, pos % wl.page_size] = 0
    assert np.array_equal(kk, k0)


def test_tiny_multi_step_greedy(tiny):
    wl, W, Wd, kv, tok = tiny
    gpu, _ = run_gpu(wl, Wd, kv, tok, steps=4)
    ref, _ = run_oracle(wl, W, kv, tok, steps=4)
    check_steps(gpu, ref)


@pytest.mark.parametrize("mode", [mpk.MODE_KPO, mpk.MODE_KPO_GRAPH])
def test_tiny_kernel_per_operator_bitwise_equal(tiny, mode):
    wl, W, Wd, kv, tok = tiny
    mega, kv_m = run_gpu(wl, Wd, kv, tok, steps=3)
    kpo, kv_k = run_gpu(wl, Wd, kv, tok, steps=3, mode=mode)
    for (ml, mt), (kl, kt) in zip(mega, kpo):
        assert np.array_equal(ml, kl) and np.array_equal(mt, kt)
    assert torch.equal(kv_m.k_pool, kv_k.k_pool)
    assert torch.equal(kv_m.v_pool, kv_k.v_pool)


@pytest.mark.parametrize("workers,rows,chunks,sched", [
    (4, 0, 0, (1, 1)),        # few workers: many tasks per worker
    (7, 40, 3, (2, 3)),       # ragged tiles, odd chunk count
    (0, 8, 1, (4, 4)),        # smallest tiles, one chunk (no split)
])
def test_tiny_tilings_match_oracle(tiny, workers, rows, chunks, sched):
    wl, W, Wd, kv, tok = tiny
    gpu, _ = run_gpu(wl, Wd, kv, tok, steps=2, num_workers=workers,
                     gemv_rows_per_task=rows, attn_chunks=chunks,
                     num_sched_sms=sched[0], sched_warps_per_sm=sched[1])
    ref, _ = run_oracle(wl, W, kv, tok, steps=2)
    check_steps(gpu, ref)


def test_tiny_coarse_events_match_oracle(tiny):
    """Operator-level events (the coarse-grained graph of the Figure 4c
    ablation: every task of an operator waits for all of the previous
    operator) compute the same step, through the megakernel and the
    kernel-per-operator build alike."""
    wl, W, Wd, kv, tok = tiny
    ref, _ = run_oracle(wl, W, kv, tok, steps=2)
    for mode in (mpk.MODE_MEGAKERNEL, mpk.MODE_KPO):
        gpu, _ = run_gpu(wl, Wd, kv, tok, steps=2, mode=mode, num_workers=5,
                         coarse_events=1)
        check_steps(gpu, ref)


def test_tiny_batch_ragged_contexts():
    """Three sequences with contexts 0, 37 and 128 (an empty prior context,
    a ragged last page, full pages) and more chunks than tokens."""
    base = synth.WORKLOADS["tiny"]
    wl = dataclasses.replace(base, name="tiny_b3", batch=3, ctx=(0, 37, 128),
                             steps=2)
    W, kv, tok = _inputs(wl, seed=3)
    gpu, _ = run_gpu(wl, dev_weights(W, wl.shape), kv, tok, steps=2,
                     attn_chunks=4)
    ref, _ = run_oracle(wl, W, kv, tok, steps=2)
    check_steps(gpu, ref)


def test_qk_norm_small_shape():
    """Per-head q/k RMSNorm (Qwen3-style) with head_dim 128."""
    shape = synth.ModelShape(2, 512, 8, 2, 128, 1024, 2048, 1e-6, 1e6, True)
    wl = synth.Workload("qk", shape, 2, (100, 31), 16, 2)
    W, kv, tok = _inputs(wl, seed=4)
    gpu, _ = run_gpu(wl, dev_weights(W, shape), kv, tok, steps=2)
    ref, _ = run_oracle(wl, W, kv, tok, steps=2)
    check_steps(gpu, ref)


def test_chain_small():
    shape = synth.ModelShape(0, 512, 1, 1, 32, 0, 3000, chain_ffn=1536)
    for B in (1, 8):
        wl = synth.Workload("chain_small", shape, B, (), 64, 1)
        W, _, tok = _inputs(wl, seed=5)
        gpu, _ = run_gpu(wl, dev_weights(W, shape), None, tok)
        ref, _ = run_oracle(wl, W, None, tok)
        check_steps(gpu, ref)


# ------------------------------------------------------- bounded waits
def test_unsatisfiable_event_times_out_and_recovers(tiny):
    wl, W, Wd, kv, tok = tiny
    g = _graph(wl)
    g.bind(Wd)
    ex = g.export()
    # the event the QKV tiles of layer 0 wait on
    first_qkv = int(np.flatnonzero(
        ex["task_kind"] == mpk.TASK_KINDS.index("qkv"))[0])
    e = int(ex["task_dep"][first_qkv])
    g.add_event_count(e, +1)
    g.set_wait_timeout_ms(300)
    kvd = dev_kv(kv)
    t = torch.from_numpy(tok).cuda()
    logits, nxt = _outputs(wl.batch, wl.shape.vocab)
    g.decode_step(t, kvd, logits, nxt)
    assert g.status() == mpk.MPK_ERR_TIMEOUT
    # a step enqueued while the abort flag is up does nothing
    g.decode_step(t, kvd, logits, nxt)
    assert g.status() == mpk.MPK_ERR_TIMEOUT
    g.add_event_count(e, -1)
    g.reset()
    kvd = dev_kv(kv)
    g.decode_step(t, kvd, logits, nxt)
    assert g.status() == mpk.MPK_OK
    ref, _ = run_oracle(wl, W, kv, tok)
    check_steps([(logits.cpu().numpy(), nxt.cpu().numpy())], ref)
    g.close()


def test_unmapped_kv_page_is_reported(tiny):
    wl, W, Wd, kv, tok = tiny
    bad = dataclasses.replace(kv, page_table=kv.page_table.copy())
    bad.page_table[0, int(kv.seq_lens[0]) // wl.page_size] = -1
    g = _graph(wl)
    g.bind(Wd)
    logits, nxt = _outputs(wl.batch, wl.shape.vocab)
    g.decode_step(torch.from_numpy(tok).cuda(), dev_kv(bad), logits, nxt)
    assert g.status() == mpk.MPK_ERR_KV_PAGE
    g.reset()
    g.close()


# ----------------------------------------------------- configured sizes
@pytest.mark.parametrize("name", ["chain_b1", "chain_b8"])
def test_chain_full_size(name):
    wl = synth.WORKLOADS[name]
    W, _, tok = _inputs(wl)
    gpu, _ = run_gpu(wl, dev_weights(W, wl.shape), None, tok)
    ref, _ = run_oracle(wl, W, None, tok)
    check_steps(gpu, ref)


# ---------------------------------------------------- several steps a launch
def _steps_both_ways(wl, W_host, kv_host, tok, n, **kw):
    """n greedy steps as n launches and as one launch (mpk_decode_steps),
    from the same inputs; returns both (tokens [n][B], last logits, K, V,
    seq_lens)."""
    shape = wl.shape
    Wd = dev_weights(W_host, shape)
    out = []
    for one_launch in (False, True):
        g = _graph(wl, **kw)
        g.bind(Wd)
        kv = dev_kv(kv_host) if kv_host is not None else None
        t = torch.from_numpy(np.asarray(tok, np.int32)).cuda()
        logits = torch.empty(wl.batch, shape.vocab, device="cuda")
        nxt = torch.empty(n, wl.batch, dtype=torch.int32, device="cuda")
        if one_launch:
            g.decode_steps(t, kv, logits, nxt, n)
        else:
            for i in range(n):
                g.decode_step(t if i == 0 else nxt[i - 1], kv, logits, nxt[i])
        torch.cuda.synchronize()
        assert g.status() == mpk.MPK_OK, mpk.STATUS_NAMES[g.status()]
        out.append((nxt.cpu().numpy(), logits.cpu().numpy(),
                    None if kv is None else (kv.k_pool.clone(), kv.v_pool.clone(),
                                             kv.seq_lens.cpu().numpy())))
        g.close()
    return out


@pytest.mark.parametrize("case", ["tiny", "tiny_b3_jit", "chain_b4"])
def test_several_steps_in_one_launch_equal_step_by_step(case):
    """Figure 1 of the MPK summary: the decode loop inside one launch.  Step
    i + 1 embeds step i's tokens and waits for its end; the result must be
    bit-identical to one launch per step."""
    base = synth.WORKLOADS["tiny"]
    if case == "tiny":
        wl = base
    elif case == "tiny_b3_jit":
        wl = dataclasses.replace(base, name="tiny_b3", batch=3,
                                 ctx=(5, 37, 120), steps=4)
    else:
        shape = synth.ModelShape(0, 256, 1, 1, 32, 0, 1024, chain_ffn=512)
        wl = synth.Workload("chain_small", shape, 4, (), 64, 1)
    W, kv, tok = _inputs(wl, seed=9)
    (t1, l1, kv1), (tn, ln, kvn) = _steps_both_ways(wl, W, kv, tok, 4)
    assert np.array_equal(t1, tn)
    assert np.array_equal(l1, ln)
    if kv1 is not None:
        assert torch.equal(kv1[0], kvn[0]) and torch.equal(kv1[1], kvn[1])
        assert np.array_equal(kv1[2], kvn[2])
