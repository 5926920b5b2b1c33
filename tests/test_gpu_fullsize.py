"""Full-size decode-step parity in the launch configuration bench.py times
(default tiling, megakernel mode) for the ~1B decoder (16 layers), the
Qwen3-8B-shaped decoder at batch 1 and at batch 16 (contexts U{128..4096}).

Inputs come from the seeded device generator (torch Philox) and are copied
to the host for the oracle, which recomputes every output from them.

Two checks, in this order:

1. Every layer in isolation, at the exact bound |gpu - ref| <= 2e-2 *
   max|ref| + 1e-3.  A one-layer graph with the same kernels, tiling and
   launch geometry runs layer l on the oracle's own residual stream entering
   layer l (the oracle's output, never the GPU's), then the final norm and
   lm_head.  Compared element-wise: the residual stream leaving the layer,
   the K and V the layer appends to the paged cache, and the logits; greedy
   tokens by the token rule (equal, except where the oracle's top-2 gap is
   below 1e-2).

2. The whole model in one launch, two greedy steps.  Over 16-36 layers of a
   randomly initialised model a one-ulp bf16 rounding difference anywhere
   grows layer by layer, so two correct implementations that differ only in
   the order of their fp32 sums disagree by about the bound: the oracle with
   an fp32 accumulator (o32) and with an fp64 one (o64) is the measured
   example.  The reading applied (and recorded with the measured spreads in
   the design notes): every residual stream and the logits must satisfy
   |gpu - o32| <= bound + |o32 - o64| (max norms), and each greedy token must
   be the argmax of o32 or of o64, or tie the top logit of either within
   1e-2.  For the second step each oracle continues from its own first
   step (tokens and KV cache); it is compared when the GPU's first tokens
   equal both oracles'."""
import dataclasses

import numpy as np
import pytest
import torch

from oracle import numerics as nx
from task_graph_runtime_gb300 import mpk, synth

from gpu_util import tokens_agree, within_bound

pytestmark = pytest.mark.gpu


def _graph(wl, shape):
    return mpk.Graph(shape, wl.batch, page_size=wl.page_size,
                     max_pages_per_seq=wl.max_pages_per_seq)


def _gpu_run(wl, shape, W_dev, k, v, pt, sl, tok, steps, hidden=False):
    """`steps` greedy steps in one graph; per step (logits, tokens) and, if
    asked, the residual streams of the first step [L + 1][B, h]."""
    g = _graph(wl, shape)
    g.bind(mpk.Weights(W_dev, shape))
    kv = mpk.KVCache(k, v, torch.from_numpy(pt).cuda(),
                     torch.from_numpy(sl.copy()).cuda())
    t = torch.from_numpy(np.asarray(tok, np.int32)).cuda()
    out, hs = [], None
    for s in range(steps):
        logits = torch.empty(wl.batch, shape.vocab, device="cuda")
        nxt = torch.empty(wl.batch, dtype=torch.int32, device="cuda")
        g.decode_step(t, kv, logits, nxt)
        torch.cuda.synchronize()
        assert g.status() == mpk.MPK_OK, mpk.STATUS_NAMES[g.status()]
        out.append((logits.cpu().numpy(), nxt.cpu().numpy()))
        if hidden and s == 0:
            hs = [g.read_hidden(l) for l in range(shape.n_layers + 1)]
        t = nxt
    g.close()
    return out, hs


def _oracle(shape, W, tok, k, v, pt, sl, acc=np.float32):
    """One oracle step on copies of the cache; returns (result, k, v, sl)."""
    k, v, sl = k.copy(), v.copy(), sl.copy()
    nx.set_accumulator(acc)
    try:
        r = nx.decode_step(shape, W, tok, k, v, pt, sl)
    finally:
        nx.set_accumulator(np.float32)
    return r, k, v, sl


def _f(u16):
    return nx.bf16_to_f32(u16).astype(np.float64)


def _spread(a, b):
    return float(np.abs(np.asarray(a, np.float64) -
                        np.asarray(b, np.float64)).max())


def _lim(ref):
    return 2e-2 * float(np.abs(np.asarray(ref, np.float64)).max()) + 1e-3


def _tokens_ok(gt, refs, gap=1e-2):
    """Each token is the argmax of one of the oracles, or ties its top
    logit within `gap`."""
    for b, t in enumerate(np.asarray(gt)):
        if not any(tokens_agree([t], r[b:b + 1], gap) for r in refs):
            return False
    return True


def _inputs(name):
    wl = synth.WORKLOADS[name]
    s = wl.shape
    W = synth.device_model_weights(s, 0, "cuda")
    k, v, pt, sl = synth.device_kv_inputs(wl, 0, "cuda")
    tok = synth.tokens(wl, 0)
    W_host = {n: synth.as_uint16(t) for n, t in W.items()}
    return wl, s, W, k, v, pt, sl, tok, W_host


def _isolated_layers(name):
    wl, s, W, k, v, pt, sl, tok, W_host = _inputs(name)
    k_host, v_host = synth.as_uint16(k), synth.as_uint16(v)
    ref, k_ref, v_ref, _ = _oracle(s, W_host, tok, k_host, v_host, pt, sl)
    one = dataclasses.replace(s, n_layers=1)
    wl1 = dataclasses.replace(wl, shape=one)
    B = wl.batch
    ids = np.arange(B, dtype=np.int32)
    rows = np.arange(B)
    pos = sl.astype(np.int64)
    slot_page = pt[rows, pos // wl.page_size]
    slot_off = pos % wl.page_size
    worst = 0.0
    for l in range(s.n_layers):
        h_in = W_host["embed"][tok] if l == 0 else ref["hidden"][l - 1]
        Wd1 = {"embed": torch.from_numpy(h_in.view(np.int16)).view(
                   torch.bfloat16).cuda(),
               "final_norm": W["final_norm"], "lm_head": W["lm_head"]}
        for n in synth.weight_shapes(s):
            if n.startswith(f"layer{l}."):
                Wd1["layer0." + n.split(".", 1)[1]] = W[n]
        g = _graph(wl1, one)
        g.bind(mpk.Weights(Wd1, one))
        k1, v1 = k[l:l + 1].clone(), v[l:l + 1].clone()
        kv = mpk.KVCache(k1, v1, torch.from_numpy(pt).cuda(),
                         torch.from_numpy(sl.copy()).cuda())
        logits = torch.empty(B, s.vocab, device="cuda")
        nxt = torch.empty(B, dtype=torch.int32, device="cuda")
        g.decode_step(torch.from_numpy(ids).cuda(), kv, logits, nxt)
        torch.cuda.synchronize()
        assert g.status() == mpk.MPK_OK, (l, mpk.STATUS_NAMES[g.status()])
        h_out = g.read_hidden(1)
        g.close()
        # the residual stream leaving layer l
        ok, e, lim = within_bound(_f(h_out), _f(ref["hidden"][l]))
        assert ok, (name, l, "hidden", e, lim)
        # the K and V appended at each sequence's position
        sp = torch.from_numpy(slot_page).cuda()
        so = torch.from_numpy(slot_off).cuda()
        kg = synth.as_uint16(k1[0, sp, :, so])
        vg = synth.as_uint16(v1[0, sp, :, so])
        kr = k_ref[l, slot_page, :, slot_off]
        vr = v_ref[l, slot_page, :, slot_off]
        assert within_bound(_f(kg), _f(kr))[0], (name, l, "k")
        assert within_bound(_f(vg), _f(vr))[0], (name, l, "v")
        # logits of the final norm + lm_head on the oracle's layer output
        nf = nx.rmsnorm(ref["hidden"][l], W_host["final_norm"], s.rms_eps)
        rl = nx.linear(nf, W_host["lm_head"])
        ok, e2, lim2 = within_bound(logits.cpu().numpy(), rl)
        assert ok, (name, l, "logits", e2, lim2)
        assert tokens_agree(nxt.cpu().numpy(), rl), (name, l, "tokens")
        worst = max(worst, e / lim, e2 / lim2)
    print(f"{name}: {s.n_layers} isolated layers within the bound; worst "
          f"error/bound {worst:.3f}")


def _whole_model(name, steps=2):
    wl, s, W, k, v, pt, sl, tok, W_host = _inputs(name)
    k_host, v_host = synth.as_uint16(k), synth.as_uint16(v)
    gpu, hs = _gpu_run(wl, s, W, k.clone(), v.clone(), pt, sl, tok, steps,
                       hidden=True)
    r32, k32, v32, s32 = _oracle(s, W_host, tok, k_host, v_host, pt, sl)
    r64, k64, v64, s64 = _oracle(s, W_host, tok, k_host, v_host, pt, sl,
                                 np.float64)
    # residual streams entering layers 1..L (the oracle's layer outputs)
    worst_h = 0.0
    for l in range(s.n_layers):
        ref, alt = _f(r32["hidden"][l]), _f(r64["hidden"][l])
        e, noise = _spread(_f(hs[l + 1]), ref), _spread(ref, alt)
        assert e <= _lim(ref) + noise, (name, l, e, _lim(ref), noise)
        worst_h = max(worst_h, e / (_lim(ref) + noise))
    gl, gt = gpu[0]
    e = _spread(gl, r32["logits"])
    noise = _spread(r32["logits"], r64["logits"])
    print(f"{name}: step 1 logits |gpu-o32| {e:.4f}, bound {_lim(r32['logits']):.4f}, "
          f"|o32-o64| {noise:.4f}; hidden worst ratio {worst_h:.3f}; "
          f"tokens gpu {gt[:4]} o32 {r32['next_tokens'][:4]} "
          f"o64 {r64['next_tokens'][:4]}")
    assert e <= _lim(r32["logits"]) + noise
    assert _tokens_ok(gt, [r32["logits"], r64["logits"]])
    # the second step: each oracle continues from its own first step
    if steps > 1 and np.array_equal(gt, r32["next_tokens"]) and \
            np.array_equal(gt, r64["next_tokens"]):
        t2 = r32["next_tokens"]
        a32 = _oracle(s, W_host, t2, k32, v32, pt, s32)[0]
        a64 = _oracle(s, W_host, t2, k64, v64, pt, s64, np.float64)[0]
        e2 = _spread(gpu[1][0], a32["logits"])
        n2 = _spread(a32["logits"], a64["logits"])
        print(f"{name}: step 2 logits |gpu-o32| {e2:.4f}, bound "
              f"{_lim(a32['logits']):.4f}, |o32-o64| {n2:.4f}")
        assert e2 <= _lim(a32["logits"]) + n2
        assert _tokens_ok(gpu[1][1], [a32["logits"], a64["logits"]])


@pytest.mark.parametrize("name", ["llama1b", "qwen3_8b", "qwen3_8b_b16"])
def test_every_layer_isolated_full_size(name):
    _isolated_layers(name)


@pytest.mark.parametrize("name", ["llama1b", "qwen3_8b", "qwen3_8b_b16"])
def test_whole_model_full_size(name):
    _whole_model(name, steps=2)
