"""The allocation-free decode step (mpk_decode_step_noalloc).

It exists for callers that may not allocate device memory while they run
(memory reserved up front by their own allocator, loops that cannot take the
synchronisation cudaMalloc implies, plugin hosts that own every
allocation).  Its scratch lives in one static device array, so these tests
check that two calls in a row give the same outputs as mpk_decode_step on
the same inputs (within the decode-step bound), that the calls leave the
device's free memory unchanged, and that a graph too large for the array is
refused.  This file is collected last on purpose."""
import numpy as np
import pytest
import torch

from task_graph_runtime_gb300 import mpk, synth

from gpu_util import dev_kv, dev_weights, within_bound

pytestmark = pytest.mark.gpu


def _two_steps_existing(wl, Wd, kv, tok):
    g = mpk.Graph(wl.shape, wl.batch, page_size=wl.page_size,
                  max_pages_per_seq=max(1, wl.max_pages_per_seq))
    g.bind(Wd)
    kvd = dev_kv(kv) if kv is not None else None
    t = torch.from_numpy(tok).cuda()
    out = []
    for _ in range(2):
        lg = torch.empty(wl.batch, wl.shape.vocab, device="cuda")
        nt = torch.empty(wl.batch, dtype=torch.int32, device="cuda")
        g.decode_step(t, kvd, lg, nt)
        torch.cuda.synchronize()
        assert g.status() == mpk.MPK_OK
        out.append((lg.cpu().numpy(), nt.cpu().numpy()))
        t = nt
    g.close()
    return out


@pytest.mark.parametrize("name", ["tiny", "chain_small"])
def test_noalloc_matches_decode_step_two_calls(name):
    if name == "tiny":
        wl = synth.WORKLOADS["tiny"]
    else:
        shape = synth.ModelShape(0, 512, 1, 1, 32, 0, 3000, chain_ffn=1536)
        wl = synth.Workload("chain_small", shape, 2, (), 64, 1)
    W = synth.model_weights(wl.shape, 11)
    kv = synth.kv_inputs(wl, 11) if not wl.shape.is_chain else None
    tok = synth.tokens(wl, 11)
    Wd = dev_weights(W, wl.shape)
    ref = _two_steps_existing(wl, Wd, kv, tok)

    g = mpk.Graph(wl.shape, wl.batch, page_size=wl.page_size,
                  max_pages_per_seq=max(1, wl.max_pages_per_seq))
    kvd = dev_kv(kv) if kv is not None else None
    t = torch.from_numpy(tok).cuda()
    status = torch.full((1,), 99, dtype=torch.int32, device="cuda")
    lgs = [torch.empty(wl.batch, wl.shape.vocab, device="cuda")
           for _ in range(2)]
    nts = [torch.empty(wl.batch, dtype=torch.int32, device="cuda")
           for _ in range(2)]
    free = []
    for step in range(2):
        torch.cuda.synchronize()
        free.append(torch.cuda.mem_get_info()[0])
        mpk.mpk_decode_step_noalloc(g, Wd, t, kvd, lgs[step], nts[step],
                                    status)
        torch.cuda.synchronize()
        free.append(torch.cuda.mem_get_info()[0])
        assert int(status.item()) == mpk.MPK_OK
        rl, rt = ref[step]
        ok, err, lim = within_bound(lgs[step].cpu().numpy(), rl)
        assert ok, f"step {step}: {err} > {lim}"
        assert np.array_equal(nts[step].cpu().numpy(), rt)
        t = nts[step]
    # the second call (after the first call's one-time set-up) leaves the
    # device's free memory unchanged
    assert free[3] == free[2]
    if kvd is not None:
        assert np.array_equal(kvd.seq_lens.cpu().numpy(), kv.seq_lens + 2)
    g.close()


def test_noalloc_refuses_graph_larger_than_its_array():
    wl = synth.WORKLOADS["qwen3_8b"]
    g = mpk.Graph(wl.shape, 1, num_workers=148, page_size=wl.page_size,
                  max_pages_per_seq=wl.max_pages_per_seq)
    dummy = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    tensors = {n: dummy for n in synth.weight_shapes(wl.shape)}
    w = mpk.Weights(tensors, wl.shape)
    small = torch.zeros(4, dtype=torch.int32, device="cuda")
    kv = mpk.KVCache(dummy.view(1, 1, 1, 1, 16), dummy.view(1, 1, 1, 1, 16),
                     small, small)
    with pytest.raises(mpk.MpkError) as e:
        mpk.mpk_decode_step_noalloc(g, w, small, kv,
                                    torch.zeros(1, device="cuda"), small)
    assert e.value.status == mpk.MPK_ERR_UNSUPPORTED
    g.close()
