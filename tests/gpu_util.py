"""Helpers shared by the GPU tests: device copies of the seeded inputs, one
call through the C-ABI binding, and the parity bound of the decode step."""
import numpy as np
import torch

from task_graph_runtime_gb300 import mpk, synth


def to_dev(u16: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).view(
        torch.bfloat16).cuda()


def dev_weights(W_host, shape):
    return mpk.Weights({k: to_dev(v) for k, v in W_host.items()}, shape)


def dev_kv(kv: synth.KVInputs):
    return mpk.KVCache(to_dev(kv.k_pool), to_dev(kv.v_pool),
                       torch.from_numpy(kv.page_table).cuda(),
                       torch.from_numpy(kv.seq_lens.copy()).cuda())


def within_bound(got, ref, rel=2e-2, absol=1e-3):
    """|gpu - ref| <= rel * max|ref| + abs (the decode-step bound)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    lim = rel * np.abs(ref).max() + absol
    err = np.abs(got - ref).max()
    return err <= lim, err, lim


def tokens_agree(got_tokens, ref_logits, gap=1e-2):
    """Greedy tokens equal, except rows whose oracle top-2 gap is below
    ``gap`` (there any of the near-tied tokens is accepted)."""
    for b, t in enumerate(np.asarray(got_tokens)):
        row = np.asarray(ref_logits[b], np.float64)
        top = np.sort(row)[-2:]
        best = int(np.argmax(row))
        if t == best:
            continue
        if top[1] - top[0] < gap and row[t] >= top[1] - gap:
            continue
        return False
    return True


def bf16_to_f32(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy()
