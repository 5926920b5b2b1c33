"""Planted mistakes in the oracle, each of which some pin must catch.

Each case swaps one oracle function (on the CPU, for the duration of the
test only) for a plausibly wrong variant -- a shifted position, a dropped
term, a swapped operand, a wrong index, a missing fusion rule -- and runs
the pin that guards it; the pin must fail.  This checks the pins
themselves: an oracle that agrees with its pins only because the pins are
weak would pass them with these mistakes too."""
import collections

import numpy as np
import pytest

from oracle import numerics as nx
from oracle import tgraph
from task_graph_runtime_gb300 import synth

import test_oracle_graph as graph_pins
import test_oracle_numerics as pins

_rope = nx.rope
_gather = nx.gather_kv
_swiglu = nx.swiglu
_split = nx._split_qkv
_attn = nx.attention_decode
_rms = nx.rmsnorm
_linear = nx.linear
_merge = nx.merge_partials


def _rope_shifted(x, pos, theta):
    return _rope(x, np.asarray(pos) + 1, theta)


def _rope_wrong_sign(x, pos, theta):
    return _rope(x, -np.asarray(pos), theta)


def _gather_drop_last(pool, row, layer, g, n):
    return _gather(pool, row, layer, g, max(n - 1, 1))


def _swiglu_swapped(g, u):
    return _swiglu(u, g)


def _residual_dropped(a, b):
    return np.asarray(b).copy()


def _split_wrong_kv_head(qkv, shape):
    q, k, v = _split(qkv, shape)
    return q, k[:, ::-1], v[:, ::-1]


def _attn_unscaled(q, k, v):
    d = nx.bf16_to_f32(q).shape[-1]
    return _attn(nx.f32_to_bf16(nx.bf16_to_f32(q) * np.float32(np.sqrt(d))),
                 k, v)


def _rms_no_gain(x, w, eps):
    return _rms(x, np.full_like(w, 0x3F80), eps)   # bf16 1.0 gains


def _linear_transposed(x, w):
    return _linear(x, np.ascontiguousarray(np.asarray(w).T))


def _argmax_highest(logits):
    l = np.asarray(logits)
    return (l.shape[-1] - 1 - np.argmax(l[..., ::-1], axis=-1)).astype(
        np.int32)


def _merge_unshifted(parts):
    return _merge([(np.zeros_like(p[0]), p[1], p[2]) for p in parts])


def _overlap_closed(a, b):
    return (a[0] == b[0] and a[1] <= b[2] and b[1] <= a[2]
            and a[3] <= b[4] and b[3] <= a[4])


def _fuse_def41_once(raw):
    """Def 4.1 only, one pass (no Def 4.2, no fixpoint)."""
    ev = {i: ({p}, {c}) for i, (p, c) in enumerate(raw)}
    groups = collections.defaultdict(list)
    for i in sorted(ev):
        groups[frozenset(ev[i][1])].append(i)
    for ids in groups.values():
        merged = set()
        for i in ids:
            merged |= ev[i][0]
        ev[ids[0]] = (merged, ev[ids[0]][1])
        for i in ids[1:]:
            del ev[i]
    return ev


CASES = [
    ("rope at position + 1", nx, "rope", _rope_shifted,
     pins.test_rope_equals_complex_rotation),
    ("rope rotating the wrong way", nx, "rope", _rope_wrong_sign,
     pins.test_rope_equals_complex_rotation),
    ("attention misses the newest token", nx, "gather_kv", _gather_drop_last,
     lambda: pins.test_decode_step_equals_last_row_of_full_forward(
         synth.TINY)),
    ("gate and up swapped", nx, "swiglu", _swiglu_swapped,
     lambda: pins.test_full_forward_matches_torch_float64_model(synth.TINY)),
    ("residual dropped", nx, "residual_add", _residual_dropped,
     lambda: pins.test_full_forward_matches_torch_float64_model(synth.TINY)),
    ("query heads read the wrong KV head", nx, "_split_qkv",
     _split_wrong_kv_head,
     lambda: pins.test_full_forward_matches_torch_float64_model(pins.SMALL)),
    ("scores not scaled by 1/sqrt(d)", nx, "attention_decode",
     _attn_unscaled, pins.test_attention_matches_torch_sdpa_gqa),
    ("RMSNorm gain ignored", nx, "rmsnorm", _rms_no_gain,
     pins.test_rmsnorm_matches_torch_rms_norm),
    ("weight matrix transposed", nx, "linear", _linear_transposed,
     pins.test_linear_basis_vector_selects_column),
    ("argmax takes the highest index on ties", nx, "argmax_lowest",
     _argmax_highest, pins.test_argmax_lowest_index_on_ties),
    ("chunk merge without the max shift", nx, "merge_partials",
     _merge_unshifted, pins.test_split_kv_merge_equals_naive_softmax),
    ("touching regions counted as overlapping", tgraph, "_overlap",
     _overlap_closed, graph_pins.test_overlap_is_strict_on_both_axes),
    ("fusion: Def 4.1 once, no Def 4.2", tgraph, "fuse", _fuse_def41_once,
     graph_pins.test_golden_fusion_and_fanout),
]


@pytest.mark.parametrize("name,module,attr,mutant,pin", CASES,
                         ids=[c[0] for c in CASES])
def test_planted_mistake_is_caught(monkeypatch, name, module, attr, mutant,
                                   pin):
    monkeypatch.setattr(module, attr, mutant)
    with pytest.raises((AssertionError, ValueError, IndexError)):
        pin()
