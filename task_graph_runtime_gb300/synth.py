"""Seeded synthetic inputs shared, as data, by the CUDA path and the oracle.

This module holds workload shapes and random-number recipes only: it does no
part of the decode step's arithmetic.  Both sides receive the same bf16 bit
patterns (numpy ``uint16`` on the host, or ``torch.bfloat16`` on the device).

Recipe (every tensor is seeded independently):
  * per-tensor seed = crc32(name) XOR base_seed;
  * linear weights  = bf16_rne(0.02 * N(0, 1));
  * norm gains      = bf16_rne(1 + 0.02 * N(0, 1))  (a zero-mean gain would
    collapse the activations of a randomly initialised model);
  * KV pool         = bf16_rne(N(0, 1)) everywhere (slots past a sequence's
    length are stale data that is never read);
  * page table      = a seeded permutation of the pool's page ids, each
    sequence owning ceil((ctx + steps) / page_size) pages, -1 past that;
  * tokens          = uniform integers in [0, vocab).

On the host the normals come from numpy's PCG64 (``standard_normal``,
float32); on a CUDA device from torch's Philox generator, which is much
faster for the 8B-parameter shapes.  The two sources give different values
for the same seed; a test uses one source for both sides.  The fp32 -> bf16
step is torch's round-to-nearest-even conversion.
"""
from __future__ import annotations

import dataclasses
import zlib
from typing import Dict, List, Optional

import numpy as np

WEIGHT_STD = 0.02
NORM_STD = 0.02


@dataclasses.dataclass(frozen=True)
class ModelShape:
    """Decoder shape.  ``chain_ffn > 0`` (with n_layers == 0) selects the
    chained-linear microbenchmark: RMSNorm -> W1 [ffn, hidden] -> SiLU ->
    W2 [hidden, ffn] -> vocab projection."""
    n_layers: int
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    rms_eps: float = 1e-6
    rope_theta: float = 1e4
    qk_norm: bool = False
    chain_ffn: int = 0

    @property
    def qkv_rows(self) -> int:
        return (self.n_q_heads + 2 * self.n_kv_heads) * self.head_dim

    @property
    def is_chain(self) -> bool:
        return self.chain_ffn > 0


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    shape: ModelShape
    batch: int
    ctx: tuple            # prior context length per sequence
    page_size: int
    steps: int            # greedy decode steps the workload runs

    @property
    def pages_per_seq(self) -> List[int]:
        return [-(-(c + self.steps) // self.page_size) for c in self.ctx]

    @property
    def max_pages_per_seq(self) -> int:
        return max(self.pages_per_seq) if self.ctx else 0

    @property
    def num_pages(self) -> int:
        return sum(self.pages_per_seq)


TINY = ModelShape(2, 256, 4, 2, 64, 688, 1024, 1e-6, 1e4, False)
LLAMA_1B = ModelShape(16, 2048, 32, 8, 64, 8192, 32000, 1e-6, 1e4, False)
QWEN3_8B = ModelShape(36, 4096, 32, 8, 128, 12288, 151936, 1e-6, 1e6, True)
CHAIN = ModelShape(0, 4096, 1, 1, 128, 12288, 151936, 1e-6, 1e4, False,
                   chain_ffn=12288)


def _varlen_ctx(batch: int, lo: int, hi: int, seed: int) -> tuple:
    rng = np.random.Generator(np.random.PCG64(seed))
    return tuple(int(v) for v in rng.integers(lo, hi + 1, size=batch))


WORKLOADS: Dict[str, Workload] = {
    # one decode step of a 2-layer toy decoder over 128 cached tokens
    "tiny": Workload("tiny", TINY, 1, (128,), 16, 1),
    # ~1B Llama-style decoder, 1024-token context, 32 greedy steps
    "llama1b": Workload("llama1b", LLAMA_1B, 1, (1024,), 64, 32),
    # Qwen3-8B-shaped decoder, 2048-token context, 32 greedy steps
    "qwen3_8b": Workload("qwen3_8b", QWEN3_8B, 1, (2048,), 64, 32),
    # same shape, 16 sequences with contexts drawn from U{128..4096}
    "qwen3_8b_b16": Workload("qwen3_8b_b16", QWEN3_8B, 16,
                             _varlen_ctx(16, 128, 4096, 0xC4), 64, 32),
    # chained linear layers, batch 1 and batch 8 (no KV cache)
    "chain_b1": Workload("chain_b1", CHAIN, 1, (), 64, 1),
    "chain_b8": Workload("chain_b8", CHAIN, 8, (), 64, 1),
}


def tensor_seed(name: str, base_seed: int = 0) -> int:
    return (zlib.crc32(name.encode()) ^ base_seed) & 0xFFFFFFFF


# ---------------------------------------------------------------- host side
def _to_bf16_bits(f32: np.ndarray) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.ascontiguousarray(f32, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def normal_bf16(shape, seed: int, std: float = 1.0, mean: float = 0.0,
                chunk: int = 1 << 24) -> np.ndarray:
    """bf16 bits of mean + std * N(0,1), drawn with numpy PCG64(seed)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        v = rng.standard_normal(e - s, dtype=np.float32)
        if std != 1.0:
            v *= np.float32(std)
        if mean != 0.0:
            v += np.float32(mean)
        out[s:e] = _to_bf16_bits(v)
    return out.reshape(shape)


def weight_shapes(shape: ModelShape) -> Dict[str, tuple]:
    """Name -> shape of every weight tensor (row-major, [out, in] for linear)."""
    h, d, F, V = shape.hidden, shape.head_dim, shape.ffn, shape.vocab
    out: Dict[str, tuple] = {"embed": (V, h), "final_norm": (h,),
                             "lm_head": (V, h)}
    if shape.is_chain:
        out["chain_w1"] = (shape.chain_ffn, h)
        out["chain_w2"] = (h, shape.chain_ffn)
        return out
    for l in range(shape.n_layers):
        out[f"layer{l}.ln1"] = (h,)
        out[f"layer{l}.wqkv"] = (shape.qkv_rows, h)
        if shape.qk_norm:
            out[f"layer{l}.q_norm"] = (d,)
            out[f"layer{l}.k_norm"] = (d,)
        out[f"layer{l}.wo"] = (h, shape.n_q_heads * d)
        out[f"layer{l}.ln2"] = (h,)
        out[f"layer{l}.wgu"] = (2 * F, h)      # rows [0,F) gate, [F,2F) up
        out[f"layer{l}.wd"] = (h, F)
    return out


def _is_norm(name: str) -> bool:
    return name.endswith(("ln1", "ln2", "q_norm", "k_norm", "final_norm"))


def model_weights(shape: ModelShape, base_seed: int = 0) -> Dict[str, np.ndarray]:
    """All weights as host bf16 bit arrays (uint16)."""
    out = {}
    for name, shp in weight_shapes(shape).items():
        seed = tensor_seed(name, base_seed)
        if _is_norm(name):
            out[name] = normal_bf16(shp, seed, NORM_STD, 1.0)
        else:
            out[name] = normal_bf16(shp, seed, WEIGHT_STD)
    return out


@dataclasses.dataclass
class KVInputs:
    k_pool: np.ndarray       # uint16 [L][num_pages][Hkv][page_size][d]
    v_pool: np.ndarray
    page_table: np.ndarray   # int32 [B][max_pages_per_seq], -1 = unmapped
    seq_lens: np.ndarray     # int32 [B], tokens already cached


def kv_pool_shape(wl: Workload) -> tuple:
    s = wl.shape
    return (s.n_layers, wl.num_pages, s.n_kv_heads, wl.page_size, s.head_dim)


def page_table(wl: Workload, base_seed: int = 0) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(tensor_seed("page_table",
                                                          base_seed)))
    perm = rng.permutation(wl.num_pages).astype(np.int32)
    pt = np.full((wl.batch, max(1, wl.max_pages_per_seq)), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(wl.pages_per_seq):
        pt[b, :n] = perm[off:off + n]
        off += n
    return pt


def kv_inputs(wl: Workload, base_seed: int = 0) -> KVInputs:
    shp = kv_pool_shape(wl)
    k = normal_bf16(shp, tensor_seed("k_pool", base_seed))
    v = normal_bf16(shp, tensor_seed("v_pool", base_seed))
    return KVInputs(k, v, page_table(wl, base_seed),
                    np.array(wl.ctx if wl.ctx else [0] * wl.batch,
                             dtype=np.int32))


def tokens(wl: Workload, base_seed: int = 0, step: int = 0) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(
        tensor_seed(f"tokens{step}", base_seed)))
    return rng.integers(0, wl.shape.vocab, size=wl.batch).astype(np.int32)


# -------------------------------------------------------------- device side
def device_normal_bf16(shape, seed: int, std: float = 1.0, mean: float = 0.0,
                       device="cuda"):
    """torch.bfloat16 tensor of mean + std * N(0,1) from torch's generator on
    ``device`` (fast path for the multi-GB shapes)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    t = torch.empty(shape, dtype=torch.float32, device=device)
    t.normal_(mean, std, generator=g)
    return t.to(torch.bfloat16)


def device_model_weights(shape: ModelShape, base_seed: int = 0,
                         device="cuda") -> Dict[str, "object"]:
    out = {}
    for name, shp in weight_shapes(shape).items():
        seed = tensor_seed(name, base_seed)
        if _is_norm(name):
            out[name] = device_normal_bf16(shp, seed, NORM_STD, 1.0, device)
        else:
            out[name] = device_normal_bf16(shp, seed, WEIGHT_STD, 0.0, device)
    return out


def device_kv_inputs(wl: Workload, base_seed: int = 0, device="cuda"):
    """(k_pool, v_pool) as device bf16 tensors plus host page table and
    seq_lens (numpy)."""
    shp = kv_pool_shape(wl)
    k = device_normal_bf16(shp, tensor_seed("k_pool", base_seed), 1.0, 0.0,
                           device)
    v = device_normal_bf16(shp, tensor_seed("v_pool", base_seed), 1.0, 0.0,
                           device)
    return (k, v, page_table(wl, base_seed),
            np.array(wl.ctx if wl.ctx else [0] * wl.batch, dtype=np.int32))


def as_uint16(t) -> np.ndarray:
    """Host copy of a torch bf16 tensor as uint16 bits."""
    import torch
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(
        np.uint16)
