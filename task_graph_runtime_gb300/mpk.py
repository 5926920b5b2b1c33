"""ctypes binding of ``libmpk.so`` (include/mpk.h).  Argument marshalling
only: every step of the decode path runs in the library's kernels.  Loading
fails loudly when the library is missing; there is no fallback.

Functions keep the C names (``mpk_build_tgraph``, ``mpk_decode_step``, ...).
``Graph`` wraps a graph handle for convenience; ``Weights`` and ``KVCache``
hold the device tensors a step borrows (torch tensors are used for device
memory and streams only)."""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional, Sequence

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmpk.so")

MPK_OK = 0
STATUS_NAMES = {
    0: "MPK_OK", 1: "MPK_ERR_INVALID_ARG", 2: "MPK_ERR_UNSUPPORTED",
    3: "MPK_ERR_CUDA", 4: "MPK_ERR_OOM", 5: "MPK_ERR_NOT_CORESIDENT",
    6: "MPK_ERR_TIMEOUT", 7: "MPK_ERR_KV_PAGE", 8: "MPK_ERR_QUEUE_OVERFLOW",
    9: "MPK_ERR_GRAPH_INVALID", 10: "MPK_ERR_NOT_BOUND"}
globals().update({v: k for k, v in STATUS_NAMES.items()})

TASK_KINDS = ["empty", "qkv", "attn", "o", "gateup", "down", "lm_head",
              "argmax", "chain_up", "chain_down"]
MODE_MEGAKERNEL, MODE_KPO, MODE_KPO_GRAPH = 0, 1, 2
LAYER_TENSORS = ["ln1", "wqkv", "q_norm", "k_norm", "wo", "ln2", "wgu", "wd"]


class MpkError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")


class ModelShape(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("hidden", ctypes.c_int),
                ("n_q_heads", ctypes.c_int), ("n_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("ffn", ctypes.c_int),
                ("vocab", ctypes.c_int), ("rms_eps", ctypes.c_float),
                ("rope_theta", ctypes.c_float), ("qk_norm", ctypes.c_int),
                ("chain_ffn", ctypes.c_int), ("page_size", ctypes.c_int),
                ("max_pages_per_seq", ctypes.c_int)]


class TileSizes(ctypes.Structure):
    _fields_ = [("num_workers", ctypes.c_int),
                ("gemv_rows_per_task", ctypes.c_int),
                ("mma_rows_per_task", ctypes.c_int),
                ("attn_chunks", ctypes.c_int),
                ("num_sched_sms", ctypes.c_int),
                ("sched_warps_per_sm", ctypes.c_int),
                ("smem_pages", ctypes.c_int),
                ("coarse_events", ctypes.c_int)]


class _Weights(ctypes.Structure):
    _fields_ = [("embed", ctypes.c_void_p), ("final_norm", ctypes.c_void_p),
                ("lm_head", ctypes.c_void_p),
                ("layers", ctypes.POINTER(ctypes.c_void_p)),
                ("chain_w1", ctypes.c_void_p), ("chain_w2", ctypes.c_void_p)]


class _KVCache(ctypes.Structure):
    _fields_ = [("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p),
                ("page_table", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
                ("num_pages", ctypes.c_int)]


_P32 = ctypes.POINTER(ctypes.c_int32)


class SimReport(ctypes.Structure):
    _fields_ = [("tasks_run", ctypes.c_int64),
                ("order_violations", ctypes.c_int64),
                ("duplicate_runs", ctypes.c_int64),
                ("missing_runs", ctypes.c_int64),
                ("deadlocked", ctypes.c_int32),
                ("steps_completed", ctypes.c_int32),
                ("seconds", ctypes.c_double)]


class GraphExport(ctypes.Structure):
    _fields_ = [("n_tasks", ctypes.c_int), ("n_events", ctypes.c_int),
                ("n_ops", ctypes.c_int), ("n_empty", ctypes.c_int),
                ("n_workers", ctypes.c_int), ("attn_chunks", ctypes.c_int)] + [
        (n, _P32) for n in (
            "task_kind", "task_op", "task_layer", "task_tile", "task_row0",
            "task_row1", "task_b", "task_g", "task_c", "task_dep",
            "task_trig", "task_launch", "task_worker", "task_pre_id",
            "event_count", "event_first", "event_last", "op_kind",
            "op_layer", "op_n_tasks")] + [
        ("n_raw_events", ctypes.c_int64), ("n_fused_events", ctypes.c_int64),
        ("n_sched_sms", ctypes.c_int), ("sched_warps_per_sm", ctypes.c_int)]


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libmpk.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with "
            "`python -m task_graph_runtime_gb300.build` (no fallback exists)")
    lib = ctypes.CDLL(path)
    vp, i, st = ctypes.c_void_p, ctypes.c_int, ctypes.c_int
    sig = {
        "mpk_build_tgraph": ([ctypes.POINTER(ModelShape),
                              ctypes.POINTER(TileSizes), i,
                              ctypes.POINTER(vp)], st),
        "mpk_bind_weights": ([vp, ctypes.POINTER(_Weights)], st),
        "mpk_decode_step": ([vp, vp, ctypes.POINTER(_KVCache), vp, vp, vp],
                            st),
        "mpk_decode_steps": ([vp, vp, ctypes.POINTER(_KVCache), vp, vp, i,
                              vp], st),
        "mpk_get_status": ([vp], st),
        "mpk_set_mode": ([vp, i], st),
        "mpk_export_tgraph": ([vp, ctypes.POINTER(GraphExport)], st),
        "mpk_reset": ([vp], st),
        "mpk_destroy_tgraph": ([vp], None),
        "mpk_status_string": ([i], ctypes.c_char_p),
        "mpk_debug_set_wait_timeout_ms": ([vp, i], st),
        "mpk_debug_add_event_count": ([vp, i, i], st),
        "mpk_debug_set_trace": ([vp, i], st),
        "mpk_debug_read_trace": ([vp, vp, i, ctypes.POINTER(i)], st),
        "mpk_debug_read_hidden": ([vp, i, vp], st),
        "mpk_debug_simulate": ([vp, i, ctypes.c_uint32, i, i,
                                ctypes.POINTER(SimReport)], st),
        "mpk_decode_step_noalloc": ([vp, ctypes.POINTER(_Weights), vp,
                                     ctypes.POINTER(_KVCache), vp, vp, vp,
                                     vp], st),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    _lib = lib
    return lib


def _check(status: int, where: str):
    if status != MPK_OK:
        raise MpkError(status, where)


def model_shape(shape, page_size: int = 16, max_pages_per_seq: int = 1
                ) -> ModelShape:
    """ModelShape from a ``synth.ModelShape``-like object."""
    return ModelShape(shape.n_layers, shape.hidden, shape.n_q_heads,
                      shape.n_kv_heads, shape.head_dim, shape.ffn,
                      shape.vocab, shape.rms_eps, shape.rope_theta,
                      int(shape.qk_norm), shape.chain_ffn, page_size,
                      max_pages_per_seq)


# --------------------------------------------------------- C-named calls
def mpk_build_tgraph(shape: ModelShape, tiles: Optional[TileSizes],
                     batch: int) -> int:
    lib = load_library()
    h = ctypes.c_void_p()
    _check(lib.mpk_build_tgraph(ctypes.byref(shape),
                                ctypes.byref(tiles) if tiles else None,
                                batch, ctypes.byref(h)), "mpk_build_tgraph")
    return h.value


def mpk_export_tgraph(handle: int) -> Dict[str, np.ndarray]:
    lib = load_library()
    ex = GraphExport()
    _check(lib.mpk_export_tgraph(handle, ctypes.byref(ex)),
           "mpk_export_tgraph")

    def arr(ptr, n):
        return np.ctypeslib.as_array(ptr, shape=(n,)).copy() if n else \
            np.zeros(0, np.int32)
    out = {k: getattr(ex, k) for k in ("n_tasks", "n_events", "n_ops",
                                        "n_empty", "n_workers", "attn_chunks",
                                        "n_raw_events", "n_fused_events",
                                        "n_sched_sms", "sched_warps_per_sm")}
    for k in ("task_kind", "task_op", "task_layer", "task_tile", "task_row0",
              "task_row1", "task_b", "task_g", "task_c", "task_dep",
              "task_trig", "task_launch", "task_worker", "task_pre_id"):
        out[k] = arr(getattr(ex, k), ex.n_tasks)
    for k in ("event_count", "event_first", "event_last"):
        out[k] = arr(getattr(ex, k), ex.n_events)
    for k in ("op_kind", "op_layer", "op_n_tasks"):
        out[k] = arr(getattr(ex, k), ex.n_ops)
    return out


def mpk_destroy_tgraph(handle: int):
    if handle:
        load_library().mpk_destroy_tgraph(handle)


def mpk_status_string(status: int) -> str:
    return load_library().mpk_status_string(status).decode()


# -------------------------------------------------------------- wrappers
class Weights:
    """Device weight tensors (torch.bfloat16, caller-owned)."""

    def __init__(self, tensors: Dict[str, "object"], shape):
        self.tensors = tensors
        self.shape = shape

    def c_struct(self):
        t = self.tensors
        s = self.shape
        ptr = lambda name: t[name].data_ptr() if name in t else None
        if s.chain_ffn > 0:
            layers = (ctypes.c_void_p * 1)()
            st = _Weights(ptr("embed"), ptr("final_norm"), ptr("lm_head"),
                          ctypes.cast(layers, ctypes.POINTER(ctypes.c_void_p)),
                          ptr("chain_w1"), ptr("chain_w2"))
            return st, layers
        layers = (ctypes.c_void_p * (s.n_layers * len(LAYER_TENSORS)))()
        for l in range(s.n_layers):
            for k, name in enumerate(LAYER_TENSORS):
                layers[l * len(LAYER_TENSORS) + k] = ptr(f"layer{l}.{name}")
        st = _Weights(ptr("embed"), ptr("final_norm"), ptr("lm_head"),
                      ctypes.cast(layers, ctypes.POINTER(ctypes.c_void_p)),
                      None, None)
        return st, layers


class KVCache:
    """Paged KV cache on the device (caller-owned torch tensors)."""

    def __init__(self, k_pool, v_pool, page_table, seq_lens):
        self.k_pool, self.v_pool = k_pool, v_pool
        self.page_table, self.seq_lens = page_table, seq_lens

    def c_struct(self) -> _KVCache:
        return _KVCache(self.k_pool.data_ptr(), self.v_pool.data_ptr(),
                        self.page_table.data_ptr(), self.seq_lens.data_ptr(),
                        int(self.k_pool.shape[1]))


class Graph:
    """A built tGraph (owns the library handle)."""

    def __init__(self, shape, batch: int, num_workers: int = 0,
                 gemv_rows_per_task: int = 0, attn_chunks: int = 0,
                 num_sched_sms: int = 0, sched_warps_per_sm: int = 0,
                 smem_pages: int = 0, page_size: int = 16,
                 max_pages_per_seq: int = 1, mma_rows_per_task: int = 0,
                 coarse_events: int = 0):
        self.shape = shape
        self.batch = batch
        self.c_shape = model_shape(shape, page_size, max_pages_per_seq)
        self.tiles = TileSizes(num_workers, gemv_rows_per_task,
                               mma_rows_per_task, attn_chunks, num_sched_sms,
                               sched_warps_per_sm, smem_pages,
                               coarse_events)
        self.handle = mpk_build_tgraph(self.c_shape, self.tiles, batch)
        self._keep = None

    def export(self) -> Dict[str, np.ndarray]:
        return mpk_export_tgraph(self.handle)

    def bind(self, weights: Weights):
        st, layers = weights.c_struct()
        self._keep = (weights, layers)
        _check(load_library().mpk_bind_weights(self.handle, ctypes.byref(st)),
               "mpk_bind_weights")

    def set_mode(self, mode: int):
        _check(load_library().mpk_set_mode(self.handle, mode), "mpk_set_mode")

    def decode_step(self, tokens, kv: Optional[KVCache], logits, next_tokens,
                    stream=None):
        """Enqueue one step on ``stream`` (a torch.cuda.Stream, a raw
        cudaStream_t int, or None for torch's current stream)."""
        import torch
        if stream is None:
            s = torch.cuda.current_stream().cuda_stream
        elif isinstance(stream, int):
            s = stream
        else:
            s = stream.cuda_stream
        kvs = kv.c_struct() if kv is not None else None
        _check(load_library().mpk_decode_step(
            self.handle, tokens.data_ptr(),
            ctypes.byref(kvs) if kvs is not None else None,
            logits.data_ptr(), next_tokens.data_ptr(), s), "mpk_decode_step")

    def decode_steps(self, tokens, kv: Optional[KVCache], logits,
                     next_tokens, n_steps: int, stream=None):
        """Enqueue ``n_steps`` greedy steps in one launch (megakernel mode);
        ``next_tokens`` is int32 [n_steps, batch], ``logits`` receives the
        last step's."""
        import torch
        if stream is None:
            s = torch.cuda.current_stream().cuda_stream
        elif isinstance(stream, int):
            s = stream
        else:
            s = stream.cuda_stream
        kvs = kv.c_struct() if kv is not None else None
        _check(load_library().mpk_decode_steps(
            self.handle, tokens.data_ptr(),
            ctypes.byref(kvs) if kvs is not None else None,
            logits.data_ptr(), next_tokens.data_ptr(), n_steps, s),
            "mpk_decode_steps")

    def status(self) -> int:
        return load_library().mpk_get_status(self.handle)

    def reset(self):
        _check(load_library().mpk_reset(self.handle), "mpk_reset")

    def set_wait_timeout_ms(self, ms: int):
        _check(load_library().mpk_debug_set_wait_timeout_ms(self.handle, ms),
               "mpk_debug_set_wait_timeout_ms")

    def add_event_count(self, event: int, delta: int):
        _check(load_library().mpk_debug_add_event_count(self.handle, event,
                                                        delta),
               "mpk_debug_add_event_count")

    def set_trace(self, capacity: int):
        _check(load_library().mpk_debug_set_trace(self.handle, capacity),
               "mpk_debug_set_trace")

    def read_trace(self, capacity: int) -> np.ndarray:
        """uint64 [n, 8]: task | worker << 32, looked, ready, staged, pages
        done, body done, triggered (ns; 0 where not recorded), 0."""
        buf = np.zeros((capacity, 8), np.uint64)
        n = ctypes.c_int(0)
        _check(load_library().mpk_debug_read_trace(
            self.handle, buf.ctypes.data, capacity, ctypes.byref(n)),
            "mpk_debug_read_trace")
        return buf[:n.value]

    def simulate(self, steps: int = 2, seed: int = 0, max_delay_us: int = 20,
                 timeout_ms: int = 20000) -> Dict[str, float]:
        """CPU model of the runtime protocol on this graph's encoding
        (mpk_debug_simulate): host threads for workers and scheduler warps,
        random task delays."""
        rep = SimReport()
        _check(load_library().mpk_debug_simulate(
            self.handle, steps, seed, max_delay_us, timeout_ms,
            ctypes.byref(rep)), "mpk_debug_simulate")
        return {k: getattr(rep, k) for k, _ in SimReport._fields_}

    def read_hidden(self, layer: int) -> np.ndarray:
        """bf16 bits [batch, hidden] of the residual stream entering decoder
        layer ``layer`` (``n_layers``: the final RMSNorm's input) in the last
        step."""
        out = np.zeros((self.batch, self.shape.hidden), np.uint16)
        _check(load_library().mpk_debug_read_hidden(
            self.handle, layer, out.ctypes.data), "mpk_debug_read_hidden")
        return out

    def close(self):
        if self.handle:
            mpk_destroy_tgraph(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def mpk_decode_step_noalloc(graph: "Graph", weights: Weights, tokens, kv,
                            logits, next_tokens, status=None, stream=None):
    """One decode step with every piece of scratch in the library's static
    device array (no device allocation); see include/mpk.h."""
    import torch
    s = (torch.cuda.current_stream().cuda_stream if stream is None
         else stream if isinstance(stream, int) else stream.cuda_stream)
    st, layers = weights.c_struct()
    kvs = kv.c_struct() if kv is not None else None
    _check(load_library().mpk_decode_step_noalloc(
        graph.handle, ctypes.byref(st), tokens.data_ptr(),
        ctypes.byref(kvs) if kvs is not None else None, logits.data_ptr(),
        next_tokens.data_ptr(),
        status.data_ptr() if status is not None else None, s),
        "mpk_decode_step_noalloc")
    return layers          # keep the host pointer array alive until here
