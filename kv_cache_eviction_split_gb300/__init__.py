"""GB300-native KV-cache eviction: DropKV removal scores, budgeted top-k, ragged compaction.

A thin ctypes binding over ``libkvevict.so`` (the C ABI in ``include/kvevict.h``).
Every step of the path runs in the library's CUDA kernels; this module only
marshals arguments (torch tensors -> pointers, sizes, the caller's stream)
and allocates outputs and workspaces with torch.  There is no CPU fallback:
if the library is missing, ``load()`` raises.

Names follow the C ABI: ``kv_score``, ``kv_score_attention``,
``kv_score_rescore``, ``kv_make_offsets``, ``kv_select_topk``, ``kv_compact``,
``kv_check_status``, ``kv_budgets_pyramid``, ``kv_budgets_ripple``.
"""
from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np

from . import _build

__all__ = ["KvError", "Problem", "load", "build", "kv_score", "kv_score_attention",
           "kv_score_rescore", "kv_make_offsets", "kv_select_topk", "kv_compact",
           "kv_check_status", "kv_score_noalloc", "kv_budgets_pyramid", "kv_budgets_ripple", "kv_budgets_uniform",
           "kv_set_wait_limit_ns", "kv_get_wait_limit_ns", "kv_pool_scores", "kv_head_budgets",
           "kv_block_scores", "kv_compact_blocks", "kv_budgets_fraction", "BlockBuffers",
           "evict_blocks", "EXPORTED_SYMBOLS", "HostPipeline", "PinnedTensor", "kv_evict_host",
           "kv_evict_host_workspace_size",
           "evict", "KV_SCORE_DROPKV", "KV_SCORE_DROPKV_SQUARED", "KV_SCORE_ATTN_SUM"]

KV_OK, KV_ERR_INVALID_ARG, KV_ERR_BUDGET, KV_ERR_WORKSPACE, KV_ERR_CUDA, KV_ERR_TIMEOUT, \
    KV_ERR_UNSUPPORTED = range(7)
# kv_problem.score_rule
KV_SCORE_DROPKV, KV_SCORE_DROPKV_SQUARED, KV_SCORE_ATTN_SUM = range(3)

EXPORTED_SYMBOLS = ("kv_score_workspace_size", "kv_score", "kv_score_attention",
                    "kv_score_rescore", "kv_make_offsets", "kv_select_workspace_size",
                    "kv_select_topk", "kv_compact", "kv_check_status", "kv_status_string",
                    "kv_budgets_pyramid", "kv_budgets_ripple", "kv_score_noalloc",
                    "kv_set_wait_limit_ns", "kv_get_wait_limit_ns", "kv_pool_scores",
                    "kv_head_budgets", "kv_block_scores", "kv_compact_blocks",
                    "kv_budgets_fraction", "kv_evict_fused", "kv_evict_host_workspace_size",
                    "kv_evict_host")


class KvError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__("%s: %s" % (where, status_string(code)))


class _KvProblem(ctypes.Structure):
    _fields_ = [("num_requests", ctypes.c_int32), ("num_layers", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("window", ctypes.c_int32),
                ("num_sinks", ctypes.c_int32), ("score_rule", ctypes.c_int32),
                ("seq_offsets_host", ctypes.POINTER(ctypes.c_int64)),
                ("seq_offsets_dev", ctypes.c_void_p), ("softmax_scale", ctypes.c_float)]


class _KvHostPlan(ctypes.Structure):
    _fields_ = [("group_layers", ctypes.c_int32), ("pool_kernel", ctypes.c_int32),
                ("head_budgets", ctypes.c_int32), ("fused", ctypes.c_int32)]


_lib = None


def build(force: bool = False, debug: bool = False) -> str:
    """Build libkvevict.so (debug=True: the bounds-checked libkvevict_debug.so)."""
    return _build.build(force=force, debug=debug)


_debug_lib = None


def load_debug():
    """The bounds-checked build (libkvevict_debug.so), bound like load()'s library:
    the same C ABI, with every TMA coordinate, workspace offset and gather index
    checked on the device (KV_ERR_INVALID_ARG in the status word on a failed
    check).  Its functions are called on the returned handle directly."""
    global _debug_lib
    if _debug_lib is None:
        if not os.path.exists(_build.LIB_PATH_DEBUG):
            raise RuntimeError("libkvevict_debug.so not found: run build(debug=True)")
        _debug_lib = _bind(ctypes.CDLL(_build.LIB_PATH_DEBUG))
    return _debug_lib


def load(path: Optional[str] = None):
    """Load ``libkvevict.so``; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or _build.LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError("libkvevict.so not found at %s: run "
                           "kv_cache_eviction_split_gb300.build() (needs nvcc)" % path)
    _lib = _bind(ctypes.CDLL(path))
    return _lib


def _bind(lib):
    """Sets the argument and result types of every exported function of `lib`."""
    P = ctypes.POINTER(_KvProblem)
    vp, sz, i32, i64, f64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.c_int64, \
        ctypes.c_double
    szp = ctypes.POINTER(ctypes.c_size_t)
    sig = {
        "kv_score_workspace_size": [P, szp],
        "kv_score": [P, vp, vp, vp, vp, vp, sz, vp],
        "kv_score_attention": [P, vp, vp, vp, vp, sz, vp],
        "kv_score_rescore": [P, vp, vp, vp, vp, vp, sz, vp],
        "kv_make_offsets": [P, ctypes.POINTER(i32), ctypes.POINTER(i64)],
        "kv_select_workspace_size": [P, szp],
        "kv_select_topk": [P, vp, vp, vp, vp, vp, sz, vp],
        "kv_compact": [P, vp, vp, vp, vp, i64, vp, vp, vp],
        "kv_check_status": [vp, vp, ctypes.POINTER(i32)],
        "kv_budgets_pyramid": [i32, i32, f64, f64, f64, ctypes.POINTER(i32)],
        "kv_budgets_ripple": [i32, i32, ctypes.POINTER(f64), f64, f64, ctypes.POINTER(i32)],
        "kv_score_noalloc": [P, vp, vp, vp, vp, vp],
        "kv_pool_scores": [P, i32, vp, vp, vp],
        "kv_head_budgets": [P, vp, vp, vp, vp, vp, vp, sz, vp],
        "kv_block_scores": [P, i32, vp, vp, vp],
        "kv_compact_blocks": [P, i32, vp, vp, vp, vp, vp, i64, vp, vp, vp],
        "kv_budgets_fraction": [P, f64, ctypes.POINTER(i32)],
        "kv_evict_fused": [P, vp, vp, vp, vp, vp, i64, vp, vp, vp, vp, vp, sz, vp],
        "kv_evict_host_workspace_size": [P, ctypes.POINTER(_KvHostPlan), ctypes.POINTER(i32),
                                         szp],
        "kv_evict_host": [P, ctypes.POINTER(_KvHostPlan), vp, vp, vp, ctypes.POINTER(i32),
                          ctypes.POINTER(i64), vp, vp, vp, vp, sz, vp, ctypes.POINTER(i32)],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.kv_status_string.argtypes = [ctypes.c_int]
    lib.kv_status_string.restype = ctypes.c_char_p
    lib.kv_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    lib.kv_set_wait_limit_ns.restype = None
    lib.kv_get_wait_limit_ns.argtypes = []
    lib.kv_get_wait_limit_ns.restype = ctypes.c_uint64
    return lib


def status_string(code: int) -> str:
    return load().kv_status_string(int(code)).decode()


def _check(code: int, where: str):
    if code != KV_OK:
        raise KvError(code, where)


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


@dataclass
class Problem:
    """Shapes of one eviction problem; owns the host and device cu_seqlens."""
    lengths: Sequence[int]
    num_layers: int
    num_kv_heads: int
    num_q_heads: int
    head_dim: int
    window: int
    num_sinks: int = 4
    softmax_scale: Optional[float] = None
    device: object = "cuda"
    score_rule: int = KV_SCORE_DROPKV   # what kv_score sums (KV_SCORE_*)
    pool_kernel: int = 1                # evict(): max-pool width before selection (1: none)
    head_budgets: bool = False          # evict(): per-head budgets from the scores (AdaDropKV)

    def __post_init__(self):
        import torch
        self.cu_host = np.concatenate([[0], np.cumsum(np.asarray(self.lengths, dtype=np.int64))]
                                      ).astype(np.int64)
        self.cu_dev = torch.from_numpy(self.cu_host).to(self.device) if len(self.lengths) else \
            torch.zeros(1, dtype=torch.int64, device=self.device)
        scale = self.softmax_scale if self.softmax_scale is not None else 1.0 / math.sqrt(self.head_dim)
        self._c = _KvProblem(len(self.lengths), self.num_layers, self.num_kv_heads,
                             self.num_q_heads, self.head_dim, self.window, self.num_sinks,
                             int(self.score_rule),
                             self.cu_host.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                             self.cu_dev.data_ptr(), float(scale))

    @property
    def c(self):
        return ctypes.byref(self._c)

    @property
    def num_requests(self) -> int:
        return len(self.lengths)

    @property
    def num_units(self) -> int:
        return self.num_requests * self.num_layers * self.num_kv_heads

    @property
    def total_tokens(self) -> int:
        return int(self.cu_host[-1])

    def block_view(self, block_layers: int) -> "Problem":
        """The problem whose units are (request, block of `block_layers` layers): one KV
        head and one query head per block, same requests, window and sinks."""
        if block_layers < 1 or self.num_layers % block_layers:
            raise ValueError("num_layers must be a multiple of block_layers")
        return Problem(list(self.lengths), self.num_layers // block_layers, 1, 1, self.head_dim,
                       self.window, self.num_sinks, self.softmax_scale, self.cu_dev.device)

    @classmethod
    def for_workload(cls, wl, device="cuda", score_rule: int = KV_SCORE_DROPKV,
                     pool_kernel: int = 1, head_budgets: bool = False) -> "Problem":
        return cls(wl.seq_lengths(), wl.num_layers, wl.num_kv_heads, wl.num_q_heads,
                   wl.head_dim, wl.window, wl.num_sinks, device=device, score_rule=score_rule,
                   pool_kernel=pool_kernel, head_budgets=head_budgets)


# ---------------------------------------------------------------------------
# entry points (same names as the C ABI)
# ---------------------------------------------------------------------------
def kv_score_workspace_size(prob: Problem) -> int:
    n = ctypes.c_size_t()
    _check(load().kv_score_workspace_size(prob.c, ctypes.byref(n)), "kv_score_workspace_size")
    return n.value


def kv_select_workspace_size(prob: Problem) -> int:
    n = ctypes.c_size_t()
    _check(load().kv_select_workspace_size(prob.c, ctypes.byref(n)), "kv_select_workspace_size")
    return n.value


def kv_score(prob, q, k, v, scores, workspace, stream=None):
    _check(load().kv_score(prob.c, _ptr(q), _ptr(k), _ptr(v), _ptr(scores), _ptr(workspace),
                           workspace.numel() * workspace.element_size(), _stream(stream)),
           "kv_score")


def kv_score_attention(prob, q, k, v, workspace, stream=None):
    _check(load().kv_score_attention(prob.c, _ptr(q), _ptr(k), _ptr(v), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(),
                                     _stream(stream)), "kv_score_attention")


def kv_score_rescore(prob, q, k, v, scores, workspace, stream=None):
    _check(load().kv_score_rescore(prob.c, _ptr(q), _ptr(k), _ptr(v), _ptr(scores),
                                   _ptr(workspace), workspace.numel() * workspace.element_size(),
                                   _stream(stream)), "kv_score_rescore")


def kv_score_noalloc(prob, q, k, v, scores, stream=None):
    """kv_score with the library's own fixed scratch (no workspace argument)."""
    _check(load().kv_score_noalloc(prob.c, _ptr(q), _ptr(k), _ptr(v), _ptr(scores),
                                   _stream(stream)), "kv_score_noalloc")


def kv_pool_scores(prob, kernel: int, scores_in, scores_out, stream=None):
    _check(load().kv_pool_scores(prob.c, int(kernel), _ptr(scores_in), _ptr(scores_out),
                                 _stream(stream)), "kv_pool_scores")


def kv_head_budgets(prob, scores, budgets_dev, offsets_dev, budgets_out, offsets_out, workspace,
                    stream=None):
    _check(load().kv_head_budgets(prob.c, _ptr(scores), _ptr(budgets_dev), _ptr(offsets_dev),
                                  _ptr(budgets_out), _ptr(offsets_out), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), _stream(stream)),
           "kv_head_budgets")


def kv_block_scores(prob, block_layers: int, scores, block_scores, stream=None):
    _check(load().kv_block_scores(prob.c, int(block_layers), _ptr(scores), _ptr(block_scores),
                                  _stream(stream)), "kv_block_scores")


def kv_compact_blocks(prob, block_layers: int, k, v, block_sel, block_offsets, offsets,
                      total_rows: int, k_out, v_out, stream=None):
    _check(load().kv_compact_blocks(prob.c, int(block_layers), _ptr(k), _ptr(v), _ptr(block_sel),
                                    _ptr(block_offsets), _ptr(offsets), int(total_rows),
                                    _ptr(k_out), _ptr(v_out), _stream(stream)),
           "kv_compact_blocks")


def kv_budgets_fraction(prob, q: float) -> np.ndarray:
    out = np.zeros(prob.num_units, dtype=np.int32)
    _check(load().kv_budgets_fraction(prob.c, float(q),
                                      out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))),
           "kv_budgets_fraction")
    return out


def kv_make_offsets(prob, budgets_host: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(budgets_host, dtype=np.int32).reshape(-1)
    out = np.zeros(b.size + 1, dtype=np.int64)
    _check(load().kv_make_offsets(prob.c, b.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                  out.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))),
           "kv_make_offsets")
    return out


def kv_select_topk(prob, scores, budgets_dev, offsets_dev, sel_idx, workspace, stream=None):
    _check(load().kv_select_topk(prob.c, _ptr(scores), _ptr(budgets_dev), _ptr(offsets_dev),
                                 _ptr(sel_idx), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _stream(stream)),
           "kv_select_topk")


def kv_evict_fused(prob, q_win, k, v, budgets_dev, offsets_dev, total_rows: int, scores,
                   sel_idx, k_out, v_out, workspace, stream=None):
    """kv_score + kv_select_topk + kv_compact in one cooperative launch; device errors
    (selection budgets included) go to the score workspace's status word."""
    _check(load().kv_evict_fused(prob.c, _ptr(q_win), _ptr(k), _ptr(v), _ptr(budgets_dev),
                                 _ptr(offsets_dev), int(total_rows), _ptr(scores),
                                 _ptr(sel_idx), _ptr(k_out), _ptr(v_out), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _stream(stream)),
           "kv_evict_fused")


def kv_compact(prob, k, v, sel_idx, offsets_dev, total_rows: int, k_out, v_out, stream=None):
    _check(load().kv_compact(prob.c, _ptr(k), _ptr(v), _ptr(sel_idx), _ptr(offsets_dev),
                             int(total_rows), _ptr(k_out), _ptr(v_out), _stream(stream)),
           "kv_compact")


def kv_check_status(workspace, stream=None) -> int:
    st = ctypes.c_int32()
    _check(load().kv_check_status(_ptr(workspace), _stream(stream), ctypes.byref(st)),
           "kv_check_status")
    return st.value


def kv_set_wait_limit_ns(ns: int) -> None:
    """Limit of the kernels' device waits for launches after this call (default 2 s)."""
    load().kv_set_wait_limit_ns(int(ns))


def kv_get_wait_limit_ns() -> int:
    return int(load().kv_get_wait_limit_ns())


def kv_budgets_uniform(num_layers: int, mean_budget: int) -> np.ndarray:
    return np.full(num_layers, int(mean_budget), dtype=np.int32)


def kv_budgets_pyramid(num_layers: int, mean_budget: int, hi: float = 1.8, lo: float = 0.2,
                       curve: float = 1.0) -> np.ndarray:
    out = np.zeros(num_layers, dtype=np.int32)
    _check(load().kv_budgets_pyramid(num_layers, mean_budget, hi, lo, curve,
                                     out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))),
           "kv_budgets_pyramid")
    return out


def kv_budgets_ripple(num_layers: int, mean_budget: int, profile, beta: float = 2.0,
                      gamma: float = math.inf) -> np.ndarray:
    prof = np.ascontiguousarray(profile, dtype=np.float64)
    out = np.zeros(num_layers, dtype=np.int32)
    _check(load().kv_budgets_ripple(num_layers, mean_budget,
                                    prof.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), beta,
                                    gamma, out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))),
           "kv_budgets_ripple")
    return out


# ---------------------------------------------------------------------------
# convenience: the whole path with torch-allocated outputs
# ---------------------------------------------------------------------------
class Buffers:
    """Device outputs and workspaces of one problem, allocated once and reused."""

    def __init__(self, prob: Problem, budgets_host: np.ndarray):
        import torch
        dev = prob.cu_dev.device
        self.budgets_host = np.ascontiguousarray(budgets_host, dtype=np.int32).reshape(-1)
        self.offsets_host = kv_make_offsets(prob, self.budgets_host)
        self.total_rows = int(self.offsets_host[-1])
        self.budgets = torch.from_numpy(self.budgets_host).to(dev)
        self.offsets = torch.from_numpy(self.offsets_host).to(dev)
        N, d = prob.total_tokens, prob.head_dim
        self.scores = torch.empty((prob.num_layers, prob.num_kv_heads, N), dtype=torch.float32,
                                  device=dev)
        self.score_ws = torch.zeros(max(kv_score_workspace_size(prob), 256), dtype=torch.uint8,
                                    device=dev)
        self.select_ws = torch.zeros(max(kv_select_workspace_size(prob), 256), dtype=torch.uint8,
                                     device=dev)
        self.sel = torch.empty(max(self.total_rows, 1), dtype=torch.int32, device=dev)
        self.k_out = torch.empty((max(self.total_rows, 1), d), dtype=torch.bfloat16, device=dev)
        self.v_out = torch.empty_like(self.k_out)
        self.pooled = torch.empty_like(self.scores) if prob.pool_kernel > 1 else None
        # per-head budgets and their offsets (written on the device by kv_head_budgets)
        self.head_budgets = torch.empty_like(self.budgets) if prob.head_budgets else None
        self.head_offsets = torch.empty_like(self.offsets) if prob.head_budgets else None


def evict(prob: Problem, q, k, v, bufs: Buffers, stream=None, fused: bool = False):
    """Score (pool, if prob.pool_kernel > 1; per-head budgets, if prob.head_budgets),
    select and compact on `stream`; returns (sel_idx, k_out, v_out, offsets).  With
    fused=True (no pooling, no per-head budgets) the path runs as one launch."""
    if fused:
        if prob.pool_kernel > 1 or prob.head_budgets:
            raise ValueError("the fused path takes neither pooling nor per-head budgets")
        kv_evict_fused(prob, q, k, v, bufs.budgets, bufs.offsets, bufs.total_rows, bufs.scores,
                       bufs.sel, bufs.k_out, bufs.v_out, bufs.score_ws, stream)
        n = bufs.total_rows
        return bufs.sel[:n], bufs.k_out[:n], bufs.v_out[:n], bufs.offsets
    kv_score(prob, q, k, v, bufs.scores, bufs.score_ws, stream)
    ranked = bufs.scores
    if prob.pool_kernel > 1:
        kv_pool_scores(prob, prob.pool_kernel, bufs.scores, bufs.pooled, stream)
        ranked = bufs.pooled
    budgets, offsets = bufs.budgets, bufs.offsets
    if prob.head_budgets:
        kv_head_budgets(prob, ranked, bufs.budgets, bufs.offsets, bufs.head_budgets,
                        bufs.head_offsets, bufs.select_ws, stream)
        budgets, offsets = bufs.head_budgets, bufs.head_offsets
    kv_select_topk(prob, ranked, budgets, offsets, bufs.sel, bufs.select_ws, stream)
    kv_compact(prob, k, v, bufs.sel, offsets, bufs.total_rows, bufs.k_out, bufs.v_out, stream)
    n = bufs.total_rows
    return bufs.sel[:n], bufs.k_out[:n], bufs.v_out[:n], offsets


# ---------------------------------------------------------------------------
# block eviction (BellowsKV): one decision per block of consecutive layers
# ---------------------------------------------------------------------------
class BlockBuffers:
    """Buffers of block eviction for `prob`: blocks of `block_layers` layers, each keeping
    its sinks, window and the fraction `q` of the rest, pooled with `pool_kernel`."""

    def __init__(self, prob: Problem, block_layers: int, q: float, pool_kernel: int = 13):
        import torch
        dev = prob.cu_dev.device
        self.block_layers = block_layers
        self.pool_kernel = pool_kernel
        self.bprob = prob.block_view(block_layers)
        nblk = self.bprob.num_layers
        N = prob.total_tokens
        self.block_budgets_host = kv_budgets_fraction(self.bprob, q)
        self.block_offsets_host = kv_make_offsets(self.bprob, self.block_budgets_host)
        # every (layer, head) of a block keeps its block's tokens
        per_unit = np.repeat(self.block_budgets_host.reshape(prob.num_requests, nblk),
                             block_layers, axis=1)
        per_unit = np.repeat(per_unit[:, :, None], prob.num_kv_heads, axis=2).reshape(-1)
        self.unit_offsets_host = kv_make_offsets(prob, per_unit)
        self.total_rows = int(self.unit_offsets_host[-1])
        self.block_budgets = torch.from_numpy(self.block_budgets_host).to(dev)
        self.block_offsets = torch.from_numpy(self.block_offsets_host).to(dev)
        self.unit_offsets = torch.from_numpy(self.unit_offsets_host).to(dev)
        self.block_scores = torch.empty((nblk, 1, N), dtype=torch.float32, device=dev)
        self.pooled = torch.empty_like(self.block_scores) if pool_kernel > 1 else None
        self.select_ws = torch.zeros(max(kv_select_workspace_size(self.bprob), 256),
                                     dtype=torch.uint8, device=dev)
        self.sel = torch.empty(max(int(self.block_offsets_host[-1]), 1), dtype=torch.int32,
                               device=dev)
        self.k_out = torch.empty((max(self.total_rows, 1), prob.head_dim), dtype=torch.bfloat16,
                                 device=dev)
        self.v_out = torch.empty_like(self.k_out)


def evict_blocks(prob, scores, k, v, bb: BlockBuffers, stream=None):
    """Block eviction from per-(layer, head) scores already computed by kv_score:
    block sums, pooling, one selection per (request, block), and the compaction of every
    layer and head with its block's tokens.  Returns (block_sel, k_out, v_out, offsets)."""
    kv_block_scores(prob, bb.block_layers, scores, bb.block_scores, stream)
    ranked = bb.block_scores
    if bb.pool_kernel > 1:
        kv_pool_scores(bb.bprob, bb.pool_kernel, bb.block_scores, bb.pooled, stream)
        ranked = bb.pooled
    kv_select_topk(bb.bprob, ranked, bb.block_budgets, bb.block_offsets, bb.sel, bb.select_ws,
                   stream)
    kv_compact_blocks(prob, bb.block_layers, k, v, bb.sel, bb.block_offsets, bb.unit_offsets,
                      bb.total_rows, bb.k_out, bb.v_out, stream)
    n = bb.total_rows
    return bb.sel[:int(bb.block_offsets_host[-1])], bb.k_out[:n], bb.v_out[:n], bb.unit_offsets


# ---------------------------------------------------------------------------
# eviction from host memory, layer groups pipelined against the copies
# ---------------------------------------------------------------------------
def kv_evict_host_workspace_size(prob: Problem, plan, budgets_host: np.ndarray) -> int:
    b = np.ascontiguousarray(budgets_host, dtype=np.int32).reshape(-1)
    n = ctypes.c_size_t()
    _check(load().kv_evict_host_workspace_size(
        prob.c, ctypes.byref(plan), b.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
        ctypes.byref(n)), "kv_evict_host_workspace_size")
    return n.value


def kv_evict_host(prob: Problem, plan, q_host, k_host, v_host, budgets_host: np.ndarray,
                  offsets_host: np.ndarray, sel_host, k_out_host, v_out_host, workspace,
                  stream=None) -> int:
    """The C entry point: host inputs in, host outputs out; returns the device status."""
    b = np.ascontiguousarray(budgets_host, dtype=np.int32).reshape(-1)
    assert offsets_host.dtype == np.int64 and offsets_host.flags.c_contiguous
    st = ctypes.c_int32()
    _check(load().kv_evict_host(
        prob.c, ctypes.byref(plan), _ptr(q_host), _ptr(k_host), _ptr(v_host),
        b.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
        offsets_host.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), _ptr(sel_host),
        _ptr(k_out_host), _ptr(v_out_host), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream), ctypes.byref(st)),
        "kv_evict_host")
    return st.value


_cudart_lib = None


def _cudart():
    """The CUDA runtime library torch loaded (for cudaHostAlloc / cudaFreeHost)."""
    global _cudart_lib
    if _cudart_lib is None:
        import torch  # noqa: F401  (loads the runtime)
        for name in ("libcudart.so.13", "libcudart.so.12", "libcudart.so"):
            try:
                lib = ctypes.CDLL(name)
            except OSError:
                continue
            lib.cudaHostAlloc.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_size_t,
                                          ctypes.c_uint]
            lib.cudaHostAlloc.restype = ctypes.c_int
            lib.cudaFreeHost.argtypes = [ctypes.c_void_p]
            lib.cudaFreeHost.restype = ctypes.c_int
            _cudart_lib = lib
            break
    return _cudart_lib


class _HostAllocation:
    """One cudaHostAlloc block, freed when the last tensor viewing it is gone."""

    def __init__(self, nbytes: int):
        self.ptr = None
        lib = _cudart()
        if lib is None:
            raise RuntimeError("no CUDA runtime library to page-lock host memory with")
        p = ctypes.c_void_p()
        err = lib.cudaHostAlloc(ctypes.byref(p), ctypes.c_size_t(nbytes), 0)
        if err != 0 or not p.value:
            raise RuntimeError("cudaHostAlloc of %d bytes failed (error %d)" % (nbytes, err))
        self.ptr = p.value
        self.lib = lib

    def __del__(self):
        if self.ptr:
            self.lib.cudaFreeHost(ctypes.c_void_p(self.ptr))
            self.ptr = None


def PinnedTensor(shape, dtype):
    """A page-locked host tensor of exactly its size (cudaHostAlloc; torch's own
    pinned allocator rounds every block up to a power of two, which at tens of GB
    nearly doubles the locked host memory).  The allocation lives as long as any
    tensor that views it."""
    import torch
    numel = int(np.prod(shape)) if isinstance(shape, (tuple, list)) else int(shape)
    elsize = torch.empty((), dtype=dtype).element_size()
    nbytes = max(numel * elsize, elsize)
    block = _HostAllocation(nbytes)
    buf = (ctypes.c_uint8 * nbytes).from_address(block.ptr)
    buf._owner = block                      # the buffer, hence every view, holds the block
    arr = np.frombuffer(buf, dtype=np.uint8, count=nbytes)
    return torch.from_numpy(arr).view(dtype)[:numel].view(shape)


class HostPipeline:
    """Eviction of a problem whose Q, K and V are in host memory, through kv_evict_host.

    The layers are taken in groups of `group_layers`: while group g is scored,
    selected and compacted, group g+1's inputs are copied in and group g-1's kept
    indices and rows are copied out (the copies overlap the kernels when the host
    buffers are pinned).  Device memory holds two groups, not the whole problem.
    This class allocates the device workspace and pinned host outputs once;
    run() is one C call.  Outputs are in the standard unit order.
    """

    def __init__(self, prob: Problem, budgets_host: np.ndarray, group_layers: int = 4,
                 fused: bool = False):
        import torch
        if fused and (prob.pool_kernel > 1 or prob.head_budgets):
            raise ValueError("the fused path takes neither pooling nor per-head budgets")
        dev = prob.cu_dev.device
        self.prob = prob
        self.fused = fused
        L = prob.num_layers
        group_layers = max(1, min(int(group_layers), L))
        self.group_layers = group_layers
        self.groups = [(l0, min(L, l0 + group_layers)) for l0 in range(0, L, group_layers)]
        self.plan = _KvHostPlan(int(group_layers), int(prob.pool_kernel), int(prob.head_budgets),
                                int(fused))
        self.budgets_host = np.ascontiguousarray(budgets_host, dtype=np.int32).reshape(-1)
        self.offsets = kv_make_offsets(prob, self.budgets_host)
        self.total_rows = int(self.offsets[-1])
        nbytes = kv_evict_host_workspace_size(prob, self.plan, self.budgets_host)
        self.workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
        rows, d = max(self.total_rows, 1), prob.head_dim
        self.sel_host = PinnedTensor(rows, torch.int32)
        self.k_out_host = PinnedTensor((rows, d), torch.bfloat16)
        self.v_out_host = PinnedTensor((rows, d), torch.bfloat16)

    @property
    def h2d_bytes(self) -> int:
        p = self.prob
        q = p.num_requests * p.num_layers * p.num_q_heads * p.window * p.head_dim * 2
        return q + 2 * p.num_layers * p.num_kv_heads * p.total_tokens * p.head_dim * 2

    @property
    def d2h_bytes(self) -> int:
        return self.total_rows * (4 + 2 * self.prob.head_dim * 2)

    def run(self, q_host, k_host, v_host, stream=None):
        """One kv_evict_host call; returns (sel, k_out, v_out, offsets) in host memory.
        Raises KvError if a kernel posted a device status."""
        offsets = np.zeros(self.prob.num_units + 1, dtype=np.int64)
        code = kv_evict_host(self.prob, self.plan, q_host, k_host, v_host, self.budgets_host,
                             offsets, self.sel_host, self.k_out_host, self.v_out_host,
                             self.workspace, stream)
        if code != KV_OK:
            raise KvError(code, "kv_evict_host (device status)")
        self.offsets = offsets
        n = self.total_rows
        return self.sel_host[:n], self.k_out_host[:n], self.v_out_host[:n], self.offsets
