"""Python binding of libdsa (the GB300 DSA sparse-attention path).

Argument marshalling only: every step runs in the CUDA kernels behind the C ABI
declared in ``include/dsa.h``.  torch is used for device memory and streams.
There is no CPU fallback: importing this package raises if ``libdsa.so`` has
not been built (``python -c "import __graft_entry__ as g; g.build()"``).
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdsa.so")

DSA_OK = 0
STATUS_NAMES = {0: "DSA_OK", 1: "DSA_ERR_INVALID_ARG", 2: "DSA_ERR_UNSUPPORTED", 3: "DSA_ERR_WORKSPACE",
                4: "DSA_ERR_CUDA", 5: "DSA_ERR_TIMEOUT", 6: "DSA_ERR_DEVICE_CHECK"}
DSA_F32, DSA_BF16, DSA_E4M3, DSA_MXFP8_E4M3, DSA_E4M3_T128 = 0, 1, 2, 3, 4

EXPORTED = ("dsa_abi_version", "dsa_status_string", "dsa_last_error", "dsa_last_plan",
            "dsa_indexer_scores", "dsa_topk", "dsa_sparse_mla_attn_workspace_size",
            "dsa_sparse_mla_attn", "dsa_decode_workspace_size", "dsa_decode_step",
            "dsa_decode_step_static_ws", "dsa_index_cache_append", "dsa_index_cache_append_mx",
            "dsa_latent_cache_append", "dsa_debug_withhold_arrival",
            "dsa_indexer_prolog_workspace_size", "dsa_indexer_prolog",
            "dsa_check_status")
STATIC_WORKSPACE_BYTES = 32 << 20   # DSA_STATIC_WORKSPACE_BYTES


class SeqDesc(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("T", ctypes.c_int32), ("max_ctx", ctypes.c_int32),
                ("q_per_seq", ctypes.c_int32), ("q_seq", ctypes.c_void_p), ("q_pos", ctypes.c_void_p),
                ("block_table", ctypes.c_void_p), ("bt_stride", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("cache_rows", ctypes.c_int64)]


class IndexerDesc(ctypes.Structure):
    _fields_ = [("H_I", ctypes.c_int32), ("D_I", ctypes.c_int32), ("dtype", ctypes.c_int),
                ("q", ctypes.c_void_p), ("q_scale", ctypes.c_void_p), ("w", ctypes.c_void_p),
                ("k_cache", ctypes.c_void_p), ("k_scale", ctypes.c_void_p)]


class MlaDesc(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int32), ("d_latent", ctypes.c_int32), ("d_rope", ctypes.c_int32),
                ("dtype", ctypes.c_int), ("q", ctypes.c_void_p), ("kv_cache", ctypes.c_void_p),
                ("row_bytes", ctypes.c_int64), ("softmax_scale", ctypes.c_float)]


class PrologDesc(ctypes.Structure):
    _fields_ = [("d_model", ctypes.c_int32), ("d_q", ctypes.c_int32), ("H_I", ctypes.c_int32),
                ("D_I", ctypes.c_int32), ("x", ctypes.c_void_p), ("x_q", ctypes.c_void_p), ("w_q", ctypes.c_void_p),
                ("w_k", ctypes.c_void_p), ("w_w", ctypes.c_void_p), ("gamma", ctypes.c_void_p),
                ("beta", ctypes.c_void_p)]


class DSAError(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {detail}")
        self.status = status


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it first (__graft_entry__.build())")
    lib = ctypes.CDLL(LIB_PATH)
    P, C = ctypes.c_void_p, ctypes.c_int
    sig = {
        "dsa_abi_version": (C, []),
        "dsa_status_string": (ctypes.c_char_p, [C]),
        "dsa_last_error": (ctypes.c_char_p, []),
        "dsa_last_plan": (ctypes.c_char_p, []),
        "dsa_indexer_scores": (C, [P, P, P, ctypes.c_int64, P]),
        "dsa_topk": (C, [P, P, ctypes.c_int64, ctypes.c_int32, P, P]),
        "dsa_sparse_mla_attn_workspace_size": (ctypes.c_size_t, [P, P, ctypes.c_int32]),
        "dsa_sparse_mla_attn": (C, [P, P, P, ctypes.c_int32, P, P, P, ctypes.c_size_t, P]),
        "dsa_decode_workspace_size": (ctypes.c_size_t, [P, P, P, ctypes.c_int32]),
        "dsa_decode_step": (C, [P, P, P, ctypes.c_int32, P, P, P, P, ctypes.c_size_t, P]),
        "dsa_decode_step_static_ws": (C, [P, P, P, ctypes.c_int32, P, P, P, P]),
        "dsa_index_cache_append": (C, [P, ctypes.c_int32, C, P, P, P, P]),
        "dsa_index_cache_append_mx": (C, [P, ctypes.c_int32, C, P, P, P, P]),
        "dsa_latent_cache_append": (C, [P, P, P, P, P]),
        "dsa_debug_withhold_arrival": (C, [ctypes.c_int32, ctypes.c_uint64]),
        "dsa_indexer_prolog_workspace_size": (ctypes.c_size_t, [P, P]),
        "dsa_indexer_prolog": (C, [P, P, P, P, P, P, P, P, ctypes.c_size_t, P]),
        "dsa_check_status": (C, [P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    return lib


_lib = _load()


def abi_version() -> int:
    return _lib.dsa_abi_version()


def last_plan() -> str:
    return _lib.dsa_last_plan().decode()


def last_error() -> str:
    return _lib.dsa_last_error().decode()


def _check(status: int):
    if status != DSA_OK:
        raise DSAError(status, last_error())


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to libdsa must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype in (torch.uint8, torch.float8_e4m3fn):
        return DSA_E4M3
    if t.dtype == torch.float32:
        return DSA_F32
    if t.dtype == torch.bfloat16:
        return DSA_BF16
    raise ValueError(f"unsupported dtype {t.dtype}")


class _CachedDesc:
    """The C descriptor is built on first use and kept until a field is reassigned
    (a step call then costs no Python-side struct building).  Tensors are
    referenced by their data pointers, so resizing a tensor in place needs the
    field reassigned."""

    def __setattr__(self, name, value):
        if name != "_desc":
            object.__setattr__(self, "_desc", None)
        object.__setattr__(self, name, value)

    def desc(self):
        d = self.__dict__.get("_desc")
        if d is None:
            d = self._build_desc()
            object.__setattr__(self, "_desc", d)
        return d


@dataclasses.dataclass
class Seq(_CachedDesc):
    """Queries and paging (device int32 tensors); see dsa_seq_desc_t."""
    q_seq: torch.Tensor
    q_pos: torch.Tensor
    block_table: torch.Tensor          # [B, bt_stride]
    max_ctx: int
    cache_rows: int
    page_size: int = 64
    q_per_seq: int = 0

    def _build_desc(self) -> SeqDesc:
        B, stride = self.block_table.shape
        return SeqDesc(B, self.q_seq.shape[0], self.max_ctx, self.q_per_seq, _ptr(self.q_seq),
                       _ptr(self.q_pos), _ptr(self.block_table), stride, self.page_size, self.cache_rows)


@dataclasses.dataclass
class Indexer(_CachedDesc):
    """Lightning-indexer inputs; see dsa_indexer_desc_t."""
    q: torch.Tensor                    # [T, H_I, D_I] e4m3 codes (uint8) or fp32
    w: torch.Tensor                    # [T, H_I] fp32
    k_cache: torch.Tensor              # [cache_rows, D_I]
    q_scale: Optional[torch.Tensor] = None   # fp32 [T, H_I], or uint8 E8M0 [T, H_I, D_I/32] (MXFP8)
    k_scale: Optional[torch.Tensor] = None   # fp32 [cache_rows], or uint8 E8M0 [cache_rows, D_I/32] (MXFP8)
    dtype: Optional[int] = None              # DSA_MXFP8_E4M3 for MXFP8 codes; else from k_cache

    def _build_desc(self) -> IndexerDesc:
        _, H_I, D_I = self.q.shape
        dt = self.dtype if self.dtype is not None else _dtype_code(self.k_cache)
        return IndexerDesc(H_I, D_I, dt, _ptr(self.q), _ptr(self.q_scale),
                           _ptr(self.w), _ptr(self.k_cache), _ptr(self.k_scale))


@dataclasses.dataclass
class Mla(_CachedDesc):
    """Latent attention inputs; see dsa_mla_desc_t.  kv_cache is [cache_rows, row] of
    bf16/fp32 values or uint8 656-byte FP8 rows (dtype given explicitly then)."""
    q: torch.Tensor                    # [T, H, d_latent + d_rope]
    kv_cache: torch.Tensor
    d_latent: int
    d_rope: int
    softmax_scale: float
    dtype: Optional[int] = None

    def _build_desc(self) -> MlaDesc:
        dt = self.dtype if self.dtype is not None else _dtype_code(self.kv_cache)
        row_bytes = self.kv_cache.stride(0) * self.kv_cache.element_size()
        return MlaDesc(self.q.shape[1], self.d_latent, self.d_rope, dt, _ptr(self.q), _ptr(self.kv_cache),
                       row_bytes, self.softmax_scale)


@dataclasses.dataclass
class Prolog(_CachedDesc):
    """Indexer prolog inputs; see dsa_prolog_desc_t (bf16 tensors, weights as
    [output, input])."""
    x: torch.Tensor                    # [T, d_model] bf16
    x_q: torch.Tensor                  # [T, d_q] bf16
    w_q: torch.Tensor                  # [H_I * D_I, d_q] bf16
    w_k: torch.Tensor                  # [D_I, d_model] bf16
    w_w: torch.Tensor                  # [H_I, d_model] bf16
    gamma: torch.Tensor                # [D_I] fp32
    beta: torch.Tensor                 # [D_I] fp32

    def _build_desc(self) -> PrologDesc:
        return PrologDesc(self.x.shape[1], self.x_q.shape[1], self.w_w.shape[0], self.w_k.shape[0], _ptr(self.x),
                          _ptr(self.x_q), _ptr(self.w_q), _ptr(self.w_k), _ptr(self.w_w), _ptr(self.gamma),
                          _ptr(self.beta))


def indexer_prolog_workspace_size(seq: Seq, pro: Prolog) -> int:
    s, d = seq.desc(), pro.desc()
    return _lib.dsa_indexer_prolog_workspace_size(ctypes.byref(s), ctypes.byref(d))


def indexer_prolog(seq: Seq, pro: Prolog, q_codes: torch.Tensor, q_scale: torch.Tensor, w: torch.Tensor,
                   k_cache: torch.Tensor, k_scale: torch.Tensor, workspace: torch.Tensor, stream=None) -> None:
    """The indexer's query (E4M3 codes + per-head scales), head weights and the new
    tokens' normalised keys (quantised into k_cache / k_scale at their positions)."""
    s, d = seq.desc(), pro.desc()
    _check(_lib.dsa_indexer_prolog(ctypes.byref(s), ctypes.byref(d), _ptr(q_codes), _ptr(q_scale), _ptr(w),
                                   _ptr(k_cache), _ptr(k_scale), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _stream(stream)))


def indexer_scores(seq: Seq, idx: Indexer, scores: torch.Tensor, stream=None) -> torch.Tensor:
    s, x = seq.desc(), idx.desc()
    _check(_lib.dsa_indexer_scores(ctypes.byref(s), ctypes.byref(x), _ptr(scores), scores.stride(0),
                                   _stream(stream)))
    return scores


def topk(seq: Seq, scores: torch.Tensor, K: int, out: torch.Tensor, stream=None) -> torch.Tensor:
    s = seq.desc()
    _check(_lib.dsa_topk(ctypes.byref(s), _ptr(scores), scores.stride(0), K, _ptr(out), _stream(stream)))
    return out


def sparse_mla_attn_workspace_size(seq: Seq, mla: Mla, K: int) -> int:
    s, m = seq.desc(), mla.desc()
    return _lib.dsa_sparse_mla_attn_workspace_size(ctypes.byref(s), ctypes.byref(m), K)


def sparse_mla_attn(seq: Seq, mla: Mla, idx: torch.Tensor, K: int, out: torch.Tensor,
                    lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                    stream=None) -> torch.Tensor:
    s, m = seq.desc(), mla.desc()
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(_lib.dsa_sparse_mla_attn(ctypes.byref(s), ctypes.byref(m), _ptr(idx), K, _ptr(out), _ptr(lse),
                                    _ptr(workspace), ws_bytes, _stream(stream)))
    return out


def decode_workspace_size(seq: Seq, idx: Indexer, mla: Mla, K: int) -> int:
    s, x, m = seq.desc(), idx.desc(), mla.desc()
    return _lib.dsa_decode_workspace_size(ctypes.byref(s), ctypes.byref(x), ctypes.byref(m), K)


def decode_step(seq: Seq, idx: Indexer, mla: Mla, K: int, out: torch.Tensor, workspace: torch.Tensor,
                lse: Optional[torch.Tensor] = None, idx_out: Optional[torch.Tensor] = None,
                stream=None) -> torch.Tensor:
    s, x, m = seq.desc(), idx.desc(), mla.desc()
    _check(_lib.dsa_decode_step(ctypes.byref(s), ctypes.byref(x), ctypes.byref(m), K, _ptr(out), _ptr(lse),
                                _ptr(idx_out), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                _stream(stream)))
    return out


def decode_step_static_ws(seq: Seq, idx: Indexer, mla: Mla, K: int, out: torch.Tensor,
                          lse: Optional[torch.Tensor] = None, idx_out: Optional[torch.Tensor] = None,
                          stream=None) -> torch.Tensor:
    """decode_step with the scratch in the library's own device array (no workspace
    argument, nothing allocated) -- for callers that cannot allocate device memory.
    Calls overlapping on the GPU race on that shared array."""
    s, x, m = seq.desc(), idx.desc(), mla.desc()
    _check(_lib.dsa_decode_step_static_ws(ctypes.byref(s), ctypes.byref(x), ctypes.byref(m), K, _ptr(out),
                                          _ptr(lse), _ptr(idx_out), _stream(stream)))
    return out


def index_cache_append(seq: Seq, k_new: torch.Tensor, k_cache: torch.Tensor, k_scale: torch.Tensor,
                       stream=None, mx: bool = False) -> None:
    """Quantises the new tokens' index keys k_new [T, D_I] (fp32 or bf16) to e4m3
    + per-token fp32 scale (k_scale [cache_rows]), or with mx to MXFP8 (k_scale
    uint8 [cache_rows, D_I / 32] E8M0 bytes), and writes them at their
    positions' cache rows."""
    s = seq.desc()
    fn = _lib.dsa_index_cache_append_mx if mx else _lib.dsa_index_cache_append
    _check(fn(ctypes.byref(s), k_new.shape[1], _dtype_code(k_new), _ptr(k_new), _ptr(k_cache), _ptr(k_scale),
              _stream(stream)))


def latent_cache_append(seq: Seq, mla: Mla, kv_new: torch.Tensor, stream=None) -> None:
    """Writes the new tokens' latent rows kv_new [T, d_latent + d_rope] into
    mla.kv_cache (copied, or quantised into 656-byte FP8 rows)."""
    s, m = seq.desc(), mla.desc()
    _check(_lib.dsa_latent_cache_append(ctypes.byref(s), ctypes.byref(m), _ptr(kv_new), _ptr(mla.kv_cache),
                                        _stream(stream)))


def debug_withhold_arrival(enable: bool, wait_limit_ns: int = 2_000_000) -> None:
    """Testing aid of the failure-detection path: while enabled, tensor-core
    attention launches have one producer warp withhold an arrival so a bounded
    wait runs out (after wait_limit_ns) and check_status() raises DSA_ERR_TIMEOUT."""
    _check(_lib.dsa_debug_withhold_arrival(1 if enable else 0, int(wait_limit_ns)))


def check_status(stream=None) -> None:
    """Synchronises the stream and raises DSAError if a device-side check fired."""
    _check(_lib.dsa_check_status(_stream(stream)))
