"""ctypes binding of libgqadecode.so -- argument marshalling only.

Every function here has the name of the C entry point it calls (include/gqa_decode.h)
and does nothing but check tensor metadata, pick the current CUDA stream and pass
raw device pointers.  All of the attention arithmetic runs in the library's CUDA
kernels; there is no fallback: if the library cannot be built or loaded, the
first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

GQA_OK = 0
GQA_ERR_INVALID_ARGUMENT = 1
GQA_ERR_UNSUPPORTED = 2
GQA_ERR_WORKSPACE = 3
GQA_ERR_CUDA = 4

GQA_OUT_BF16 = 0
GQA_OUT_F32 = 1

GQA_DEVICE_WAIT_TIMEOUT = 1
GQA_DEVICE_BAD_PAGE = 2
GQA_DEVICE_BAD_LENGTH = 4

GQA_KERNEL_NONE = 0
GQA_KERNEL_SPLIT_DECODE = 1
GQA_KERNEL_TCGEN05 = 2

GQA_TEST_SINGLE_PIECE = 1
GQA_TEST_STALL = 2

PAGE_SIZE = 16
GQA_MAX_SEQ = 262144   # longest cache (positions) a call accepts

EXPORTED_SYMBOLS = ("gqa_workspace_size", "gqa_workspace_init", "gqa_decode", "gqa_decode_paged",
                    "gqa_device_status", "gqa_decode_noalloc", "gqa_decode_ring",
                    "gqa_decode_keqv", "gqa_decode_keqv_paged", "gqa_prepare_decode",
                    "gqa_prepare_decode_paged", "gqa_workspace_size_mq", "gqa_decode_mq",
                    "gqa_decode_mq_paged",
                    "gqa_check_inputs_host", "gqa_noalloc_status", "gqa_decode_keqv_kernel",
                    "gqa_set_test_mode", "gqa_get_test_mode",
                    "gqa_status_string")

_lock = threading.Lock()
_lib = None


class GQAError(RuntimeError):
    """A gqa_* call returned a status other than GQA_OK."""

    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {gqa_status_string(status)} ({status})")


def library_path() -> str:
    return _build.LIB_PATH


def load_library(build_if_needed: bool = True) -> ctypes.CDLL:
    """Load libgqadecode.so (building it first when missing or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if build_if_needed and not _build.up_to_date():
            _build.build()
        if not os.path.exists(_build.LIB_PATH):
            raise RuntimeError(f"CUDA library not built: {_build.LIB_PATH}")
        lib = ctypes.CDLL(_build.LIB_PATH)
        vp, sz, ci = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
        lib.gqa_workspace_size.argtypes = [ci, ci, ci, ci, ci, ci]
        lib.gqa_workspace_size.restype = sz
        lib.gqa_workspace_init.argtypes = [vp, sz, vp]
        lib.gqa_workspace_init.restype = ci
        lib.gqa_decode.argtypes = [vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, vp, ci, vp, sz, vp]
        lib.gqa_decode.restype = ci
        lib.gqa_decode_paged.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, ci, vp,
                                         ci, vp, sz, vp]
        lib.gqa_decode_paged.restype = ci
        lib.gqa_decode_noalloc.argtypes = [vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, vp, ci, vp]
        lib.gqa_decode_noalloc.restype = ci
        lib.gqa_decode_ring.argtypes = [vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, vp, ci, vp, sz, vp]
        lib.gqa_decode_ring.restype = ci
        lib.gqa_decode_keqv.argtypes = [vp, vp, vp, vp, ci, ci, ci, ci, ci, vp, ci, vp, sz, vp]
        lib.gqa_decode_keqv.restype = ci
        lib.gqa_decode_keqv_paged.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, vp,
                                              ci, vp, sz, vp]
        lib.gqa_decode_keqv_paged.restype = ci
        lib.gqa_prepare_decode.argtypes = [vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, vp, vp, vp, ci,
                                           ci, vp]
        lib.gqa_prepare_decode.restype = ci
        lib.gqa_prepare_decode_paged.argtypes = [vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci,
                                                 ci, vp, vp, vp, vp]
        lib.gqa_prepare_decode_paged.restype = ci
        lib.gqa_workspace_size_mq.argtypes = [ci, ci, ci, ci, ci]
        lib.gqa_workspace_size_mq.restype = sz
        lib.gqa_decode_mq.argtypes = [vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, vp, ci, vp, sz, vp]
        lib.gqa_decode_mq.restype = ci
        lib.gqa_decode_mq_paged.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, ci, ci,
                                            vp, ci, vp, sz, vp]
        lib.gqa_decode_mq_paged.restype = ci
        lib.gqa_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), vp]
        lib.gqa_device_status.restype = ci
        lib.gqa_check_inputs_host.argtypes = [vp, ci, ci, ci, vp, ci, ci, ctypes.POINTER(ci)]
        lib.gqa_check_inputs_host.restype = ci
        lib.gqa_noalloc_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), vp]
        lib.gqa_noalloc_status.restype = ci
        lib.gqa_decode_keqv_kernel.argtypes = [ci, ci, ci, ci, ci]
        lib.gqa_decode_keqv_kernel.restype = ci
        lib.gqa_set_test_mode.argtypes = [ctypes.c_uint32]
        lib.gqa_set_test_mode.restype = ctypes.c_uint32
        lib.gqa_get_test_mode.argtypes = []
        lib.gqa_get_test_mode.restype = ctypes.c_uint32
        lib.gqa_status_string.argtypes = [ci]
        lib.gqa_status_string.restype = ctypes.c_char_p
        _lib = lib
        return lib


def gqa_status_string(status: int) -> str:
    return load_library().gqa_status_string(int(status)).decode()


def gqa_workspace_size(B: int, max_seq: int, H: int, KVH: int, D: int, window: int) -> int:
    return int(load_library().gqa_workspace_size(B, max_seq, H, KVH, D, window))


def _stream_handle(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _check(fn: str, status: int):
    if status != GQA_OK:
        raise GQAError(fn, status)


class _OnDevice:
    """The library's entry points, each called with ``device`` current: the library
    takes its SM count, scratch and launch device from the current device."""

    def __init__(self, device):
        self._lib = load_library()
        self._device = device

    def __getattr__(self, name):
        fn = getattr(self._lib, name)

        def call(*args):
            with torch.cuda.device(self._device):
                return fn(*args)
        return call


def _lib_on(device) -> _OnDevice:
    return _OnDevice(device)


def _same_device(ref: torch.Tensor, **tensors):
    """Every tensor argument must sit on the device of ``ref`` (q)."""
    for name, t in tensors.items():
        if t is not None:
            _require(t.device == ref.device, f"{name} must be on {ref.device} (q's device)")


def gqa_workspace_init(workspace: torch.Tensor, stream=None) -> None:
    """Zero a caller-owned workspace before its first use."""
    st = load_library().gqa_workspace_init(_ptr(workspace), workspace.numel() * workspace.element_size(),
                                           _stream_handle(stream, workspace.device))
    _check("gqa_workspace_init", st)


def new_workspace(B: int, max_seq: int, H: int, KVH: int, D: int, window: int,
                  device=None, stream=None) -> torch.Tensor:
    """Allocate (torch caching allocator) and zero a workspace for this call shape."""
    n = gqa_workspace_size(B, max_seq, H, KVH, D, window)
    if n == 0:
        raise GQAError("gqa_workspace_size", GQA_ERR_INVALID_ARGUMENT)
    ws = torch.empty(n, dtype=torch.uint8, device=device or "cuda")
    gqa_workspace_init(ws, stream)
    return ws


def _out_code(out: torch.Tensor) -> int:
    if out.dtype == torch.float32:
        return GQA_OUT_F32
    if out.dtype == torch.bfloat16:
        return GQA_OUT_BF16
    raise TypeError("out must be bf16 or fp32")


def _require(cond: bool, msg: str):
    if not cond:
        raise ValueError(msg)


def _check_tensor(name, t, dtype, ndim):
    _require(isinstance(t, torch.Tensor), f"{name} must be a torch.Tensor")
    _require(t.is_cuda, f"{name} must be on a CUDA device")
    _require(t.dtype == dtype, f"{name} must be {dtype}")
    _require(t.dim() == ndim, f"{name} must have {ndim} dims")
    _require(t.is_contiguous(), f"{name} must be contiguous")


def gqa_decode(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, seq_lens: torch.Tensor,
               window: int, out: torch.Tensor | None = None, out_dtype=torch.bfloat16,
               workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """attn.core over a contiguous cache: q [B,H,D], k/v [B,S,KVH,D] (bf16), seq_lens int32 [B]."""
    _check_tensor("q", q, torch.bfloat16, 3)
    _check_tensor("k", k, torch.bfloat16, 4)
    _check_tensor("v", v, torch.bfloat16, 4)
    _check_tensor("seq_lens", seq_lens, torch.int32, 1)
    B, H, D = q.shape
    _, S, KVH, _ = k.shape
    _require(tuple(k.shape) == (B, S, KVH, D) and v.shape == k.shape, "k/v shape mismatch")
    _require(seq_lens.shape[0] == B, "seq_lens must have B entries")
    if out is None:
        out = torch.empty((B, H, D), dtype=out_dtype, device=q.device)
    _check_tensor("out", out, out.dtype, 3)
    _require(tuple(out.shape) == (B, H, D), "out must be [B, H, D]")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _same_device(q, k=k, v=v, seq_lens=seq_lens, out=out, workspace=workspace)
    st = _lib_on(q.device).gqa_decode(
        _ptr(q), _ptr(k), _ptr(v), _ptr(seq_lens), B, S, H, KVH, D, int(window), _ptr(out),
        _out_code(out), _ptr(workspace), ws_bytes, _stream_handle(stream, q.device))
    _check("gqa_decode", st)
    return out


def gqa_decode_paged(q: torch.Tensor, k_pages: torch.Tensor, v_pages: torch.Tensor,
                     block_table: torch.Tensor, seq_lens: torch.Tensor, window: int,
                     out: torch.Tensor | None = None, out_dtype=torch.bfloat16,
                     workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """attn.core over a paged cache: pools [P,16,KVH,D], block_table int32 [B,max_pages]."""
    _check_tensor("q", q, torch.bfloat16, 3)
    _check_tensor("k_pages", k_pages, torch.bfloat16, 4)
    _check_tensor("v_pages", v_pages, torch.bfloat16, 4)
    _check_tensor("block_table", block_table, torch.int32, 2)
    _check_tensor("seq_lens", seq_lens, torch.int32, 1)
    B, H, D = q.shape
    P, page_size, KVH, _ = k_pages.shape
    _require(v_pages.shape == k_pages.shape and k_pages.shape[3] == D, "page pool shape mismatch")
    _require(block_table.shape[0] == B and seq_lens.shape[0] == B, "batch size mismatch")
    if out is None:
        out = torch.empty((B, H, D), dtype=out_dtype, device=q.device)
    _check_tensor("out", out, out.dtype, 3)
    _require(tuple(out.shape) == (B, H, D), "out must be [B, H, D]")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _same_device(q, k_pages=k_pages, v_pages=v_pages, block_table=block_table,
                 seq_lens=seq_lens, out=out, workspace=workspace)
    st = _lib_on(q.device).gqa_decode_paged(
        _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table), _ptr(seq_lens), B, P,
        block_table.shape[1], page_size, H, KVH, D, int(window), _ptr(out), _out_code(out),
        _ptr(workspace), ws_bytes, _stream_handle(stream, q.device))
    _check("gqa_decode_paged", st)
    return out


def gqa_decode_ring(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, seq_lens: torch.Tensor,
                    window: int, out: torch.Tensor | None = None, out_dtype=torch.bfloat16,
                    workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """attn.core over a window-capped ring cache: k/v [B,C,KVH,D] (bf16) hold position s
    at row s % C; attends [max(0, L - window), L) with 1 <= window <= C."""
    _check_tensor("q", q, torch.bfloat16, 3)
    _check_tensor("k", k, torch.bfloat16, 4)
    _check_tensor("v", v, torch.bfloat16, 4)
    _check_tensor("seq_lens", seq_lens, torch.int32, 1)
    B, H, D = q.shape
    _, C, KVH, _ = k.shape
    _require(tuple(k.shape) == (B, C, KVH, D) and v.shape == k.shape, "k/v shape mismatch")
    _require(seq_lens.shape[0] == B, "seq_lens must have B entries")
    if out is None:
        out = torch.empty((B, H, D), dtype=out_dtype, device=q.device)
    _check_tensor("out", out, out.dtype, 3)
    _require(tuple(out.shape) == (B, H, D), "out must be [B, H, D]")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _same_device(q, k=k, v=v, seq_lens=seq_lens, out=out, workspace=workspace)
    st = _lib_on(q.device).gqa_decode_ring(
        _ptr(q), _ptr(k), _ptr(v), _ptr(seq_lens), B, C, H, KVH, D, int(window), _ptr(out),
        _out_code(out), _ptr(workspace), ws_bytes, _stream_handle(stream, q.device))
    _check("gqa_decode_ring", st)
    return out


def gqa_decode_keqv(q: torch.Tensor, v: torch.Tensor, w_k: torch.Tensor, seq_lens: torch.Tensor,
                    out: torch.Tensor | None = None, out_dtype=torch.bfloat16,
                    workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """decodeGQA over a single K=V cache: v [B,S,4,512] (bf16), w_k [512] (bf16) the
    k_norm weight; each key is rope(w_k * v, position), derived in the kernel."""
    _check_tensor("q", q, torch.bfloat16, 3)
    _check_tensor("v", v, torch.bfloat16, 4)
    _check_tensor("w_k", w_k, torch.bfloat16, 1)
    _check_tensor("seq_lens", seq_lens, torch.int32, 1)
    B, H, D = q.shape
    _, S, KVH, _ = v.shape
    _require(tuple(v.shape) == (B, S, KVH, D) and w_k.shape[0] == D, "v / w_k shape mismatch")
    _require(seq_lens.shape[0] == B, "seq_lens must have B entries")
    if out is None:
        out = torch.empty((B, H, D), dtype=out_dtype, device=q.device)
    _check_tensor("out", out, out.dtype, 3)
    _require(tuple(out.shape) == (B, H, D), "out must be [B, H, D]")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _same_device(q, v=v, w_k=w_k, seq_lens=seq_lens, out=out, workspace=workspace)
    st = _lib_on(q.device).gqa_decode_keqv(
        _ptr(q), _ptr(v), _ptr(w_k), _ptr(seq_lens), B, S, H, KVH, D, _ptr(out), _out_code(out),
        _ptr(workspace), ws_bytes, _stream_handle(stream, q.device))
    _check("gqa_decode_keqv", st)
    return out


def gqa_decode_keqv_paged(q: torch.Tensor, v_pages: torch.Tensor, w_k: torch.Tensor,
                          block_table: torch.Tensor, seq_lens: torch.Tensor,
                          out: torch.Tensor | None = None, out_dtype=torch.bfloat16,
                          workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """gqa_decode_keqv over a paged value cache: pool [P,16,4,512], block_table [B,max_pages]."""
    _check_tensor("q", q, torch.bfloat16, 3)
    _check_tensor("v_pages", v_pages, torch.bfloat16, 4)
    _check_tensor("w_k", w_k, torch.bfloat16, 1)
    _check_tensor("block_table", block_table, torch.int32, 2)
    _check_tensor("seq_lens", seq_lens, torch.int32, 1)
    B, H, D = q.shape
    P, page_size, KVH, _ = v_pages.shape
    _require(v_pages.shape[3] == D and w_k.shape[0] == D, "page pool / w_k shape mismatch")
    _require(block_table.shape[0] == B and seq_lens.shape[0] == B, "batch size mismatch")
    if out is None:
        out = torch.empty((B, H, D), dtype=out_dtype, device=q.device)
    _check_tensor("out", out, out.dtype, 3)
    _require(tuple(out.shape) == (B, H, D), "out must be [B, H, D]")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _same_device(q, v_pages=v_pages, w_k=w_k, block_table=block_table, seq_lens=seq_lens,
                 out=out, workspace=workspace)
    st = _lib_on(q.device).gqa_decode_keqv_paged(
        _ptr(q), _ptr(v_pages), _ptr(w_k), _ptr(block_table), _ptr(seq_lens), B, P,
        block_table.shape[1], page_size, H, KVH, D, _ptr(out), _out_code(out), _ptr(workspace),
        ws_bytes, _stream_handle(stream, q.device))
    _check("gqa_decode_keqv_paged", st)
    return out


GQA_MAX_QUERIES_SLIDING = 8
GQA_MAX_QUERIES_GLOBAL = 4


def gqa_workspace_size_mq(B: int, T: int, H: int, KVH: int, D: int) -> int:
    return int(load_library().gqa_workspace_size_mq(B, T, H, KVH, D))


def _mq_out(q, out, out_dtype):
    B, T, H, D = q.shape
    if out is None:
        out = torch.empty((B, T, H, D), dtype=out_dtype, device=q.device)
    _check_tensor("out", out, out.dtype, 4)
    _require(tuple(out.shape) == (B, T, H, D), "out must be [B, T, H, D]")
    return out


def gqa_decode_mq(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, seq_lens: torch.Tensor,
                  window: int, out: torch.Tensor | None = None, out_dtype=torch.bfloat16,
                  workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Multi-query decode over a contiguous cache: q [B,T,H,D], k/v [B,S,KVH,D] (bf16);
    query t sits at position seq_lens[b] - T + t.  Returns out [B,T,H,D]."""
    _check_tensor("q", q, torch.bfloat16, 4)
    _check_tensor("k", k, torch.bfloat16, 4)
    _check_tensor("v", v, torch.bfloat16, 4)
    _check_tensor("seq_lens", seq_lens, torch.int32, 1)
    B, T, H, D = q.shape
    _, S, KVH, _ = k.shape
    _require(tuple(k.shape) == (B, S, KVH, D) and v.shape == k.shape, "k/v shape mismatch")
    _require(seq_lens.shape[0] == B, "seq_lens must have B entries")
    out = _mq_out(q, out, out_dtype)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _same_device(q, k=k, v=v, seq_lens=seq_lens, out=out, workspace=workspace)
    st = _lib_on(q.device).gqa_decode_mq(
        _ptr(q), _ptr(k), _ptr(v), _ptr(seq_lens), B, T, S, H, KVH, D, int(window), _ptr(out),
        _out_code(out), _ptr(workspace), ws_bytes, _stream_handle(stream, q.device))
    _check("gqa_decode_mq", st)
    return out


def gqa_decode_mq_paged(q: torch.Tensor, k_pages: torch.Tensor, v_pages: torch.Tensor,
                        block_table: torch.Tensor, seq_lens: torch.Tensor, window: int,
                        out: torch.Tensor | None = None, out_dtype=torch.bfloat16,
                        workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Multi-query decode over a paged cache: pools [P,16,KVH,D], block_table [B,max_pages]."""
    _check_tensor("q", q, torch.bfloat16, 4)
    _check_tensor("k_pages", k_pages, torch.bfloat16, 4)
    _check_tensor("v_pages", v_pages, torch.bfloat16, 4)
    _check_tensor("block_table", block_table, torch.int32, 2)
    _check_tensor("seq_lens", seq_lens, torch.int32, 1)
    B, T, H, D = q.shape
    P, page_size, KVH, _ = k_pages.shape
    _require(v_pages.shape == k_pages.shape and k_pages.shape[3] == D, "page pool shape mismatch")
    _require(block_table.shape[0] == B and seq_lens.shape[0] == B, "batch size mismatch")
    out = _mq_out(q, out, out_dtype)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _same_device(q, k_pages=k_pages, v_pages=v_pages, block_table=block_table,
                 seq_lens=seq_lens, out=out, workspace=workspace)
    st = _lib_on(q.device).gqa_decode_mq_paged(
        _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table), _ptr(seq_lens), B, T, P,
        block_table.shape[1], page_size, H, KVH, D, int(window), _ptr(out), _out_code(out),
        _ptr(workspace), ws_bytes, _stream_handle(stream, q.device))
    _check("gqa_decode_mq_paged", st)
    return out


def gqa_prepare_decode(q_raw: torch.Tensor, k_raw: torch.Tensor, v_raw, w_q: torch.Tensor,
                       w_k: torch.Tensor, seq_lens: torch.Tensor, q_out: torch.Tensor,
                       k_cache, v_cache: torch.Tensor, ring: bool = False, stream=None):
    """Decode-step producer: q_out = rope(q_norm(q_raw)); appends rope(k_norm(k_raw)) and
    v_norm(v_raw) (v_norm(k_raw) when v_raw is None, values = keys; k_cache unused) at
    position seq_lens[b] - 1 of a contiguous cache [B, rows, KVH, D] (row (L-1) % rows
    when ring)."""
    _check_tensor("q_raw", q_raw, torch.bfloat16, 3)
    _check_tensor("k_raw", k_raw, torch.bfloat16, 3)
    if v_raw is not None:
        _check_tensor("v_raw", v_raw, torch.bfloat16, 3)
    _check_tensor("w_q", w_q, torch.bfloat16, 1)
    _check_tensor("w_k", w_k, torch.bfloat16, 1)
    _check_tensor("seq_lens", seq_lens, torch.int32, 1)
    _check_tensor("q_out", q_out, torch.bfloat16, 3)
    _check_tensor("v_cache", v_cache, torch.bfloat16, 4)
    if k_cache is not None:
        _check_tensor("k_cache", k_cache, torch.bfloat16, 4)
    B, H, D = q_raw.shape
    KVH = k_raw.shape[1]
    _require(tuple(v_cache.shape[2:]) == (KVH, D) and v_cache.shape[0] == B, "cache shape mismatch")
    _require(q_out.shape == q_raw.shape, "q_out must match q_raw")
    _same_device(q_raw, k_raw=k_raw, v_raw=v_raw, w_q=w_q, w_k=w_k, seq_lens=seq_lens,
                 q_out=q_out, k_cache=k_cache, v_cache=v_cache)
    st = _lib_on(q_raw.device).gqa_prepare_decode(
        _ptr(q_raw), _ptr(k_raw), _ptr(v_raw), _ptr(w_q), _ptr(w_k), _ptr(seq_lens), B, H, KVH, D,
        _ptr(q_out), _ptr(k_cache), _ptr(v_cache), v_cache.shape[1], 1 if ring else 0,
        _stream_handle(stream, q_raw.device))
    _check("gqa_prepare_decode", st)


def gqa_prepare_decode_paged(q_raw: torch.Tensor, k_raw: torch.Tensor, v_raw, w_q: torch.Tensor,
                             w_k: torch.Tensor, block_table: torch.Tensor, seq_lens: torch.Tensor,
                             q_out: torch.Tensor, k_pages, v_pages: torch.Tensor, stream=None):
    """gqa_prepare_decode into page pools [P, 16, KVH, D] through a block table."""
    _check_tensor("q_raw", q_raw, torch.bfloat16, 3)
    _check_tensor("k_raw", k_raw, torch.bfloat16, 3)
    if v_raw is not None:
        _check_tensor("v_raw", v_raw, torch.bfloat16, 3)
    _check_tensor("w_q", w_q, torch.bfloat16, 1)
    _check_tensor("w_k", w_k, torch.bfloat16, 1)
    _check_tensor("block_table", block_table, torch.int32, 2)
    _check_tensor("seq_lens", seq_lens, torch.int32, 1)
    _check_tensor("q_out", q_out, torch.bfloat16, 3)
    _check_tensor("v_pages", v_pages, torch.bfloat16, 4)
    if k_pages is not None:
        _check_tensor("k_pages", k_pages, torch.bfloat16, 4)
    B, H, D = q_raw.shape
    KVH = k_raw.shape[1]
    P, page_size = v_pages.shape[0], v_pages.shape[1]
    _same_device(q_raw, k_raw=k_raw, v_raw=v_raw, w_q=w_q, w_k=w_k, block_table=block_table,
                 seq_lens=seq_lens, q_out=q_out, k_pages=k_pages, v_pages=v_pages)
    st = _lib_on(q_raw.device).gqa_prepare_decode_paged(
        _ptr(q_raw), _ptr(k_raw), _ptr(v_raw), _ptr(w_q), _ptr(w_k), _ptr(block_table),
        _ptr(seq_lens), B, P, block_table.shape[1], page_size, H, KVH, D, _ptr(q_out),
        _ptr(k_pages), _ptr(v_pages), _stream_handle(stream, q_raw.device))
    _check("gqa_prepare_decode_paged", st)


def gqa_decode_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, seq_lens: torch.Tensor,
                       window: int, out: torch.Tensor, stream=None) -> torch.Tensor:
    """gqa_decode for callers that cannot allocate: the library's fixed device scratch
    replaces the workspace.  ``out`` must be supplied (bf16 or fp32 [B, H, D]), so the
    call allocates nothing on the device."""
    _check_tensor("q", q, torch.bfloat16, 3)
    _check_tensor("k", k, torch.bfloat16, 4)
    _check_tensor("v", v, torch.bfloat16, 4)
    _check_tensor("seq_lens", seq_lens, torch.int32, 1)
    B, H, D = q.shape
    _, S, KVH, _ = k.shape
    _require(tuple(k.shape) == (B, S, KVH, D) and v.shape == k.shape, "k/v shape mismatch")
    _require(seq_lens.shape[0] == B, "seq_lens must have B entries")
    _check_tensor("out", out, out.dtype, 3)
    _require(tuple(out.shape) == (B, H, D), "out must be [B, H, D]")
    _same_device(q, k=k, v=v, seq_lens=seq_lens, out=out)
    st = _lib_on(q.device).gqa_decode_noalloc(
        _ptr(q), _ptr(k), _ptr(v), _ptr(seq_lens), B, S, H, KVH, D, int(window), _ptr(out),
        _out_code(out), _stream_handle(stream, q.device))
    _check("gqa_decode_noalloc", st)
    return out


def gqa_check_inputs_host(seq_lens, capacity: int, window: int, block_table=None,
                          num_pages: int = 0) -> int:
    """Check host copies of seq_lens (and the block table): returns -1 when every
    sequence is valid, else the index of the first bad one (length outside
    [0, capacity], or an attended page outside [0, num_pages))."""
    import numpy as np
    lens = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32))
    bt = None if block_table is None else np.ascontiguousarray(np.asarray(block_table, dtype=np.int32))
    max_pages = 0 if bt is None else int(bt.shape[1])
    first = ctypes.c_int(-1)
    st = load_library().gqa_check_inputs_host(
        lens.ctypes.data if lens.size else None, int(lens.shape[0]), int(capacity), int(window),
        None if bt is None else bt.ctypes.data, max_pages, int(num_pages), ctypes.byref(first))
    if st not in (GQA_OK, GQA_ERR_INVALID_ARGUMENT) or (st != GQA_OK and first.value < 0):
        raise GQAError("gqa_check_inputs_host", st)
    return first.value


def gqa_device_status(workspace: torch.Tensor | None = None, stream=None) -> int:
    """Read and clear the device status word (GQA_DEVICE_* bits); synchronises the stream."""
    flags = ctypes.c_uint32(0)
    dev = workspace.device if workspace is not None else torch.device("cuda", torch.cuda.current_device())
    st = load_library().gqa_device_status(_ptr(workspace), ctypes.byref(flags),
                                          _stream_handle(stream, dev))
    _check("gqa_device_status", st)
    return int(flags.value)


def gqa_noalloc_status(stream=None, device=None) -> int:
    """Read and clear the status word of gqa_decode_noalloc's fixed array on ``device``
    (default: the current device); synchronises the stream.  Allocates nothing."""
    flags = ctypes.c_uint32(0)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    st = _lib_on(dev).gqa_noalloc_status(ctypes.byref(flags), _stream_handle(stream, dev))
    _check("gqa_noalloc_status", st)
    return int(flags.value)


def gqa_decode_keqv_kernel(B: int, capacity: int, H: int = 32, KVH: int = 4, D: int = 512,
                           device=None) -> int:
    """GQA_KERNEL_* code of the kernel a K=V call with these sizes runs on ``device``
    (capacity: S, or 16 * max_pages for a paged cache)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    return int(_lib_on(dev).gqa_decode_keqv_kernel(B, capacity, H, KVH, D))


def gqa_set_test_mode(flags: int) -> int:
    """Set the process-wide test mode (GQA_TEST_* bits, 0 = normal); returns the previous one."""
    return int(load_library().gqa_set_test_mode(int(flags)))


def gqa_get_test_mode() -> int:
    return int(load_library().gqa_get_test_mode())
