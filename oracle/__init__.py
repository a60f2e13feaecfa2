"""fp64 CPU oracle for the decode-step attention core (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The CUDA library never calls it and shares no code
with it.  The arithmetic lives in ``gqa_oracle.c`` (plain C, OpenMP over the
(b, h) pairs); this module compiles it with gcc and marshals numpy arrays.

What it computes (gemma-4-31B Model Spec, "Compute-graph nodes" table, the two
``attn.core`` rows; masks from the "Gemma 4 31B-it Text Architecture" page,
"Compact form"): for every sequence b and query head h, with g = H / KVH and
kvh = h // g, the softmax (scale 1) of the dot products of q[b, h] with the keys
k[b, s, kvh] over the attended positions s, used as weights on v[b, s, kvh].
The attended positions are [0, L_b) for full layers (window 0) and
[max(0, L_b - window), L_b) for sliding layers.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gqa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libgqa_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``gqa_oracle.c`` into ``libgqa_oracle.so`` (gcc, OpenMP)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-Wall",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(path: str):
    lib = ctypes.CDLL(path)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    i32p = ctypes.POINTER(ctypes.c_int32)
    f64p = ctypes.POINTER(ctypes.c_double)
    ci = ctypes.c_int
    lib.oracle_gqa_decode_f64.argtypes = [u16p, u16p, u16p, i32p, ci, ci, ci, ci, ci, ci,
                                          ctypes.c_int64, ci, f64p]
    lib.oracle_gqa_decode_f64.restype = ci
    lib.oracle_gqa_decode_paged_f64.argtypes = [u16p, u16p, u16p, i32p, i32p, ci, ci, ci,
                                                ci, ci, ci, ci, ci, ci, f64p]
    lib.oracle_gqa_decode_paged_f64.restype = ci
    lib.oracle_gqa_decode_ring_f64.argtypes = [u16p, u16p, u16p, i32p, ci, ci, ci, ci, ci, ci,
                                               ci, f64p]
    lib.oracle_gqa_decode_ring_f64.restype = ci
    lib.oracle_gqa_decode_keqv_f64.argtypes = [u16p, u16p, u16p, i32p, ci, ci, ci, ci, ci, ci,
                                               ci, ctypes.c_double, ci, f64p]
    lib.oracle_gqa_decode_keqv_f64.restype = ci
    lib.oracle_prepare_decode_f64.argtypes = [u16p, u16p, u16p, u16p, u16p, i32p, ci, ci, ci, ci,
                                              ci, ctypes.c_double, f64p, f64p, f64p]
    lib.oracle_prepare_decode_f64.restype = ci
    lib.oracle_gqa_decode_mq_f64.argtypes = [u16p, u16p, u16p, i32p, ci, ci, ci, ci, ci, ci,
                                             ci, ci, f64p]
    lib.oracle_gqa_decode_mq_f64.restype = ci
    lib.oracle_gqa_decode_mq_paged_f64.argtypes = [u16p, u16p, u16p, i32p, i32p, ci, ci, ci,
                                                   ci, ci, ci, ci, ci, ci, ci, f64p]
    lib.oracle_gqa_decode_mq_paged_f64.restype = ci
    lib.oracle_default_threads.argtypes = []
    lib.oracle_default_threads.restype = ci
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = _bind(build())
    return _lib


def _u16(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"expected bf16 bit patterns as uint16, got {a.dtype}")
    return a


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def default_threads() -> int:
    """OpenMP threads the oracle uses when ``nthreads`` is 0."""
    return int(_load().oracle_default_threads())


def gqa_decode_f64(q: np.ndarray, k: np.ndarray, v: np.ndarray, seq_lens, window: int,
                   pos_base: int = 0, nthreads: int = 0, _lib_override=None) -> np.ndarray:
    """Decode attention over a contiguous cache, exact up to fp64 rounding.

    q: uint16 [B, H, D] (bf16 bits); k, v: uint16 [B, S, KVH, D] whose row s is
    position ``pos_base + s``; seq_lens: int [B] absolute lengths; window: 0 for
    full history, else the number of most recent positions attended.
    Returns float64 [B, H, D].
    """
    q, k, v = _u16(q), _u16(k), _u16(v)
    B, H, D = q.shape
    Bk, S, KVH, Dk = k.shape
    if k.shape != v.shape or Bk != B or Dk != D:
        raise ValueError("shape mismatch between q, k and v")
    lens = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32))
    if lens.shape != (B,):
        raise ValueError("seq_lens must have shape [B]")
    out = np.zeros((B, H, D), dtype=np.float64)
    lib = _lib_override if _lib_override is not None else _load()
    rc = lib.oracle_gqa_decode_f64(
        _ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16), _ptr(v, ctypes.c_uint16),
        _ptr(lens, ctypes.c_int32), B, S, H, KVH, D, int(window), int(pos_base), int(nthreads),
        _ptr(out, ctypes.c_double))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")
    return out


def gqa_decode_paged_f64(q: np.ndarray, k_pages: np.ndarray, v_pages: np.ndarray,
                         block_table: np.ndarray, seq_lens, window: int,
                         nthreads: int = 0, _lib_override=None) -> np.ndarray:
    """Decode attention over a paged cache, exact up to fp64 rounding.

    k_pages, v_pages: uint16 [P, page_size, KVH, D]; block_table: int32
    [B, max_pages]; position s of sequence b is slot s % page_size of page
    block_table[b, s // page_size].  A sequence whose attended range names a page
    outside [0, P) gets NaN for all of its heads.
    """
    q, k_pages, v_pages = _u16(q), _u16(k_pages), _u16(v_pages)
    B, H, D = q.shape
    P, page_size, KVH, Dk = k_pages.shape
    if k_pages.shape != v_pages.shape or Dk != D:
        raise ValueError("shape mismatch between q and the page pools")
    bt = np.ascontiguousarray(np.asarray(block_table, dtype=np.int32))
    if bt.ndim != 2 or bt.shape[0] != B:
        raise ValueError("block_table must have shape [B, max_pages]")
    lens = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32))
    out = np.zeros((B, H, D), dtype=np.float64)
    lib = _lib_override if _lib_override is not None else _load()
    rc = lib.oracle_gqa_decode_paged_f64(
        _ptr(q, ctypes.c_uint16), _ptr(k_pages, ctypes.c_uint16), _ptr(v_pages, ctypes.c_uint16),
        _ptr(bt, ctypes.c_int32), _ptr(lens, ctypes.c_int32), B, P, bt.shape[1], page_size,
        H, KVH, D, int(window), int(nthreads), _ptr(out, ctypes.c_double))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")
    return out


def gqa_decode_ring_f64(q: np.ndarray, k: np.ndarray, v: np.ndarray, seq_lens, window: int,
                        nthreads: int = 0, _lib_override=None) -> np.ndarray:
    """Decode attention over a window-capped ring-buffer cache, exact up to fp64 rounding.

    k, v: uint16 [B, C, KVH, D]; position s of sequence b is row s % C.  The
    attended positions are [max(0, L - window), L) with 1 <= window <= C, so all of
    them are still in the ring; L may exceed C.
    """
    q, k, v = _u16(q), _u16(k), _u16(v)
    B, H, D = q.shape
    Bk, C, KVH, Dk = k.shape
    if k.shape != v.shape or Bk != B or Dk != D:
        raise ValueError("shape mismatch between q, k and v")
    lens = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32))
    if lens.shape != (B,):
        raise ValueError("seq_lens must have shape [B]")
    out = np.zeros((B, H, D), dtype=np.float64)
    lib = _lib_override if _lib_override is not None else _load()
    rc = lib.oracle_gqa_decode_ring_f64(
        _ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16), _ptr(v, ctypes.c_uint16),
        _ptr(lens, ctypes.c_int32), B, C, H, KVH, D, int(window), int(nthreads),
        _ptr(out, ctypes.c_double))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")
    return out


def gqa_decode_mq_f64(q: np.ndarray, k: np.ndarray, v: np.ndarray, seq_lens, window: int,
                      nthreads: int = 0, _lib_override=None) -> np.ndarray:
    """Multi-query decode attention over a contiguous cache, exact up to fp64 rounding.

    q: uint16 [B, T, H, D]; k, v: uint16 [B, S, KVH, D], row s = position s;
    seq_lens: lengths after the T new tokens were appended.  Query t of sequence b
    sits at position L_b - T + t and attends to [max(0, p + 1 - window), p + 1)
    (sliding) or [0, p + 1) (window 0); a negative position attends to nothing
    (o = 0).  Returns float64 [B, T, H, D].
    """
    q, k, v = _u16(q), _u16(k), _u16(v)
    B, T, H, D = q.shape
    Bk, S, KVH, Dk = k.shape
    if k.shape != v.shape or Bk != B or Dk != D:
        raise ValueError("shape mismatch between q, k and v")
    lens = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32))
    if lens.shape != (B,):
        raise ValueError("seq_lens must have shape [B]")
    out = np.zeros((B, T, H, D), dtype=np.float64)
    lib = _lib_override if _lib_override is not None else _load()
    rc = lib.oracle_gqa_decode_mq_f64(
        _ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16), _ptr(v, ctypes.c_uint16),
        _ptr(lens, ctypes.c_int32), B, T, S, H, KVH, D, int(window), int(nthreads),
        _ptr(out, ctypes.c_double))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")
    return out


def gqa_decode_mq_paged_f64(q: np.ndarray, k_pages: np.ndarray, v_pages: np.ndarray,
                            block_table: np.ndarray, seq_lens, window: int,
                            nthreads: int = 0, _lib_override=None) -> np.ndarray:
    """Multi-query decode attention over a paged cache, exact up to fp64 rounding.

    q: uint16 [B, T, H, D]; pools uint16 [P, page_size, KVH, D]; block_table int32
    [B, max_pages].  A query whose attended range names a page outside [0, P) gets
    NaN for all of its heads.
    """
    q, k_pages, v_pages = _u16(q), _u16(k_pages), _u16(v_pages)
    B, T, H, D = q.shape
    P, page_size, KVH, Dk = k_pages.shape
    if k_pages.shape != v_pages.shape or Dk != D:
        raise ValueError("shape mismatch between q and the page pools")
    bt = np.ascontiguousarray(np.asarray(block_table, dtype=np.int32))
    if bt.ndim != 2 or bt.shape[0] != B:
        raise ValueError("block_table must have shape [B, max_pages]")
    lens = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32))
    out = np.zeros((B, T, H, D), dtype=np.float64)
    lib = _lib_override if _lib_override is not None else _load()
    rc = lib.oracle_gqa_decode_mq_paged_f64(
        _ptr(q, ctypes.c_uint16), _ptr(k_pages, ctypes.c_uint16), _ptr(v_pages, ctypes.c_uint16),
        _ptr(bt, ctypes.c_int32), _ptr(lens, ctypes.c_int32), B, T, P, bt.shape[1], page_size,
        H, KVH, D, int(window), int(nthreads), _ptr(out, ctypes.c_double))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")
    return out


# RoPE of the global layers (Model Spec, `attn.rope` row for layers 5, 11, ..., 59)
GLOBAL_ROPE_PAIRS = 64
GLOBAL_ROPE_THETA = 1.0e6


def gqa_decode_keqv_f64(q: np.ndarray, v: np.ndarray, w_k: np.ndarray, seq_lens, window: int,
                        n_rot: int = GLOBAL_ROPE_PAIRS, theta: float = GLOBAL_ROPE_THETA,
                        nthreads: int = 0, _lib_override=None) -> np.ndarray:
    """Decode attention over a single K=V cache, exact up to fp64 rounding.

    v: uint16 [B, S, KVH, D], the cached values (row s is position s); w_k: uint16
    [D], the k_norm weight.  The key of row s is rope(w_k * v[s], s): pairs
    (i, i + D/2), i < n_rot, rotated by s * theta^(-2i/D).
    """
    q, v, w_k = _u16(q), _u16(v), _u16(w_k)
    B, H, D = q.shape
    Bv, S, KVH, Dv = v.shape
    if Bv != B or Dv != D or w_k.shape != (D,):
        raise ValueError("shape mismatch between q, v and w_k")
    lens = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32))
    if lens.shape != (B,):
        raise ValueError("seq_lens must have shape [B]")
    out = np.zeros((B, H, D), dtype=np.float64)
    lib = _lib_override if _lib_override is not None else _load()
    rc = lib.oracle_gqa_decode_keqv_f64(
        _ptr(q, ctypes.c_uint16), _ptr(v, ctypes.c_uint16), _ptr(w_k, ctypes.c_uint16),
        _ptr(lens, ctypes.c_int32), B, S, H, KVH, D, int(window), int(n_rot), float(theta),
        int(nthreads), _ptr(out, ctypes.c_double))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")
    return out


# RoPE of the sliding layers (Model Spec, `attn.rope` row for the other 50 layers)
SLIDING_ROPE_PAIRS = 128
SLIDING_ROPE_THETA = 1.0e4


def prepare_decode_f64(q_raw: np.ndarray, k_raw: np.ndarray, v_raw, w_q: np.ndarray,
                       w_k: np.ndarray, seq_lens, n_rot: int, theta: float,
                       _lib_override=None):
    """The decode-step producer for one new token per sequence, exact up to fp64.

    q_raw [B, H, D], k_raw [B, KVH, D], v_raw [B, KVH, D] or None (values = keys),
    w_q, w_k [D]: uint16 bf16 bits.  Returns (q, k, v) float64: q = rope(q_norm(q_raw)),
    k = rope(k_norm(k_raw)), v = v_norm(v_raw or k_raw), at position seq_lens[b] - 1
    (NaN where seq_lens[b] < 1).
    """
    q_raw, k_raw, w_q, w_k = _u16(q_raw), _u16(k_raw), _u16(w_q), _u16(w_k)
    B, H, D = q_raw.shape
    _, KVH, _ = k_raw.shape
    if v_raw is not None:
        v_raw = _u16(v_raw)
        if v_raw.shape != k_raw.shape:
            raise ValueError("v_raw must match k_raw")
    lens = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32))
    q = np.zeros((B, H, D)); k = np.zeros((B, KVH, D)); v = np.zeros((B, KVH, D))
    lib = _lib_override if _lib_override is not None else _load()
    rc = lib.oracle_prepare_decode_f64(
        _ptr(q_raw, ctypes.c_uint16), _ptr(k_raw, ctypes.c_uint16),
        None if v_raw is None else _ptr(v_raw, ctypes.c_uint16), _ptr(w_q, ctypes.c_uint16),
        _ptr(w_k, ctypes.c_uint16), _ptr(lens, ctypes.c_int32), B, H, KVH, D, int(n_rot),
        float(theta), _ptr(q, ctypes.c_double), _ptr(k, ctypes.c_double), _ptr(v, ctypes.c_double))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")
    return q, k, v


class OracleLibrary:
    """The oracle API bound to a specific compiled copy of the C source.

    Used by the mutation tests, which compile deliberately broken copies of
    ``gqa_oracle.c`` and check that the pins reject each of them.
    """

    def __init__(self, so_path: str):
        self._lib = _bind(so_path)

    def gqa_decode_f64(self, *args, **kw):
        return gqa_decode_f64(*args, _lib_override=self._lib, **kw)

    def gqa_decode_paged_f64(self, *args, **kw):
        return gqa_decode_paged_f64(*args, _lib_override=self._lib, **kw)

    def gqa_decode_ring_f64(self, *args, **kw):
        return gqa_decode_ring_f64(*args, _lib_override=self._lib, **kw)

    def gqa_decode_keqv_f64(self, *args, **kw):
        return gqa_decode_keqv_f64(*args, _lib_override=self._lib, **kw)

    def prepare_decode_f64(self, *args, **kw):
        return prepare_decode_f64(*args, _lib_override=self._lib, **kw)

    def gqa_decode_mq_f64(self, *args, **kw):
        return gqa_decode_mq_f64(*args, _lib_override=self._lib, **kw)

    def gqa_decode_mq_paged_f64(self, *args, **kw):
        return gqa_decode_mq_paged_f64(*args, _lib_override=self._lib, **kw)


def compile_variant(source_text: str, out_path: str) -> str:
    """Compile C source text with the oracle's flags into ``out_path``."""
    src = out_path[:-3] + ".c"
    with open(src, "w") as f:
        f.write(source_text)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-w",
                    "-o", out_path, src, "-lm"], check=True)
    return out_path


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()
