"""fp64 CPU oracle for single-query decode attention (dense, paged, sparse).

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline leg may import this package.  The library under
``token_decode_attention_split_gb300`` never imports it and shares no code with it.

The arithmetic lives in ``oracle.c`` (plain C, fp64, one thread per (b, h) shard); this module
only compiles it with gcc and marshals numpy arrays into it.  Inputs are bf16 bit patterns
(``numpy.uint16``), widened exactly to double inside the C code.

What each function computes, with the page each follows:
  * ``dense``  -- "DecodeFlashSpec" (fuel_dispatch::decode_flash), fields k / v / k_len /
    softmax_scale: rows [0, k_len) of a capacity buffer [B, Hkv, capacity, D].
  * ``paged``  -- "DflashScratch" (metrale dflash_head), field option_b_indirect_args_dev: the
    per-sequence kv_len is the first u32 of each args record; rows gathered through a block table.
  * ``sparse`` -- "AttnV41" (metrale attn_v41), method decode_fixed_topk: a fixed-width int32
    selection whose -1 entries add nothing.
  * ``dense_range`` -- the same dense definition restricted to rows [j0, j1), returning the
    normalised row and its natural-log log-sum-exp (for the split/merge identity tests).
  * ``dense_mq`` / ``paged_mq`` -- several query tokens per sequence (q, out [B, Hq, Sq, D]): the
    Sq new tokens are the last Sq rows of the live prefix; causal token i attends rows
    [0, len - Sq + i] ("DecodeFlashSpec", q [B,Hq,Sq,D] and field causal; "AttnV41", forward).
  * ``append_paged`` -- "DflashScratch", field slot_mapping_dev (reshape_and_cache): new K/V rows
    scattered to paged-cache slots; ``append_ring`` -- "AttnV41", method decode_body: the ring
    write at pos % window.  Both return updated copies of the pools.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``_build/liboracle.so`` (gcc, -O2, no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-pthread", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        u16p = ctypes.POINTER(ctypes.c_uint16)
        f64p = ctypes.POINTER(ctypes.c_double)
        i32p = ctypes.POINTER(ctypes.c_int32)
        u32p = ctypes.POINTER(ctypes.c_uint32)
        i64p = ctypes.POINTER(ctypes.c_int64)
        i, i64, d = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.oracle_dense.argtypes = [u16p, u16p, u16p, f64p, i, i, i, i, i64, i64, d, i64p, i64, i]
        lib.oracle_paged.argtypes = [u16p, u16p, u16p, f64p, i32p, i64, i64, i64, u32p, i64,
                                     i, i, i, i, d, i64p, i64, i]
        lib.oracle_sparse.argtypes = [u16p, u16p, u16p, f64p, i64, i32p, i64, i, i, i, i, d,
                                      i64p, i64, i]
        lib.oracle_dense_range.argtypes = [u16p, u16p, u16p, i, i, i, i, i64, i, i, i64, i64, d,
                                           f64p, f64p]
        lib.oracle_dense_mq.argtypes = [u16p, u16p, u16p, f64p, i, i, i, i, i, i, i64, i64, d, i]
        lib.oracle_paged_mq.argtypes = [u16p, u16p, u16p, f64p, i32p, i64, i64, i64, u32p, i64,
                                        i, i, i, i, i, i, d, i]
        lib.oracle_append_paged.argtypes = [u16p, u16p, u16p, u16p, i64p, i64, i, i, i64, i64]
        lib.oracle_append_ring.argtypes = [u16p, u16p, u16p, u16p, i64p, i, i, i, i64, i64]
        for f in (lib.oracle_dense, lib.oracle_paged, lib.oracle_sparse, lib.oracle_dense_range,
                  lib.oracle_append_paged, lib.oracle_append_ring, lib.oracle_dense_mq,
                  lib.oracle_paged_mq):
            f.restype = ctypes.c_int
        _lib = lib
        return lib


def _bits(a) -> np.ndarray:
    """bf16 bit patterns as a C-contiguous uint16 array (accepts uint16 arrays or bf16 torch tensors)."""
    if not isinstance(a, np.ndarray):
        import torch  # only for unwrapping torch tensors handed in by tests
        t = a.detach().to("cpu").contiguous()
        if t.dtype != torch.bfloat16:
            raise TypeError("oracle inputs must be bfloat16 tensors or uint16 bit arrays")
        a = t.view(torch.int16).numpy().view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError("oracle inputs must be bf16 bit patterns (uint16)")
    return np.ascontiguousarray(a)


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _pairs_arg(pairs):
    if pairs is None:
        return None, None, 0
    p = np.ascontiguousarray(np.asarray(pairs, dtype=np.int64).reshape(-1))
    return p, _ptr(p, ctypes.c_int64), p.size


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle_{what} rejected its arguments (code {rc})")


def dense(q, k, v, k_len: int, scale: float, pairs=None, nthreads: int = 0) -> np.ndarray:
    """q [B,Hq,1,D] or [B,Hq,D]; k, v [B,Hkv,capacity,D]; returns fp64 [B,Hq,D].

    With ``pairs`` (flat b*Hq + h indices) only those rows are computed; the rest stay NaN.
    """
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    B, Hkv, cap, D = kb.shape
    Hq = qb.size // (B * D)
    out = np.full((B, Hq, D), np.nan, dtype=np.float64)
    p, pp, n = _pairs_arg(pairs)
    if pairs is None:
        out[:] = 0.0
    rc = _load().oracle_dense(_ptr(qb, ctypes.c_uint16), _ptr(kb, ctypes.c_uint16),
                              _ptr(vb, ctypes.c_uint16), _ptr(out, ctypes.c_double), B, Hq, Hkv,
                              D, cap, int(k_len), float(scale), pp, n, int(nthreads))
    _check(rc, "dense")
    return out


def paged(q, k_pool, v_pool, block_table, kv_lens, scale: float, kv_len_stride: int = 1,
          Hq: int | None = None, pairs=None, nthreads: int = 0) -> np.ndarray:
    """Pools [num_pages,Hkv,page_size,D]; block_table int32 [B,max_pages]; kv_lens uint32 args
    buffer read at ``b * kv_len_stride``; returns fp64 [B,Hq,D]."""
    qb, kb, vb = _bits(q), _bits(k_pool), _bits(v_pool)
    num_pages, Hkv, P, D = kb.shape
    bt = np.ascontiguousarray(np.asarray(block_table, dtype=np.int32))
    B, max_pages = bt.shape
    kl = np.ascontiguousarray(np.asarray(kv_lens, dtype=np.uint32).reshape(-1))
    if kl.size < (B - 1) * kv_len_stride + 1 and B > 0:
        raise ValueError("kv_lens buffer too short for B and stride")
    Hq = qb.size // (B * D) if Hq is None else Hq
    out = np.full((B, Hq, D), np.nan, dtype=np.float64)
    p, pp, n = _pairs_arg(pairs)
    if pairs is None:
        out[:] = 0.0
    rc = _load().oracle_paged(_ptr(qb, ctypes.c_uint16), _ptr(kb, ctypes.c_uint16),
                              _ptr(vb, ctypes.c_uint16), _ptr(out, ctypes.c_double),
                              _ptr(bt, ctypes.c_int32), max_pages, P, num_pages,
                              _ptr(kl, ctypes.c_uint32), int(kv_len_stride), B, Hq, Hkv, D,
                              float(scale), pp, n, int(nthreads))
    _check(rc, "paged")
    return out


def sparse(q, k_pool, v_pool, sel, scale: float, pairs=None, nthreads: int = 0) -> np.ndarray:
    """Pools [B,Hkv,pool_rows,D]; sel int32 [B,width]; returns fp64 [B,Hq,D]."""
    qb, kb, vb = _bits(q), _bits(k_pool), _bits(v_pool)
    B, Hkv, R, D = kb.shape
    s = np.ascontiguousarray(np.asarray(sel, dtype=np.int32))
    if s.ndim != 2 or s.shape[0] != B:
        raise ValueError("sel must be [B, width]")
    W = s.shape[1]
    Hq = qb.size // (B * D)
    out = np.full((B, Hq, D), np.nan, dtype=np.float64)
    p, pp, n = _pairs_arg(pairs)
    if pairs is None:
        out[:] = 0.0
    rc = _load().oracle_sparse(_ptr(qb, ctypes.c_uint16), _ptr(kb, ctypes.c_uint16),
                               _ptr(vb, ctypes.c_uint16), _ptr(out, ctypes.c_double), R,
                               _ptr(s, ctypes.c_int32), W, B, Hq, Hkv, D, float(scale), pp, n,
                               int(nthreads))
    _check(rc, "sparse")
    return out


def dense_range(q, k, v, b: int, h: int, j0: int, j1: int, scale: float):
    """Dense attention of (b, h) over rows [j0, j1): (o [D] fp64, lse natural log)."""
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    B, Hkv, cap, D = kb.shape
    Hq = qb.size // (B * D)
    o = np.zeros(D, dtype=np.float64)
    lse = ctypes.c_double(0.0)
    rc = _load().oracle_dense_range(_ptr(qb, ctypes.c_uint16), _ptr(kb, ctypes.c_uint16),
                                    _ptr(vb, ctypes.c_uint16), B, Hq, Hkv, D, cap, b, h, j0, j1,
                                    float(scale), _ptr(o, ctypes.c_double), ctypes.byref(lse))
    _check(rc, "dense_range")
    return o, lse.value


def append_paged(k_new, v_new, k_pool, v_pool, slot_mapping, inplace: bool = False):
    """k_new, v_new [T,Hkv,D]; pools [num_pages,Hkv,page_size,D]; slot_mapping int64 [T].
    Returns (k_pool', v_pool') as new uint16 arrays (inplace=True writes into the given uint16
    pool arrays instead and returns them)."""
    kn, vn = _bits(k_new), _bits(v_new)
    if inplace:
        kp, vp = k_pool, v_pool
        if not (isinstance(kp, np.ndarray) and kp.dtype == np.uint16 and kp.flags.c_contiguous
                and isinstance(vp, np.ndarray) and vp.dtype == np.uint16 and vp.flags.c_contiguous):
            raise TypeError("inplace append needs C-contiguous uint16 pool arrays")
    else:
        kp, vp = _bits(k_pool).copy(), _bits(v_pool).copy()
    sm = np.ascontiguousarray(np.asarray(slot_mapping, dtype=np.int64).reshape(-1))
    T = sm.size
    num_pages, Hkv, P, D = kp.shape
    if kn.size != T * Hkv * D or vn.size != kn.size:
        raise ValueError("k_new / v_new must be [T, Hkv, D]")
    rc = _load().oracle_append_paged(_ptr(kn, ctypes.c_uint16), _ptr(vn, ctypes.c_uint16),
                                     _ptr(kp, ctypes.c_uint16), _ptr(vp, ctypes.c_uint16),
                                     _ptr(sm, ctypes.c_int64), T, Hkv, D, P, num_pages)
    _check(rc, "append_paged")
    return kp, vp


def append_ring(k_new, v_new, k_pool, v_pool, positions, window: int):
    """k_new, v_new [B,Hkv,D]; pools [B,Hkv,pool_rows,D]; positions int64 [B].
    Returns (k_pool', v_pool') as new uint16 arrays; the inputs are not modified."""
    kn, vn = _bits(k_new), _bits(v_new)
    kp, vp = _bits(k_pool).copy(), _bits(v_pool).copy()
    pos = np.ascontiguousarray(np.asarray(positions, dtype=np.int64).reshape(-1))
    B, Hkv, R, D = kp.shape
    if pos.size != B or kn.size != B * Hkv * D or vn.size != kn.size:
        raise ValueError("k_new / v_new must be [B, Hkv, D] and positions [B]")
    rc = _load().oracle_append_ring(_ptr(kn, ctypes.c_uint16), _ptr(vn, ctypes.c_uint16),
                                    _ptr(kp, ctypes.c_uint16), _ptr(vp, ctypes.c_uint16),
                                    _ptr(pos, ctypes.c_int64), B, Hkv, D, R, int(window))
    _check(rc, "append_ring")
    return kp, vp


def dense_mq(q, k, v, k_len: int, scale: float, causal: bool = True, nthreads: int = 0):
    """q [B,Hq,Sq,D]; k, v [B,Hkv,capacity,D]; returns fp64 [B,Hq,Sq,D]."""
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    B, Hkv, cap, D = kb.shape
    if qb.ndim != 4:
        raise ValueError("q must be [B, Hq, Sq, D]")
    Hq, Sq = qb.shape[1], qb.shape[2]
    out = np.zeros((B, Hq, Sq, D), dtype=np.float64)
    rc = _load().oracle_dense_mq(_ptr(qb, ctypes.c_uint16), _ptr(kb, ctypes.c_uint16),
                                 _ptr(vb, ctypes.c_uint16), _ptr(out, ctypes.c_double), B, Hq, Hkv,
                                 D, Sq, int(bool(causal)), cap, int(k_len), float(scale),
                                 int(nthreads))
    _check(rc, "dense_mq")
    return out


def paged_mq(q, k_pool, v_pool, block_table, kv_lens, scale: float, causal: bool = True,
             kv_len_stride: int = 1, nthreads: int = 0):
    """q [B,Hq,Sq,D]; pools [num_pages,Hkv,page_size,D]; returns fp64 [B,Hq,Sq,D]."""
    qb, kb, vb = _bits(q), _bits(k_pool), _bits(v_pool)
    num_pages, Hkv, P, D = kb.shape
    bt = np.ascontiguousarray(np.asarray(block_table, dtype=np.int32))
    B, max_pages = bt.shape
    kl = np.ascontiguousarray(np.asarray(kv_lens, dtype=np.uint32).reshape(-1))
    Hq, Sq = qb.shape[1], qb.shape[2]
    out = np.zeros((B, Hq, Sq, D), dtype=np.float64)
    rc = _load().oracle_paged_mq(_ptr(qb, ctypes.c_uint16), _ptr(kb, ctypes.c_uint16),
                                 _ptr(vb, ctypes.c_uint16), _ptr(out, ctypes.c_double),
                                 _ptr(bt, ctypes.c_int32), max_pages, P, num_pages,
                                 _ptr(kl, ctypes.c_uint32), int(kv_len_stride), B, Hq, Hkv, D, Sq,
                                 int(bool(causal)), float(scale), int(nthreads))
    _check(rc, "paged_mq")
    return out
