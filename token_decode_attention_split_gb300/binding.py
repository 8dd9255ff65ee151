"""ctypes binding of ``libdecode_attn.so`` (the C ABI in ``include/decode_attn.h``).

Argument marshalling only: tensors become device pointers, shapes become ints, the current
torch stream becomes the cudaStream_t.  Every step of the computation runs in the library's
CUDA kernels; there is no fallback, and a missing library raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

DA_VARIANT_DENSE, DA_VARIANT_PAGED, DA_VARIANT_SPARSE = 0, 1, 2
_lock = threading.Lock()
_lib = None


class DecodeAttnSpec(ctypes.Structure):
    """``decode_attn_spec``: the options of a decode-attention region (nonzero has_* = present)."""
    _fields_ = [("has_alibi", ctypes.c_int), ("causal", ctypes.c_int),
                ("has_window_left", ctypes.c_int), ("has_window_right", ctypes.c_int),
                ("has_softcap", ctypes.c_int), ("softmax_scale", ctypes.c_float)]


class DecodeAttnError(RuntimeError):
    def __init__(self, status: int, what: str, text: str):
        super().__init__(f"{what}: {text} (status {status})")
        self.status = status


def library_path() -> str:
    return _build.LIB


def load_library() -> ctypes.CDLL:
    """Loads the built library; raises if it has not been built (``__graft_entry__.build()``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise ImportError(f"decode-attention CUDA library not built: {path} is missing")
        lib = ctypes.CDLL(path)
        vp, sz, i, i64, f = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_int64, ctypes.c_float
        lib.decode_attn_abi_version.restype = i
        lib.decode_attn_abi_version.argtypes = []
        lib.decode_attn_status_string.restype = ctypes.c_char_p
        lib.decode_attn_status_string.argtypes = [i]
        lib.decode_attn_workspace_size.restype = sz
        lib.decode_attn_workspace_size.argtypes = [i, i, i, i, i, i64]
        lib.decode_attn_workspace_init.restype = i
        lib.decode_attn_workspace_init.argtypes = [vp, sz, vp]
        lib.decode_attn_dense.restype = i
        lib.decode_attn_dense.argtypes = [vp, vp, vp, vp, i, i, i, i, i64, i64, f, vp, sz, vp]
        lib.decode_attn_dense_device_len.restype = i
        lib.decode_attn_dense_device_len.argtypes = [vp, vp, vp, vp, i, i, i, i, i64, vp, f, vp, sz,
                                                     vp]
        lib.decode_attn_paged.restype = i
        lib.decode_attn_paged.argtypes = [vp, vp, vp, vp, vp, i, i, i64, vp, i, i, i, i, i, f, vp,
                                          sz, vp]
        lib.decode_attn_dense_mq.restype = i
        lib.decode_attn_dense_mq.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i64, i64, f, vp, sz,
                                             vp]
        lib.decode_attn_paged_mq.restype = i
        lib.decode_attn_paged_mq.argtypes = [vp, vp, vp, vp, vp, i, i, i64, vp, i, i, i, i, i, i,
                                             i, f, vp, sz, vp]
        lib.decode_attn_sparse.restype = i
        lib.decode_attn_sparse.argtypes = [vp, vp, vp, vp, i64, vp, i, i, i, i, i, f, vp, sz, vp]
        lib.decode_attn_append_paged.restype = i
        lib.decode_attn_append_paged.argtypes = [vp, vp, vp, vp, vp, i64, i, i, i, i64, vp]
        lib.decode_attn_append_ring.restype = i
        lib.decode_attn_append_ring.argtypes = [vp, vp, vp, vp, vp, i, i, i, i64, i, vp]
        lib.decode_attn_set_grid_limit.restype = i
        lib.decode_attn_set_grid_limit.argtypes = [i]
        lib.decode_attn_read_device_error.restype = i
        lib.decode_attn_read_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
        lib.decode_attn_check_wait_timeout.restype = i
        lib.decode_attn_check_wait_timeout.argtypes = [ctypes.c_uint32, vp]
        lib.decode_attn_spec_check.restype = i
        lib.decode_attn_spec_check.argtypes = [ctypes.POINTER(DecodeAttnSpec)]
        lib.decode_attn_dense_spec.restype = i
        lib.decode_attn_dense_spec.argtypes = [ctypes.POINTER(DecodeAttnSpec), vp, vp, vp, vp, i, i, i,
                                               i, i64, i64, vp, sz, vp]
        lib.decode_attn_dense_noalloc.restype = i
        lib.decode_attn_dense_noalloc.argtypes = [vp, vp, vp, vp, i, i, i, i, i64, i64, f, vp]
        _lib = lib
        return lib


def _check(status: int, what: str):
    if status != 0:
        text = load_library().decode_attn_status_string(status).decode()
        raise DecodeAttnError(status, what, text)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def abi_version() -> int:
    return load_library().decode_attn_abi_version()


def decode_attn_abi_version() -> int:
    return abi_version()


def decode_attn_status_string(status: int) -> str:
    return load_library().decode_attn_status_string(int(status)).decode()


def decode_attn_spec_check(spec: DecodeAttnSpec) -> int:
    """The gate: 0 (DA_OK) when these kernels can compute the region, else the refusing status
    (DA_ERR_UNSUPPORTED for ALiBi / a window bound / a softcap).  Host only."""
    return int(load_library().decode_attn_spec_check(ctypes.byref(spec) if spec is not None else None))


def decode_attn_dense_spec(spec: DecodeAttnSpec, q, k, v, out, k_len: int, workspace, stream=None):
    """decode_attn_spec_check, then decode_attn_dense with spec.softmax_scale."""
    B, Hq, D = _dims_q(q)
    Hkv, cap = k.shape[1], k.shape[2]
    _check(load_library().decode_attn_dense_spec(
        ctypes.byref(spec), _ptr(q), _ptr(k), _ptr(v), _ptr(out), B, Hq, Hkv, D, cap, int(k_len),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream, q.device)),
        "decode_attn_dense_spec")
    return out


def decode_attn_dense_noalloc(q, k, v, out, k_len: int, softmax_scale: float, stream=None):
    """decode_attn_dense with the library-owned device scratch as its workspace (no allocation;
    calls sharing the scratch must not overlap)."""
    B, Hq, D = _dims_q(q)
    Hkv, cap = k.shape[1], k.shape[2]
    _check(load_library().decode_attn_dense_noalloc(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), B, Hq, Hkv, D, cap, int(k_len),
        float(softmax_scale), _stream(stream, q.device)), "decode_attn_dense_noalloc")
    return out


def decode_attn_workspace_size(variant: int, B: int, Hq: int, Hkv: int, D: int, max_kv: int = 0) -> int:
    return int(load_library().decode_attn_workspace_size(variant, B, Hq, Hkv, D, max_kv))


def decode_attn_workspace_init(workspace: torch.Tensor, stream=None):
    _check(load_library().decode_attn_workspace_init(
        _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream, workspace.device)), "decode_attn_workspace_init")


def new_workspace(nbytes: int, device) -> torch.Tensor:
    """A zero-filled workspace buffer (16-byte aligned torch allocation)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def decode_attn_set_grid_limit(max_ctas: int):
    _check(load_library().decode_attn_set_grid_limit(int(max_ctas)), "decode_attn_set_grid_limit")


def decode_attn_read_device_error() -> int:
    code = ctypes.c_uint32(0)
    _check(load_library().decode_attn_read_device_error(ctypes.byref(code)),
           "decode_attn_read_device_error")
    return int(code.value)


def decode_attn_check_wait_timeout(limit_us: int, stream=None, device="cuda"):
    """Enqueues the bounded-wait check: a wait that nothing completes gives up after limit_us
    and records code 5 in the device error word (read it with decode_attn_read_device_error)."""
    _check(load_library().decode_attn_check_wait_timeout(int(limit_us), _stream(stream, device)),
           "decode_attn_check_wait_timeout")


def _dims_q(q):
    if q.dim() != 4 or q.shape[2] != 1:
        raise ValueError("q must be [B, Hq, 1, D]")
    return q.shape[0], q.shape[1], q.shape[3]


def decode_attn_dense(q, k, v, out, k_len: int, softmax_scale: float, workspace, stream=None):
    """q, out [B,Hq,1,D]; k, v [B,Hkv,capacity,D]; all bf16 CUDA tensors, contiguous."""
    B, Hq, D = _dims_q(q)
    Hkv, cap = k.shape[1], k.shape[2]
    _check(load_library().decode_attn_dense(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), B, Hq, Hkv, D, cap, int(k_len), float(softmax_scale),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream, q.device)),
        "decode_attn_dense")
    return out


def decode_attn_dense_device_len(q, k, v, out, k_len_dev, softmax_scale: float, workspace,
                                 stream=None):
    """As decode_attn_dense, with the live length read on the device from k_len_dev (a one-word
    int32 CUDA tensor holding the u32 length)."""
    B, Hq, D = _dims_q(q)
    Hkv, cap = k.shape[1], k.shape[2]
    _check(load_library().decode_attn_dense_device_len(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), B, Hq, Hkv, D, cap, _ptr(k_len_dev),
        float(softmax_scale), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream, q.device)), "decode_attn_dense_device_len")
    return out


def decode_attn_paged(q, k_pool, v_pool, out, block_table, kv_lens, kv_len_stride: int,
                      softmax_scale: float, workspace, stream=None):
    """Pools [num_pages,Hkv,page_size,D] bf16; block_table int32 [B,max_pages]; kv_lens int32
    tensor holding the u32 words (kv_len of sequence b at b * kv_len_stride)."""
    B, Hq, D = _dims_q(q)
    num_pages, Hkv, P = k_pool.shape[0], k_pool.shape[1], k_pool.shape[2]
    _check(load_library().decode_attn_paged(
        _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(out), _ptr(block_table), block_table.shape[1], P,
        num_pages, _ptr(kv_lens), int(kv_len_stride), B, Hq, Hkv, D, float(softmax_scale),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream, q.device)),
        "decode_attn_paged")
    return out


def decode_attn_dense_mq(q, k, v, out, k_len: int, causal: bool, softmax_scale: float, workspace,
                         stream=None):
    """q, out [B,Hq,Sq,D]; k, v [B,Hkv,capacity,D]: Sq query tokens per sequence."""
    B, Hq, Sq, D = q.shape
    Hkv, cap = k.shape[1], k.shape[2]
    _check(load_library().decode_attn_dense_mq(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), B, Hq, Hkv, D, Sq, int(bool(causal)), cap,
        int(k_len), float(softmax_scale), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream, q.device)),
        "decode_attn_dense_mq")
    return out


def decode_attn_paged_mq(q, k_pool, v_pool, out, block_table, kv_lens, kv_len_stride: int,
                         causal: bool, softmax_scale: float, workspace, stream=None):
    """q, out [B,Hq,Sq,D]; pools and lengths as for decode_attn_paged."""
    B, Hq, Sq, D = q.shape
    num_pages, Hkv, P = k_pool.shape[0], k_pool.shape[1], k_pool.shape[2]
    _check(load_library().decode_attn_paged_mq(
        _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(out), _ptr(block_table), block_table.shape[1], P,
        num_pages, _ptr(kv_lens), int(kv_len_stride), B, Hq, Hkv, D, Sq, int(bool(causal)),
        float(softmax_scale), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream, q.device)), "decode_attn_paged_mq")
    return out


def decode_attn_sparse(q, k_pool, v_pool, out, sel, softmax_scale: float, workspace, stream=None):
    """Pools [B,Hkv,pool_rows,D] bf16; sel int32 [B,width]."""
    B, Hq, D = _dims_q(q)
    Hkv, R = k_pool.shape[1], k_pool.shape[2]
    _check(load_library().decode_attn_sparse(
        _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(out), R, _ptr(sel), sel.shape[1], B, Hq, Hkv, D,
        float(softmax_scale), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream, q.device)), "decode_attn_sparse")
    return out


def decode_attn_append_paged(k_new, v_new, k_pool, v_pool, slot_mapping, stream=None):
    """k_new, v_new [T,Hkv,D] bf16; pools [num_pages,Hkv,page_size,D]; slot_mapping int64 [T]."""
    T, Hkv, D = k_new.shape
    _check(load_library().decode_attn_append_paged(
        _ptr(k_new), _ptr(v_new), _ptr(k_pool), _ptr(v_pool), _ptr(slot_mapping), T, Hkv, D,
        k_pool.shape[2], k_pool.shape[0], _stream(stream, k_new.device)), "decode_attn_append_paged")


def decode_attn_append_ring(k_new, v_new, k_pool, v_pool, positions, window: int, stream=None):
    """k_new, v_new [B,Hkv,D] bf16; pools [B,Hkv,pool_rows,D]; positions int64 [B]."""
    B, Hkv, D = k_new.shape
    _check(load_library().decode_attn_append_ring(
        _ptr(k_new), _ptr(v_new), _ptr(k_pool), _ptr(v_pool), _ptr(positions), B, Hkv, D,
        k_pool.shape[2], int(window), _stream(stream, k_new.device)), "decode_attn_append_ring")


def run_case(case, out=None, workspace=None, stream=None):
    """Runs one workload object (``workloads.DenseCase`` / ``PagedCase`` / ``SparseCase``) through
    the matching entry point, allocating the output and a zeroed workspace when not given."""
    if case.kind == "append":
        decode_attn_append_paged(case.k_new, case.v_new, case.k_pool, case.v_pool,
                                 case.slot_mapping, stream)
        return case.k_pool
    dev = case.q.device
    if out is None:
        out = torch.empty(case.out_shape(), dtype=torch.bfloat16, device=dev)
    if case.kind == "dense":
        sq = getattr(case, "sq", 1)
        if workspace is None:
            workspace = new_workspace(decode_attn_workspace_size(
                DA_VARIANT_DENSE, case.B, case.Hq * sq, case.Hkv, case.D), dev)
        if sq > 1:
            return decode_attn_dense_mq(case.q, case.k, case.v, out, case.k_len, case.causal,
                                        case.scale, workspace, stream)
        if getattr(case, "k_len_dev", None) is not None:
            return decode_attn_dense_device_len(case.q, case.k, case.v, out, case.k_len_dev,
                                                case.scale, workspace, stream)
        return decode_attn_dense(case.q, case.k, case.v, out, case.k_len, case.scale, workspace,
                                 stream)
    if case.kind == "paged":
        if workspace is None:
            workspace = new_workspace(decode_attn_workspace_size(
                DA_VARIANT_PAGED, case.B, case.Hq, case.Hkv, case.D), dev)
        return decode_attn_paged(case.q, case.k_pool, case.v_pool, out, case.block_table,
                                 case.kv_args, case.kv_len_stride, case.scale, workspace, stream)
    if case.kind == "sparse":
        if workspace is None:
            workspace = new_workspace(decode_attn_workspace_size(
                DA_VARIANT_SPARSE, case.B, case.Hq, case.Hkv, case.D, case.width), dev)
        return decode_attn_sparse(case.q, case.k_pool, case.v_pool, out, case.sel, case.scale,
                                  workspace, stream)
    raise ValueError(case.kind)
