"""decode_attn_dense_noalloc, the dense entry point for callers that cannot allocate device
memory where they call it (a framework that owns every allocation and hands an operator only its
inputs and outputs, a latency-critical loop where cudaMalloc may synchronise): it runs the same
kernel with its workspace in a library-owned device array, so its output must match the fp64
oracle, and decode_attn_dense called with a caller-allocated workspace.  Kept in a file of its own
that runs last."""
import ctypes

import pytest
import torch

from token_decode_attention_split_gb300 import binding as B_
from token_decode_attention_split_gb300 import workloads as W

from helpers import assert_close, oracle_for, out_f64

pytestmark = pytest.mark.gpu
DEV = "cuda"
FAKE = 0x10000


def noalloc_fn():
    lib = B_.load_library()
    fn = lib.decode_attn_dense_noalloc
    vp, i, i64, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    fn.argtypes = [vp, vp, vp, vp, i, i, i, i, i64, i64, f, vp]
    fn.restype = i
    return fn


def call_noalloc(fn, c, out, stream):
    return fn(c.q.data_ptr(), c.k.data_ptr(), c.v.data_ptr(), out.data_ptr(), c.B, c.Hq, c.Hkv,
              c.D, c.capacity, c.k_len, c.scale, stream.cuda_stream)


@pytest.mark.parametrize("grid_limit", [0, 3])
def test_noalloc_matches_oracle_and_workspace_entry_point(grid_limit):
    """Two calls in a row through the C ABI, each compared with the oracle and with
    decode_attn_dense; with a grid of 3 CTAs every head is merged from several partials, so the
    shared counters are exercised."""
    fn = noalloc_fn()
    B_.decode_attn_set_grid_limit(grid_limit)
    try:
        c = W.make_dense(2, 32, 4, 128, 3000, 2900, seed=77, device=DEV, k_scale=2.0,
                         poison_tail=True)
        ref = B_.run_case(c)
        want = oracle_for(c)
        stream = torch.cuda.current_stream()
        for _ in range(2):
            out = torch.full(c.out_shape(), float("nan"), dtype=torch.bfloat16, device=DEV)
            assert call_noalloc(fn, c, out, stream) == 0
            torch.cuda.synchronize()
            assert_close(out_f64(out), out_f64(ref), "noalloc vs workspace entry point")
            assert_close(out_f64(out), want, "noalloc vs oracle")
    finally:
        B_.decode_attn_set_grid_limit(0)


def test_noalloc_clears_what_an_earlier_call_left():
    """A call with few units leaves partial rows where a later call with many units keeps its
    merge counters; the later call still matches the oracle because each call clears its
    counters first."""
    fn = noalloc_fn()
    stream = torch.cuda.current_stream()
    B_.decode_attn_set_grid_limit(3)
    try:
        small = W.make_dense(1, 16, 1, 128, 2000, 1999, seed=78, device=DEV, k_scale=2.0)
        big = W.make_dense(16, 16, 8, 128, 800, 777, seed=79, device=DEV, k_scale=2.0)
        for c in (small, big, small, big):
            out = torch.full(c.out_shape(), float("nan"), dtype=torch.bfloat16, device=DEV)
            assert call_noalloc(fn, c, out, stream) == 0
            torch.cuda.synchronize()
            assert_close(out_f64(out), oracle_for(c), f"noalloc B={c.B} Hkv={c.Hkv}")
    finally:
        B_.decode_attn_set_grid_limit(0)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    fn = noalloc_fn()
    need = B_.decode_attn_workspace_size(0, 1024, 64, 64, 128)
    assert need > 4 * 1024 * 1024
    status = fn(FAKE, FAKE, FAKE, FAKE, 1024, 64, 64, 128, 16, 8, 0.1, None)
    assert status == 3    # DA_ERR_WORKSPACE_TOO_SMALL, nothing launched
    assert B_.decode_attn_read_device_error() == 0


def test_noalloc_argument_errors_enqueue_nothing():
    """The dense call's argument checks run before the scratch is touched: a length past the
    capacity and a capacity of 2^31 rows are refused with nothing launched."""
    fn = noalloc_fn()
    assert fn(FAKE, FAKE, FAKE, FAKE, 1, 8, 2, 128, 16, 17, 0.1, None) == 1
    assert fn(FAKE, FAKE, FAKE, FAKE, 1, 8, 2, 128, 1 << 31, 8, 0.1, None) == 2
    assert B_.decode_attn_read_device_error() == 0


def test_noalloc_binding_wrapper_matches_the_plain_call():
    c = W.make_dense(2, 16, 4, 128, 600, 555, seed=161, device=DEV, k_scale=2.0)
    ref = B_.run_case(c)
    out = B_.decode_attn_dense_noalloc(c.q, c.k, c.v, torch.empty_like(ref), c.k_len, c.scale)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
