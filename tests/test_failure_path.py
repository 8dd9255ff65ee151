"""The kernels' failure path on the GPU, without a fault: a bounded wait that nothing completes
gives up after its limit, records a code in the device error word and returns, and the context
stays usable for the next decode call (packed_fused_kda_decode's fail-closed convention carried
to the device)."""
import time

import pytest
import torch

from token_decode_attention_split_gb300 import binding as B_
from token_decode_attention_split_gb300 import workloads as W

from helpers import assert_close, oracle_for, out_f64

pytestmark = pytest.mark.gpu
DEV = "cuda"
WAIT_CHECK_CODE = 5


def test_timed_out_wait_is_reported_and_the_context_stays_usable():
    assert B_.decode_attn_read_device_error() == 0          # nothing left from earlier tests
    t0 = time.perf_counter()
    B_.decode_attn_check_wait_timeout(2000)                  # 2 ms limit
    assert B_.decode_attn_read_device_error() == WAIT_CHECK_CODE
    assert time.perf_counter() - t0 < 5.0                    # gave up, did not hang
    assert B_.decode_attn_read_device_error() == 0          # reading cleared it
    c = W.make_dense(2, 16, 4, 128, 300, 257, seed=150, device=DEV)
    out = B_.run_case(c)
    torch.cuda.synchronize()
    assert_close(out_f64(out), oracle_for(c), "decode after a timed-out wait")
    assert B_.decode_attn_read_device_error() == 0


def test_first_code_is_kept_until_read():
    B_.decode_attn_check_wait_timeout(1000)
    B_.decode_attn_check_wait_timeout(1000)
    assert B_.decode_attn_read_device_error() == WAIT_CHECK_CODE
    assert B_.decode_attn_read_device_error() == 0
