"""GPU multi-token decode (Sq query tokens per sequence, causal inside the new tail) against the
fp64 oracle ("DecodeFlashSpec", q [B,Hq,Sq,D] and field causal; "AttnV41", method forward)."""
import numpy as np
import pytest
import torch

import oracle
from token_decode_attention_split_gb300 import binding as B_
from token_decode_attention_split_gb300 import workloads as W

from helpers import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(autouse=True)
def _reset_grid():
    B_.decode_attn_set_grid_limit(0)
    yield
    B_.decode_attn_set_grid_limit(0)


def queries(B, Hq, Sq, D, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    return torch.randn(B, Hq, Sq, D, generator=g, device=DEV).to(torch.bfloat16)


def f64(t):
    return t.double().cpu().numpy()


@pytest.mark.parametrize("B,Hq,Hkv,D,cap,k_len,Sq,causal,limit", [
    (2, 32, 8, 128, 800, 777, 4, True, 0),
    (2, 32, 8, 128, 800, 777, 4, False, 0),
    (1, 16, 2, 128, 700, 640, 8, True, 0),      # G = 8, 64 query columns per unit
    (3, 8, 8, 64, 300, 200, 2, True, 0),        # G = 1
    (2, 16, 4, 128, 1200, 1100, 3, True, 5),    # several segments merged across CTAs
    (1, 8, 2, 128, 64, 5, 8, True, 0),          # tokens before the prefix: zero rows
])
def test_dense_multitoken_matches_oracle(B, Hq, Hkv, D, cap, k_len, Sq, causal, limit):
    B_.decode_attn_set_grid_limit(limit)
    d = W.make_dense(B, Hq, Hkv, D, cap, k_len, seed=120 + Sq, device=DEV, k_scale=2.0,
                     poison_tail=True)
    q = queries(B, Hq, Sq, D, 121 + Sq)
    ws = B_.new_workspace(B_.decode_attn_workspace_size(0, B, Hq * Sq, Hkv, D), DEV)
    out = torch.empty_like(q)
    B_.decode_attn_dense_mq(q, d.k, d.v, out, k_len, causal, d.scale, ws)
    torch.cuda.synchronize()
    ref = oracle.dense_mq(q, d.k.cpu(), d.v.cpu(), k_len, d.scale, causal=causal)
    assert_close(f64(out), ref, f"dense Sq={Sq} causal={causal}")


@pytest.mark.parametrize("B,Hq,Hkv,D,P,npages,Sq,causal", [
    (4, 32, 8, 128, 16, 400, 4, True),          # four KV heads per unit
    (3, 16, 2, 128, 64, 120, 2, True),          # one KV head per unit, 64-row pages
    (3, 32, 8, 128, 16, 400, 2, False),
    (3, 16, 8, 128, 16, 400, 2, True),          # G = 2: each warp holds one KV head's columns
])
def test_paged_multitoken_matches_oracle(B, Hq, Hkv, D, P, npages, Sq, causal):
    c = W.make_paged(B, Hq, Hkv, D, P, npages, 1, 600, seed=130 + P, device=DEV)
    q = queries(B, Hq, Sq, D, 131)
    ws = B_.new_workspace(B_.decode_attn_workspace_size(1, B, Hq * Sq, Hkv, D), DEV)
    out = torch.empty_like(q)
    B_.decode_attn_paged_mq(q, c.k_pool, c.v_pool, out, c.block_table, c.kv_args, 1, causal,
                            c.scale, ws)
    torch.cuda.synchronize()
    ref = oracle.paged_mq(q, c.k_pool.cpu(), c.v_pool.cpu(), c.block_table.cpu().numpy(),
                          c.kv_args.cpu().numpy().view(np.uint32), c.scale, causal=causal)
    assert_close(f64(out), ref, f"paged Sq={Sq} causal={causal}")


def test_single_token_multitoken_call_equals_decode_bitwise():
    d = W.make_dense(2, 32, 8, 128, 600, 555, seed=140, device=DEV)
    ws = B_.new_workspace(B_.decode_attn_workspace_size(0, 2, 32, 8, 128), DEV)
    a = torch.empty(d.out_shape(), dtype=torch.bfloat16, device=DEV)
    b = torch.empty_like(a)
    B_.decode_attn_dense(d.q, d.k, d.v, a, d.k_len, d.scale, ws)
    B_.decode_attn_dense_mq(d.q, d.k, d.v, b, d.k_len, True, d.scale, ws)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_no_device_error_recorded():
    assert B_.decode_attn_read_device_error() == 0


def test_named_verify_workload():
    """dense_verify4 at full size (4 query tokens, causal): every sequence against the oracle."""
    c = W.make("dense_verify4", device=DEV)
    out = B_.run_case(c)
    torch.cuda.synchronize()
    assert out.shape == (c.B, c.Hq, 4, c.D) and torch.isfinite(out.float()).all()
    ref = oracle.dense_mq(c.q.cpu(), c.k.cpu(), c.v.cpu(), c.k_len, c.scale, causal=True)
    assert_close(f64(out), ref, "dense_verify4")
