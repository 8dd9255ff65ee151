"""Pins for the multi-token oracle (CPU): several query tokens per sequence, q [B, Hq, Sq, D]
("DecodeFlashSpec", q [B,Hq,Sq,D] and field causal; "AttnV41", method forward: m tokens at
start_pos).  Reading: the Sq new tokens are the last Sq rows of the live prefix, so causal
token i attends rows [0, len - Sq + i]."""
import math

import numpy as np
import torch

import oracle
from token_decode_attention_split_gb300 import workloads as W


def bits_of(x):
    return torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(
        torch.int16).numpy().view(np.uint16)


def mq_case(B, Hq, Hkv, D, cap, Sq, seed):
    d = W.make_dense(B, Hq, Hkv, D, cap, cap, seed=seed, k_scale=2.0)
    g = torch.Generator().manual_seed(seed + 1)
    q = torch.randn(B, Hq, Sq, D, generator=g).to(torch.bfloat16)
    return d, q


def test_closed_form_two_tokens():
    """D = 1, scale = ln 2, rows k = (0, 1, 2), v = (1, 2, 4), Sq = 2, q = 1 for both tokens.
    Token 0 (row 1 of the prefix) sees rows 0..1: weights (1, 2) -> (1 + 4)/3; token 1 sees rows
    0..2: weights (1, 2, 4) -> (1 + 4 + 16)/7.  Without causal masking both give 21/7."""
    q = bits_of(np.ones((1, 1, 2, 1)))
    k = bits_of(np.array([0, 1, 2, 9], np.float32).reshape(1, 1, 4, 1))
    v = bits_of(np.array([1, 2, 4, 100], np.float32).reshape(1, 1, 4, 1))
    got = oracle.dense_mq(q, k, v, 3, math.log(2.0), causal=True)
    np.testing.assert_allclose(got.reshape(-1), [5 / 3, 21 / 7], rtol=1e-12)
    got = oracle.dense_mq(q, k, v, 3, math.log(2.0), causal=False)
    np.testing.assert_allclose(got.reshape(-1), [3.0, 3.0], rtol=1e-12)


def test_causal_token_equals_single_query_at_its_length():
    d, q = mq_case(2, 8, 2, 16, 50, 4, seed=100)
    k_len = 37
    got = oracle.dense_mq(q, d.k, d.v, k_len, d.scale, causal=True)
    for i in range(4):
        ref = oracle.dense(q[:, :, i:i + 1], d.k, d.v, k_len - 4 + i + 1, d.scale)
        np.testing.assert_array_equal(got[:, :, i], ref)


def test_non_causal_token_equals_single_query_over_the_prefix():
    d, q = mq_case(2, 8, 2, 16, 50, 3, seed=101)
    got = oracle.dense_mq(q, d.k, d.v, 41, d.scale, causal=False)
    for i in range(3):
        np.testing.assert_array_equal(got[:, :, i],
                                      oracle.dense(q[:, :, i:i + 1], d.k, d.v, 41, d.scale))


def test_matches_sdpa_with_bottom_right_causal_mask():
    B, Hq, Hkv, D, cap, Sq, k_len = 2, 16, 4, 32, 90, 5, 77
    d, q = mq_case(B, Hq, Hkv, D, cap, Sq, seed=102)
    got = oracle.dense_mq(q, d.k, d.v, k_len, d.scale, causal=True)
    G = Hq // Hkv
    kf = d.k[:, :, :k_len].double().repeat_interleave(G, dim=1)
    vf = d.v[:, :, :k_len].double().repeat_interleave(G, dim=1)
    i = torch.arange(Sq)[:, None]
    j = torch.arange(k_len)[None, :]
    mask = j <= k_len - Sq + i                      # True = attend
    ref = torch.nn.functional.scaled_dot_product_attention(q.double(), kf, vf, attn_mask=mask,
                                                           scale=d.scale)
    np.testing.assert_allclose(got, ref.numpy(), rtol=1e-12, atol=1e-13)


def test_tokens_before_the_prefix_get_zero_rows():
    d, q = mq_case(1, 4, 1, 8, 10, 6, seed=103)
    got = oracle.dense_mq(q, d.k, d.v, 3, d.scale, causal=True)   # tokens 0..2 see no row
    assert np.all(got[:, :, :3] == 0.0) and np.all(np.isfinite(got[:, :, 3:]))
    assert np.any(got[:, :, 3:] != 0.0)


def test_paged_mq_equals_dense_mq_on_the_same_rows():
    B, Hq, Hkv, D, P, L, Sq = 2, 8, 2, 16, 4, 24, 3
    d, q = mq_case(B, Hq, Hkv, D, L, Sq, seed=104)
    max_pages, num_pages = 6, 20
    perm = np.random.default_rng(3).permutation(num_pages)[:B * max_pages].reshape(B, max_pages)
    perm = perm.astype(np.int32)
    kd = d.k.view(torch.int16).numpy().view(np.uint16)
    vd = d.v.view(torch.int16).numpy().view(np.uint16)
    kp = np.zeros((num_pages, Hkv, P, D), np.uint16)
    vp = np.zeros_like(kp)
    for b in range(B):
        for j in range(L):
            kp[perm[b, j // P], :, j % P] = kd[b, :, j]
            vp[perm[b, j // P], :, j % P] = vd[b, :, j]
    lens = [24, 11]
    got = oracle.paged_mq(q, kp, vp, perm, np.array(lens, np.uint32), d.scale, causal=True)
    for b, n in enumerate(lens):
        ref = oracle.dense_mq(q[b:b + 1], d.k[b:b + 1], d.v[b:b + 1], n, d.scale, causal=True)
        np.testing.assert_array_equal(got[b:b + 1], ref)


def test_single_token_reduces_to_decode():
    d, q = mq_case(2, 8, 2, 16, 30, 1, seed=105)
    np.testing.assert_array_equal(oracle.dense_mq(q, d.k, d.v, 29, d.scale)[:, :, 0],
                                  oracle.dense(q, d.k, d.v, 29, d.scale))
