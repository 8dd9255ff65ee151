"""A seeded sweep of random shapes for every variant against the fp64 oracle, every output element
within 1e-2 + 1e-2 |ref|: GQA group sizes 1..64, head dims 64 and 128, ragged lengths, page sizes
8..256, both args-record strides, selection widths with pads, several query tokens with and
without causal masking, and forced split counts ("DecodeFlashSpec" q / k / v / k_len;
"DflashScratch" option_b_indirect_args_dev; "AttnV41" decode_fixed_topk, forward)."""
import numpy as np
import pytest
import torch

import oracle
from token_decode_attention_split_gb300 import binding as B_
from token_decode_attention_split_gb300 import workloads as W

from helpers import assert_close, oracle_for, out_f64

pytestmark = pytest.mark.gpu
DEV = "cuda"
GROUPS = [1, 2, 3, 4, 5, 6, 8, 12, 16, 24, 32, 40, 64]


@pytest.fixture(autouse=True)
def _reset_grid():
    B_.decode_attn_set_grid_limit(0)
    yield
    B_.decode_attn_set_grid_limit(0)


def dense_cases(n=12, seed=7001):
    r = np.random.default_rng(seed)
    out = []
    for i in range(n):
        G = int(r.choice(GROUPS))
        Hkv = int(r.choice([1, 2, 4])) if G > 16 else int(r.choice([1, 2, 4, 8]))
        D = int(r.choice([64, 128]))
        cap = int(r.integers(1, 900))
        k_len = int(r.integers(0, cap + 1))
        out.append((int(r.integers(1, 4)), G * Hkv, Hkv, D, cap, k_len, int(r.choice([0, 0, 1, 3, 7])),
                    seed + i))
    return out


@pytest.mark.parametrize("cfg", dense_cases(), ids=lambda c: "B{}_Hq{}_Hkv{}_D{}_cap{}_k{}_g{}".format(*c[:7]))
def test_random_dense(cfg):
    B, Hq, Hkv, D, cap, k_len, limit, seed = cfg
    B_.decode_attn_set_grid_limit(limit)
    c = W.make_dense(B, Hq, Hkv, D, cap, k_len, seed=seed, device=DEV, k_scale=2.0, poison_tail=True)
    assert_close(out_f64(B_.run_case(c)), oracle_for(c), f"dense {cfg}")


def paged_cases(n=12, seed=7101):
    r = np.random.default_rng(seed)
    out = []
    for i in range(n):
        G = int(r.choice(GROUPS))
        Hkv = int(r.choice([1, 2, 4, 8])) if G <= 8 else int(r.choice([1, 2]))
        D = int(r.choice([64, 128]))
        P = int(r.choice([8, 16, 32, 64, 128, 256]))
        B = int(r.integers(1, 6))
        hi = int(r.integers(1, 800))
        lo = int(r.integers(0, hi + 1))
        pages = B * (-(-hi // P)) + int(r.integers(0, 40))
        out.append((B, G * Hkv, Hkv, D, P, pages, lo, hi, int(r.choice([1, 3])), int(r.choice([0, 0, 2, 5])),
                    seed + i))
    return out


@pytest.mark.parametrize("cfg", paged_cases(), ids=lambda c: "B{}_Hq{}_Hkv{}_D{}_P{}_np{}_{}-{}_s{}_g{}".format(*c[:10]))
def test_random_paged(cfg):
    B, Hq, Hkv, D, P, pages, lo, hi, stride, limit, seed = cfg
    B_.decode_attn_set_grid_limit(limit)
    c = W.make_paged(B, Hq, Hkv, D, P, pages, lo, hi, seed=seed, device=DEV, kv_len_stride=stride)
    assert_close(out_f64(B_.run_case(c)), oracle_for(c), f"paged {cfg}")


def sparse_cases(n=10, seed=7201):
    r = np.random.default_rng(seed)
    out = []
    for i in range(n):
        G = int(r.choice(GROUPS))
        Hkv = int(r.choice([1, 2])) if G > 16 else int(r.choice([1, 2, 4]))
        D = int(r.choice([64, 128]))
        width = int(r.integers(1, 1600))
        window = int(r.integers(0, min(width, 128) + 1))
        pool = int(r.integers(max(width, 1) + 1, 5000))
        out.append((int(r.integers(1, 4)), G * Hkv, Hkv, D, pool, width, window,
                    int(r.integers(0, width // 2 + 1)), seed + i))
    return out


@pytest.mark.parametrize("cfg", sparse_cases(), ids=lambda c: "B{}_Hq{}_Hkv{}_D{}_R{}_W{}_win{}_pad{}".format(*c[:8]))
def test_random_sparse(cfg):
    B, Hq, Hkv, D, pool, width, window, pad, seed = cfg
    c = W.make_sparse(B, Hq, Hkv, D, pool, width, window, pad, seed=seed, device=DEV)
    assert_close(out_f64(B_.run_case(c)), oracle_for(c), f"sparse {cfg}")


def mq_cases(n=8, seed=7301):
    r = np.random.default_rng(seed)
    out = []
    for i in range(n):
        Sq = int(r.integers(2, 7))
        G = int(r.choice([g for g in GROUPS if g * Sq <= 64]))
        Hkv = int(r.choice([1, 2, 4, 8])) if G * Sq <= 16 else int(r.choice([1, 2]))
        out.append((int(r.integers(1, 4)), G * Hkv, Hkv, int(r.choice([64, 128])), Sq,
                    int(r.choice([0, 1])), int(r.choice([16, 32, 64])), seed + i))
    return out


@pytest.mark.parametrize("cfg", mq_cases(), ids=lambda c: "B{}_Hq{}_Hkv{}_D{}_Sq{}_causal{}_P{}".format(*c[:7]))
def test_random_multitoken(cfg):
    B, Hq, Hkv, D, Sq, causal, P, seed = cfg
    g = torch.Generator(device=DEV).manual_seed(seed)
    q = torch.randn(B, Hq, Sq, D, generator=g, device=DEV).to(torch.bfloat16)
    # dense
    cap = 300 + 37 * (seed % 5)
    k_len = cap - 11
    d = W.make_dense(B, Hq, Hkv, D, cap, k_len, seed=seed, device=DEV, poison_tail=True)
    ws = B_.new_workspace(B_.decode_attn_workspace_size(0, B, Hq * Sq, Hkv, D), DEV)
    out = torch.empty_like(q)
    B_.decode_attn_dense_mq(q, d.k, d.v, out, k_len, causal, d.scale, ws)
    torch.cuda.synchronize()
    ref = oracle.dense_mq(q, d.k.cpu(), d.v.cpu(), k_len, d.scale, causal=bool(causal))
    assert_close(out.double().cpu().numpy(), ref, f"dense mq {cfg}")
    # paged
    c = W.make_paged(B, Hq, Hkv, D, P, B * (-(-500 // P)) + 7, 1, 500, seed=seed + 50, device=DEV)
    ws = B_.new_workspace(B_.decode_attn_workspace_size(1, B, Hq * Sq, Hkv, D), DEV)
    out = torch.empty_like(q)
    B_.decode_attn_paged_mq(q, c.k_pool, c.v_pool, out, c.block_table, c.kv_args, 1, causal,
                            c.scale, ws)
    torch.cuda.synchronize()
    ref = oracle.paged_mq(q, c.k_pool.cpu(), c.v_pool.cpu(), c.block_table.cpu().numpy(),
                          c.kv_args.cpu().numpy().view(np.uint32), c.scale, causal=bool(causal))
    assert_close(out.double().cpu().numpy(), ref, f"paged mq {cfg}")


def test_no_device_error_recorded():
    assert B_.decode_attn_read_device_error() == 0
