"""Pins for the fp64 oracle against facts fixed by the pages and by mathematics (CPU only).

Each pin is chosen to fail on a plausible slip inside the oracle:
  * closed-form cases (tests/golden/closed_form_cases.json): exact rationals, catching a wrong
    sign in the exponent, a transposed operand (q.v instead of q.k), an off-by-one on k_len, the
    wrong GQA grouping, the wrong word of the args record, pads or duplicates mishandled;
  * k_len = 1 returns V row 0; identical keys return the mean of the V prefix;
  * permuting a selection leaves the result unchanged; trailing -1 pads are exactly neutral
    ("AttnV41", method decode_fixed_topk);
  * paged over scattered pages and sparse over [0, k_len) equal dense on the same rows exactly;
  * torch's scaled_dot_product_attention in float64 (a library routine the C oracle never calls)
    agrees to 1e-12 on seeded cases;
  * splitting the rows and merging by log-sum-exp reproduces the unsplit result.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from token_decode_attention_split_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_bits(x) -> np.ndarray:
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def widen(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float64).cpu().numpy()


def load_cases():
    with open(os.path.join(GOLDEN, "closed_form_cases.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", load_cases(), ids=lambda c: c["name"])
def test_closed_form_cases(case):
    scale = math.log(2.0)
    q = bf16_bits(case["q"]).reshape(case["B"], case["Hq"], 1, case["D"])
    if case["variant"] == "dense":
        k = bf16_bits(case["k"]).reshape(case["B"], case["Hkv"], case["capacity"], case["D"])
        v = bf16_bits(case["v"]).reshape(k.shape)
        got = oracle.dense(q, k, v, case["k_len"], scale)
    elif case["variant"] == "paged":
        shape = (case["num_pages"], case["Hkv"], case["page_size"], case["D"])
        k = bf16_bits(case["k_pool"]).reshape(shape)
        v = bf16_bits(case["v_pool"]).reshape(shape)
        got = oracle.paged(q, k, v, np.array(case["block_table"], np.int32),
                           np.array(case["kv_args"], np.uint32), scale,
                           kv_len_stride=case["kv_len_stride"])
    else:
        shape = (case["B"], case["Hkv"], case["pool_rows"], case["D"])
        k = bf16_bits(case["k_pool"]).reshape(shape)
        v = bf16_bits(case["v_pool"]).reshape(shape)
        got = oracle.sparse(q, k, v, np.array(case["sel"], np.int32), scale)
    exp = np.array([[float(Fraction(n, d)) for n, d in np.array(row).reshape(-1, 2)]
                    for row in case["expected"]]).reshape(got.shape)
    np.testing.assert_allclose(got, exp, rtol=1e-12, atol=1e-12)


def test_indirect_args_record_layout():
    """The args record is [kv_len, q_offset, q_rope_pos] u32 (DflashScratch,
    option_b_indirect_args_dev): with stride 3 the oracle reads word 0 as kv_len and ignores the
    other two, so scribbling over words 1 and 2 changes nothing."""
    with open(os.path.join(GOLDEN, "indirect_args_record.json")) as f:
        rec = json.load(f)
    stride = rec["record_bytes"] // rec["word_bytes"]
    assert stride == 3 and rec["words"][rec["kv_len_word"]] == "kv_len"
    c = W.make_paged(B=3, Hq=4, Hkv=2, D=8, page_size=4, num_pages=64, kv_min=1, kv_max=30,
                     seed=5, kv_len_stride=stride)
    ref = oracle.paged(c.q, c.k_pool, c.v_pool, c.block_table.numpy(),
                       c.kv_args.numpy().view(np.uint32), c.scale, kv_len_stride=stride)
    args = c.kv_args.numpy().view(np.uint32).reshape(-1, stride).copy()
    assert list(args[:, rec["kv_len_word"]]) == c.kv_lens_host
    args[:, 1] = 12345
    args[:, 2] = 777
    got = oracle.paged(c.q, c.k_pool, c.v_pool, c.block_table.numpy(), args.reshape(-1), c.scale,
                       kv_len_stride=stride)
    np.testing.assert_array_equal(got, ref)
    one = oracle.paged(c.q, c.k_pool, c.v_pool, c.block_table.numpy(), args[:, 0].copy(),
                       c.scale, kv_len_stride=1)
    np.testing.assert_array_equal(one, ref)


def test_klen_one_returns_v0():
    c = W.make_dense(B=2, Hq=8, Hkv=2, D=16, capacity=9, k_len=1, seed=11, k_scale=3.0)
    out = oracle.dense(c.q, c.k, c.v, 1, c.scale)
    v0 = widen(c.v[:, :, 0, :])                       # [B, Hkv, D]
    exp = np.repeat(v0, 4, axis=1)                    # G = 4, contiguous groups
    np.testing.assert_array_equal(out, exp)


def test_identical_keys_return_mean_of_v():
    c = W.make_dense(B=2, Hq=4, Hkv=2, D=8, capacity=40, k_len=33, seed=12)
    c.k[:] = c.k[:, :, :1, :]                        # every row equals row 0
    out = oracle.dense(c.q, c.k, c.v, c.k_len, c.scale)
    mean = widen(c.v[:, :, :c.k_len, :]).mean(axis=2)
    np.testing.assert_allclose(out, np.repeat(mean, 2, axis=1), rtol=1e-13, atol=1e-14)


def test_sparse_permutation_invariance():
    c = W.make_sparse(B=3, Hq=8, Hkv=2, D=16, pool_rows=300, width=64, window=8, max_pad=20,
                      seed=13)
    ref = oracle.sparse(c.q, c.k_pool, c.v_pool, c.sel.numpy(), c.scale)
    rng = np.random.default_rng(0)
    sel = c.sel.numpy().copy()
    for b in range(c.B):
        sel[b] = sel[b][rng.permutation(sel.shape[1])]   # pads move into the middle too
    got = oracle.sparse(c.q, c.k_pool, c.v_pool, sel, c.scale)
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-14)
    assert not np.array_equal(sel, c.sel.numpy())


def test_sparse_trailing_pads_exactly_neutral():
    c = W.make_sparse(B=2, Hq=4, Hkv=1, D=16, pool_rows=200, width=50, window=4, max_pad=0,
                      seed=14)
    ref = oracle.sparse(c.q, c.k_pool, c.v_pool, c.sel.numpy(), c.scale)
    padded = np.concatenate([c.sel.numpy(), np.full((c.B, 37), -1, np.int32)], axis=1)
    got = oracle.sparse(c.q, c.k_pool, c.v_pool, padded, c.scale)
    np.testing.assert_array_equal(got, ref)


def test_paged_equals_dense_on_the_same_rows():
    B, Hq, Hkv, D, P = 3, 8, 2, 16, 4
    lens = [1, 13, 24]
    d = W.make_dense(B=B, Hq=Hq, Hkv=Hkv, D=D, capacity=24, k_len=24, seed=15)
    max_pages = 6
    num_pages = 40
    rng = np.random.default_rng(1)
    perm = rng.permutation(num_pages)[:B * max_pages].reshape(B, max_pages).astype(np.int32)
    kp = np.zeros((num_pages, Hkv, P, D), np.uint16)
    vp = np.zeros_like(kp)
    kd = d.k.view(torch.int16).numpy().view(np.uint16)
    vd = d.v.view(torch.int16).numpy().view(np.uint16)
    for b in range(B):
        for j in range(24):
            kp[perm[b, j // P], :, j % P, :] = kd[b, :, j, :]
            vp[perm[b, j // P], :, j % P, :] = vd[b, :, j, :]
    got = oracle.paged(d.q, kp, vp, perm, np.array(lens, np.uint32), d.scale)
    for b, n in enumerate(lens):
        ref = oracle.dense(d.q[b:b + 1], d.k[b:b + 1], d.v[b:b + 1], n, d.scale)
        np.testing.assert_array_equal(got[b:b + 1], ref)


def test_sparse_over_prefix_equals_dense():
    d = W.make_dense(B=2, Hq=4, Hkv=2, D=32, capacity=50, k_len=37, seed=16)
    sel = np.tile(np.arange(37, dtype=np.int32), (2, 1))
    got = oracle.sparse(d.q, d.k, d.v, sel, d.scale)
    ref = oracle.dense(d.q, d.k, d.v, 37, d.scale)
    np.testing.assert_array_equal(got, ref)


def _sdpa_ref(q, k, v, k_len, scale):
    qf = q.to(torch.float64)                                  # [B, Hq, 1, D]
    G = q.shape[1] // k.shape[1]
    kf = k[:, :, :k_len].to(torch.float64).repeat_interleave(G, dim=1)
    vf = v[:, :, :k_len].to(torch.float64).repeat_interleave(G, dim=1)
    return torch.nn.functional.scaled_dot_product_attention(qf, kf, vf, scale=scale)[:, :, 0]


@pytest.mark.parametrize("name,over", [
    ("dense_tiny", {}),
    ("dense_batched", dict(B=2, capacity=640, k_len=517)),
    ("dense_long", dict(B=1, Hq=16, Hkv=2, capacity=1500, k_len=1499)),
])
def test_matches_torch_sdpa_float64(name, over):
    c = W.make(name, **over)
    out = oracle.dense(c.q, c.k, c.v, c.k_len, c.scale)
    ref = _sdpa_ref(c.q, c.k, c.v, c.k_len, c.scale).numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)


def test_lse_merge_identity():
    """Any partition of [0, k_len) merged by log-sum-exp equals the unsplit row: the identity a
    split-KV computation relies on."""
    c = W.make_dense(B=2, Hq=4, Hkv=2, D=16, capacity=300, k_len=257, seed=17, k_scale=2.0)
    full = oracle.dense(c.q, c.k, c.v, c.k_len, c.scale)
    for b, h in [(0, 0), (1, 3)]:
        for cuts in ([0, 257], [0, 1, 257], [0, 64, 128, 200, 257], [0, 37, 37, 100, 257]):
            parts = [oracle.dense_range(c.q, c.k, c.v, b, h, a, z, c.scale)
                     for a, z in zip(cuts[:-1], cuts[1:])]
            lses = np.array([p[1] for p in parts])
            M = np.max(lses)
            w = np.exp(lses - M)                   # exp(-inf) = 0 for an empty part
            merged = sum(wi * p[0] for wi, p in zip(w, parts)) / w.sum()
            np.testing.assert_allclose(merged, full[b, h], rtol=1e-12, atol=1e-13)


def test_empty_sets_give_zero_rows():
    d = W.make_dense(B=1, Hq=2, Hkv=1, D=8, capacity=4, k_len=4, seed=18)
    assert np.all(oracle.dense(d.q, d.k, d.v, 0, d.scale) == 0.0)
    s = W.make_sparse(B=2, Hq=2, Hkv=1, D=8, pool_rows=16, width=6, window=2, max_pad=0, seed=19)
    sel = s.sel.numpy().copy()
    sel[1] = -1
    out = oracle.sparse(s.q, s.k_pool, s.v_pool, sel, s.scale)
    assert np.all(out[1] == 0.0) and np.all(np.isfinite(out[0])) and np.any(out[0] != 0)


def test_paged_clamp_and_out_of_range_pages():
    c = W.make_paged(B=2, Hq=4, Hkv=2, D=8, page_size=4, num_pages=32, kv_min=8, kv_max=16,
                     seed=20, max_pages=4, poison_unused=False)
    bt = c.block_table.numpy().copy()
    lens = np.array([100, 16], np.uint32)                 # 100 clamps to 4 pages * 4 = 16
    ref = oracle.paged(c.q, c.k_pool, c.v_pool, bt, np.array([16, 16], np.uint32), c.scale)
    got = oracle.paged(c.q, c.k_pool, c.v_pool, bt, lens, c.scale)
    np.testing.assert_array_equal(got, ref)
    # an out-of-range page id drops exactly that page's rows: compare with a sparse selection
    # of the same rows laid out densely
    bt2 = bt.copy()
    bt2[1, 2] = 999
    bt2[1, 0] = -5
    got2 = oracle.paged(c.q, c.k_pool, c.v_pool, bt2, np.array([16, 16], np.uint32), c.scale)
    kept = [j for j in range(16) if j // 4 not in (0, 2)]
    kd = np.stack([c.k_pool.view(torch.int16).numpy().view(np.uint16)[bt[1, j // 4], :, j % 4]
                   for j in kept], axis=1)[None]           # [1, Hkv, rows, D]
    vd = np.stack([c.v_pool.view(torch.int16).numpy().view(np.uint16)[bt[1, j // 4], :, j % 4]
                   for j in kept], axis=1)[None]
    ref2 = oracle.dense(c.q[1:2], kd, vd, len(kept), c.scale)
    np.testing.assert_array_equal(got2[1:2], ref2)
    np.testing.assert_array_equal(got2[0:1], ref[0:1])


def test_pairs_subset_matches_full():
    c = W.make_dense(B=2, Hq=8, Hkv=2, D=16, capacity=70, k_len=65, seed=21)
    full = oracle.dense(c.q, c.k, c.v, c.k_len, c.scale)
    pairs = [0, 5, 9, 15]
    part = oracle.dense(c.q, c.k, c.v, c.k_len, c.scale, pairs=pairs)
    flat_f, flat_p = full.reshape(16, -1), part.reshape(16, -1)
    np.testing.assert_array_equal(flat_p[pairs], flat_f[pairs])
    assert np.all(np.isnan(np.delete(flat_p, pairs, axis=0)))


def test_rejects_bad_arguments():
    c = W.make_dense(B=1, Hq=4, Hkv=2, D=8, capacity=4, k_len=4, seed=22)
    with pytest.raises(ValueError):
        oracle.dense(c.q, c.k, c.v, 5, c.scale)            # k_len > capacity
    with pytest.raises(ValueError):
        oracle.dense(c.q, c.k, c.v, 2, c.scale, pairs=[8])  # pair index out of range


def test_sparse_every_negative_index_is_skipped():
    """Any negative entry (not only -1) and any entry >= pool_rows is skipped.  On the second
    sequence a wrongly kept -2 or -1000 would read rows of the first sequence's pool (set to large
    values here), so the result would change."""
    B, Hq, Hkv, D, R = 2, 4, 1, 8, 16
    g = torch.Generator().manual_seed(55)
    q = torch.randn(B, Hq, 1, D, generator=g).to(torch.bfloat16)
    k = torch.randn(B, Hkv, R, D, generator=g).to(torch.bfloat16)
    v = torch.randn(B, Hkv, R, D, generator=g).to(torch.bfloat16)
    k[0] = 40.0
    v[0] = 1000.0
    clean = torch.tensor([[0, 3, 5, -1, -1], [2, 7, 11, -1, -1]], dtype=torch.int32)
    dirty = torch.tensor([[0, -2, 3, 5, -1000], [2, -2, 7, -1000, 11]], dtype=torch.int32)
    over = torch.tensor([[0, 3, 5, 16, 99], [2, 7, 11, 16, 2 ** 30]], dtype=torch.int32)
    ref = oracle.sparse(q, k, v, clean.numpy(), 0.3)
    np.testing.assert_array_equal(oracle.sparse(q, k, v, dirty.numpy(), 0.3), ref)
    np.testing.assert_array_equal(oracle.sparse(q, k, v, over.numpy(), 0.3), ref)
