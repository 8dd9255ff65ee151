"""Pins for the KV-append oracle (CPU): the paged reshape_and_cache through an i64 slot mapping
("DflashScratch", field slot_mapping_dev) and the ring write at pos % window ("AttnV41", method
decode_body)."""
import numpy as np
import torch

import oracle
from token_decode_attention_split_gb300 import workloads as W


def bits_of(x):
    return torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(
        torch.int16).numpy().view(np.uint16)


def test_paged_slots_by_hand():
    """Two pages of 2 slots, 2 KV heads, D = 1: slots 3, 0, -1 (padding) and 4 (past the pool)."""
    k_new = bits_of([[[10], [11]], [[20], [21]], [[30], [31]], [[40], [41]]])   # [T=4, Hkv=2, D=1]
    v_new = bits_of([[[-10], [-11]], [[-20], [-21]], [[-30], [-31]], [[-40], [-41]]])
    pool = bits_of(np.zeros((2, 2, 2, 1)))                                       # [pages, Hkv, P, D]
    kp, vp = oracle.append_paged(k_new, v_new, pool, pool, [3, 0, -1, 4])
    got = torch.from_numpy(kp.view(np.int16)).view(torch.bfloat16).float().numpy()
    exp = np.zeros((2, 2, 2, 1))
    exp[1, 0, 1, 0], exp[1, 1, 1, 0] = 10, 11     # slot 3 = page 1, position 1
    exp[0, 0, 0, 0], exp[0, 1, 0, 0] = 20, 21     # slot 0 = page 0, position 0
    np.testing.assert_array_equal(got, exp)
    gotv = torch.from_numpy(vp.view(np.int16)).view(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(gotv, -exp)


def test_paged_duplicate_slots_later_row_wins():
    k_new = bits_of([[[1.0]], [[2.0]], [[3.0]]])
    pool = bits_of(np.zeros((1, 1, 4, 1)))
    kp, _ = oracle.append_paged(k_new, k_new, pool, pool, [2, 2, 1])
    got = torch.from_numpy(kp.view(np.int16)).view(torch.bfloat16).float().numpy()[0, 0, :, 0]
    np.testing.assert_array_equal(got, [0, 3, 2, 0])


def test_ring_wraps_at_window_and_skips_negative():
    B, Hkv, R, D, window = 3, 2, 6, 4, 4
    k_new = bits_of(np.arange(B * Hkv * D).reshape(B, Hkv, D) + 1)
    pool = bits_of(np.full((B, Hkv, R, D), -7.0))
    kp, vp = oracle.append_ring(k_new, k_new, pool, pool, [5, -1, 3], window)
    got = torch.from_numpy(kp.view(np.int16)).view(torch.bfloat16).float().numpy()
    exp = np.full((B, Hkv, R, D), -7.0)
    src = np.arange(B * Hkv * D).reshape(B, Hkv, D) + 1.0
    exp[0, :, 5 % window] = src[0]                 # position 5 -> ring row 1
    exp[2, :, 3] = src[2]                          # position 3 -> ring row 3; sequence 1 skipped
    np.testing.assert_array_equal(got, exp)


def test_append_then_attend_equals_attention_over_the_longer_prefix():
    """Append one new row per sequence at slot (page of position L, L % P), then paged attention
    with kv_len L + 1 equals dense attention over the old L rows plus the new row."""
    B, Hq, Hkv, D, P = 3, 8, 2, 16, 4
    lens = [5, 8, 1]
    c = W.make_paged(B, Hq, Hkv, D, P, 40, 1, 12, seed=61, kv_lens=lens, max_pages=4,
                     poison_unused=False)
    g = torch.Generator().manual_seed(62)
    k_new = torch.randn(B, Hkv, D, generator=g).to(torch.bfloat16)
    v_new = torch.randn(B, Hkv, D, generator=g).to(torch.bfloat16)
    bt = c.block_table.numpy()
    slots = [int(bt[b, n // P]) * P + n % P for b, n in enumerate(lens)]
    kp, vp = oracle.append_paged(k_new, v_new, c.k_pool, c.v_pool, slots)
    got = oracle.paged(c.q, kp, vp, bt, np.array([n + 1 for n in lens], np.uint32), c.scale)
    kpool = c.k_pool.view(torch.int16).numpy().view(np.uint16)
    vpool = c.v_pool.view(torch.int16).numpy().view(np.uint16)
    for b, n in enumerate(lens):
        kd = np.stack([kpool[bt[b, j // P], :, j % P] for j in range(n)] +
                      [k_new[b].view(torch.int16).numpy().view(np.uint16)], axis=1)[None]
        vd = np.stack([vpool[bt[b, j // P], :, j % P] for j in range(n)] +
                      [v_new[b].view(torch.int16).numpy().view(np.uint16)], axis=1)[None]
        ref = oracle.dense(c.q[b:b + 1], kd, vd, n + 1, c.scale)
        np.testing.assert_array_equal(got[b:b + 1], ref)


def test_ring_append_then_sparse_attention_sees_the_new_row():
    """A ring write at position p followed by sparse attention over a selection that names ring
    row p % window returns exactly the new V row when that is the only entry."""
    B, Hq, Hkv, D, R, window = 2, 4, 1, 8, 32, 8
    s = W.make_sparse(B, Hq, Hkv, D, R, 16, window, 0, seed=63)
    g = torch.Generator().manual_seed(64)
    k_new = torch.randn(B, Hkv, D, generator=g).to(torch.bfloat16)
    v_new = torch.randn(B, Hkv, D, generator=g).to(torch.bfloat16)
    pos = [19, 6]
    kp, vp = oracle.append_ring(k_new, v_new, s.k_pool, s.v_pool, pos, window)
    sel = np.full((B, 16), -1, np.int32)
    sel[0, 0], sel[1, 5] = 19 % window, 6
    out = oracle.sparse(s.q, kp, vp, sel, s.scale)
    for b in range(B):
        np.testing.assert_array_equal(out[b], np.repeat(v_new[b].double().numpy(), Hq // Hkv, 0))


def test_paged_slot_past_the_pool_writes_nothing():
    """A slot at or past num_pages * page_size is skipped: the pool is the first 2 pages of a
    3-page buffer, and the guard page after it must stay untouched."""
    k_new = bits_of([[[7.0]], [[8.0]], [[9.0]]])                   # [T=3, Hkv=1, D=1]
    buf_k = bits_of(np.full((3, 1, 2, 1), 5.0))
    buf_v = bits_of(np.full((3, 1, 2, 1), 5.0))
    kp, vp = buf_k[:2], buf_v[:2]                                  # C-contiguous views, 2 pages
    oracle.append_paged(k_new, k_new, kp, vp, [1, 4, 5], inplace=True)
    guard = np.full((1, 2, 1), 5.0)
    for buf in (buf_k, buf_v):
        vals = torch.from_numpy(buf.view(np.int16)).view(torch.bfloat16).float().numpy()
        np.testing.assert_array_equal(vals[2], guard)             # slots 4, 5: page 2 untouched
        assert vals[0, 0, 1, 0] == 7.0 and vals[0, 0, 0, 0] == 5.0 and (vals[1] == 5.0).all()
