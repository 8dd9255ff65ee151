"""The seeded input recipe (CPU): the structure every workload promises — distinct pages per
sequence inside the pool, lengths within their range, poisoned rows exactly where nothing may be
read, the sparse selection's window / distinct indices / trailing pads, slot mappings of distinct
slots — and that a seed reproduces its inputs exactly."""
import numpy as np
import torch

from token_decode_attention_split_gb300 import workloads as W


def test_dense_poisoned_tail_and_shapes():
    c = W.make_dense(2, 8, 2, 64, 50, 37, seed=3, poison_tail=True, sq=3, causal=1)
    assert c.q.shape == (2, 8, 3, 64) and c.out_shape() == (2, 8, 3, 64)
    assert torch.isnan(c.k[:, :, 37:].float()).all() and torch.isnan(c.v[:, :, 37:].float()).all()
    assert torch.isfinite(c.k[:, :, :37].float()).all() and torch.isfinite(c.v[:, :, :37].float()).all()
    assert c.algorithmic_bytes() == 2 * 2 * 2 * 37 * 64 * 2 + 2 * 2 * 8 * 3 * 64 * 2


def test_dense_device_len_word():
    c = W.make_dense(1, 4, 1, 64, 20, 9, seed=4, device_len=True)
    assert c.k_len_dev is not None and int(c.k_len_dev[0]) == 9


def test_paged_block_table_and_lengths():
    c = W.make_paged(6, 8, 2, 64, 16, 200, 5, 300, seed=5, kv_len_stride=3)
    bt = c.block_table.numpy()
    lens = c.kv_lens_host
    assert all(5 <= n <= 300 for n in lens)
    used = []
    for b, n in enumerate(lens):
        pages = bt[b, : -(-n // 16)]
        assert ((pages >= 0) & (pages < 200)).all()
        used.extend(pages.tolist())
    assert len(used) == len(set(used))                      # distinct pages across sequences
    words = c.kv_args.numpy().view(np.uint32)
    assert [int(words[3 * b]) for b in range(6)] == lens    # stride-3 records, kv_len first
    # slots past each length and pages no sequence uses hold NaN
    kp = c.k_pool.float()
    for b, n in enumerate(lens):
        last = bt[b, (n - 1) // 16]
        if n % 16:
            assert torch.isnan(kp[last, :, n % 16:]).all()
    unused = sorted(set(range(200)) - set(bt.flatten().tolist()))
    assert torch.isnan(kp[unused]).all()


def test_sparse_selection_structure():
    c = W.make_sparse(4, 8, 1, 64, 3000, 700, 128, 200, seed=6)
    sel = c.sel.numpy()
    for b in range(4):
        row = sel[b]
        assert (row[:128] == np.arange(128)).all()          # ring-window slots first
        nv = c.n_valid_host[b]
        rnd = row[128:nv]
        assert ((rnd >= 128) & (rnd < 3000)).all() and len(set(rnd.tolist())) == len(rnd)
        assert (row[nv:] == -1).all() and 700 - nv <= 200   # trailing pads only
    assert c.algorithmic_bytes() == 2 * sum(c.n_valid_host) * 64 * 2 + 4 * 700 * 4 + 2 * 4 * 8 * 64 * 2


def test_append_slots_distinct_with_pads():
    c = W.make_append(256, 2, 64, 8, 100, seed=7, pad_every=5)
    s = c.slot_mapping.numpy()
    assert (s[::5] == -1).all()
    valid = s[s >= 0]
    assert len(valid) == len(set(valid.tolist())) and (valid < 800).all()


def test_seeds_reproduce_and_differ():
    a = W.make("dense_tiny")
    b = W.make("dense_tiny")
    c = W.make("dense_tiny", seed=W.CONFIGS["dense_tiny"]["seed"] + 1)
    for x, y in ((a.q, b.q), (a.k, b.k), (a.v, b.v)):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    assert not torch.equal(a.q.view(torch.int16), c.q.view(torch.int16))
