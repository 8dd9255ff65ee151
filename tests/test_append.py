"""GPU KV append against the oracle, bit for bit (pure data movement): the paged reshape_and_cache
("DflashScratch", field slot_mapping_dev) and the ring write at pos % window ("AttnV41", method
decode_body); then append followed by decode attention."""
import numpy as np
import pytest
import torch

import oracle
from token_decode_attention_split_gb300 import binding as B_
from token_decode_attention_split_gb300 import workloads as W

from helpers import assert_close, bits, oracle_for, out_f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("T,Hkv,D,P,npages", [(300, 8, 128, 16, 400), (77, 2, 64, 8, 50),
                                               (1, 1, 128, 64, 3), (513, 4, 128, 32, 40)])
def test_append_paged_matches_oracle(T, Hkv, D, P, npages):
    c = W.make_append(T, Hkv, D, P, npages, seed=70 + T, device=DEV, pad_every=7)
    sm = c.slot_mapping.clone()
    sm[3 % T] = npages * P            # one past the pool: skipped
    sm[(5 * T) // 7] = -123           # any negative: skipped
    c.slot_mapping = sm
    kref, vref = oracle.append_paged(c.k_new, c.v_new, c.k_pool, c.v_pool, sm.cpu().numpy())
    B_.decode_attn_append_paged(c.k_new, c.v_new, c.k_pool, c.v_pool, c.slot_mapping)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bits(c.k_pool).view(np.uint16), kref)
    np.testing.assert_array_equal(bits(c.v_pool).view(np.uint16), vref)


def test_append_ring_matches_oracle():
    B, Hkv, D, R, window = 6, 2, 128, 300, 128
    s = W.make_sparse(B, 2 * Hkv, Hkv, D, R, 200, window, 0, seed=80, device=DEV)
    g = torch.Generator(device=DEV).manual_seed(81)
    k_new = torch.randn(B, Hkv, D, generator=g, device=DEV).to(torch.bfloat16)
    v_new = torch.randn(B, Hkv, D, generator=g, device=DEV).to(torch.bfloat16)
    pos = torch.tensor([0, 127, 128, 1000, -1, 5], dtype=torch.int64, device=DEV)
    kref, vref = oracle.append_ring(k_new, v_new, s.k_pool, s.v_pool, pos.cpu().numpy(), window)
    B_.decode_attn_append_ring(k_new, v_new, s.k_pool, s.v_pool, pos, window)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bits(s.k_pool).view(np.uint16), kref)
    np.testing.assert_array_equal(bits(s.v_pool).view(np.uint16), vref)


def test_append_then_paged_attention():
    """One new row per sequence at the slot after its last row, then decode_attn_paged with
    kv_len + 1 against the oracle on the appended pools."""
    c = W.make_paged(5, 32, 8, 128, 16, 600, 10, 900, seed=82, device=DEV, poison_unused=False)
    lens = c.kv_lens_host
    bt = c.block_table.cpu()
    slots = torch.tensor([int(bt[b, n // 16]) * 16 + n % 16 for b, n in enumerate(lens)],
                         dtype=torch.int64, device=DEV)
    g = torch.Generator(device=DEV).manual_seed(83)
    k_new = torch.randn(c.B, c.Hkv, c.D, generator=g, device=DEV).to(torch.bfloat16)
    v_new = torch.randn(c.B, c.Hkv, c.D, generator=g, device=DEV).to(torch.bfloat16)
    B_.decode_attn_append_paged(k_new, v_new, c.k_pool, c.v_pool, slots)
    c.kv_args.copy_(torch.tensor([n + 1 for n in lens], dtype=torch.int32, device=DEV))
    c.kv_lens_host = [n + 1 for n in lens]
    out = B_.run_case(c)
    assert_close(out_f64(out), oracle_for(c), "append then paged attention")


def test_append_named_workload_rows_land():
    """Full append_paged workload: every written slot holds its new row bit for bit, and a sample
    of untouched pages is unchanged."""
    c = W.make("append_paged", device=DEV)
    before = c.k_pool[:64].clone()
    B_.decode_attn_append_paged(c.k_new, c.v_new, c.k_pool, c.v_pool, c.slot_mapping)
    torch.cuda.synchronize()
    sm = c.slot_mapping
    page, off = sm // c.page_size, sm % c.page_size
    got_k = c.k_pool[page, :, off]            # [T, Hkv, D]
    got_v = c.v_pool[page, :, off]
    assert torch.equal(got_k, c.k_new) and torch.equal(got_v, c.v_new)
    touched = torch.zeros(64, dtype=torch.bool, device=DEV)
    touched[page[page < 64]] = True
    assert torch.equal(c.k_pool[:64][~touched], before[~touched])


def test_no_device_error_recorded():
    assert B_.decode_attn_read_device_error() == 0
