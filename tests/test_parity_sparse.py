"""GPU sparse decode attention against the fp64 oracle, and exact -1-pad invariance
("AttnV41", decode_fixed_topk: a -1 entry adds an exact zero to the denominator and nothing to
the output, so the padded result equals the unpadded one bit for bit)."""
import numpy as np
import pytest
import torch

from token_decode_attention_split_gb300 import binding as B_
from token_decode_attention_split_gb300 import workloads as W

from helpers import assert_close, oracle_for, out_f64

pytestmark = pytest.mark.gpu
DEV = "cuda"

CASES = [
    # B, Hq, Hkv, D, pool_rows, width, window, max_pad
    (3, 64, 1, 128, 3000, 700, 32, 200),
    (2, 8, 8, 64, 500, 63, 4, 10),          # G = 1, a single partial tile
    (4, 32, 8, 128, 2000, 257, 16, 1),      # G = 4, chunk boundary + 1
    (2, 64, 8, 128, 1500, 1000, 64, 300),   # G = 8
    (2, 16, 1, 128, 900, 256, 8, 0),        # G = 16, exactly one chunk
    (2, 32, 1, 64, 800, 513, 8, 100),       # G = 32
    (1, 48, 1, 128, 5000, 2048, 128, 512),  # G = 48: head groups of 32 and 16, two chunks
    (2, 64, 1, 128, 9000, 5000, 128, 300),  # G = 64: two head groups, five chunks
    (2, 16, 2, 64, 3000, 1100, 32, 50),     # G = 16: three chunks
]


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: "B{}_Hq{}_Hkv{}_D{}_R{}_W{}".format(*c[:6]))
def test_sparse_matches_oracle(cfg):
    B, Hq, Hkv, D, R, width, window, max_pad = cfg
    c = W.make_sparse(B, Hq, Hkv, D, R, width, window, max_pad, seed=300 + width, device=DEV,
                      poison_unselected=True)
    out = B_.run_case(c)
    assert_close(out_f64(out), oracle_for(c), f"sparse {cfg}")


def test_sparse_duplicates_interior_pads_and_bad_indices():
    c = W.make_sparse(2, 16, 2, 128, 600, 300, 8, 0, seed=41, device=DEV)
    sel = c.sel.clone()
    sel[0, 10:20] = sel[0, 0]            # duplicates count once per entry
    sel[0, 50:60] = -1                   # interior pads
    sel[1, 5] = 600                      # == pool_rows: skipped
    sel[1, 7] = -9                       # any negative: skipped
    sel[1, 100:] = -1
    c.sel = sel
    out = B_.run_case(c)
    assert_close(out_f64(out), oracle_for(c), "duplicates / pads / bad indices")


def test_sparse_all_pad_rows_are_zero():
    c = W.make_sparse(3, 8, 1, 128, 1000, 400, 4, 0, seed=42, device=DEV)
    c.sel[1] = -1
    out = B_.run_case(c)
    got = out_f64(out)
    assert np.all(got[1] == 0.0)
    assert_close(got, oracle_for(c), "all-pad row")


def test_single_valid_entry_returns_that_row():
    c = W.make_sparse(2, 64, 1, 128, 1000, 700, 1, 0, seed=43, device=DEV)
    c.sel[:] = -1
    c.sel[0, 613] = 777
    c.sel[1, 0] = 5
    out = B_.run_case(c)
    assert torch.equal(out[0, :, 0], c.v_pool[0, 0, 777].expand(64, -1))
    assert torch.equal(out[1, :, 0], c.v_pool[1, 0, 5].expand(64, -1))


@pytest.mark.parametrize("G,Hkv,D", [(64, 1, 128), (8, 2, 128), (4, 4, 64), (16, 1, 128)])
def test_pads_are_bit_exactly_neutral(G, Hkv, D):
    """Per sequence: the padded fixed-width call and the call with the pads removed give the
    same bits; batched: appending more -1 pads changes no bit."""
    c = W.make_sparse(4, G * Hkv, Hkv, D, 4000, 1500, 64, 700, seed=44 + G, device=DEV)
    full = B_.run_case(c)
    for b in range(c.B):
        n = c.n_valid_host[b]
        sub = W.SparseCase(c.q[b:b + 1], c.k_pool[b:b + 1], c.v_pool[b:b + 1],
                           c.sel[b:b + 1, :n].contiguous(), c.scale, 1, c.Hq, c.Hkv, c.D,
                           c.pool_rows, [n])
        assert torch.equal(B_.run_case(sub), full[b:b + 1]), f"sequence {b}"
    more = torch.cat([c.sel, torch.full((c.B, 999), -1, dtype=torch.int32, device=DEV)], dim=1)
    wide = W.SparseCase(c.q, c.k_pool, c.v_pool, more.contiguous(), c.scale, c.B, c.Hq, c.Hkv,
                        c.D, c.pool_rows, c.n_valid_host)
    assert torch.equal(B_.run_case(wide), full)


def test_sparse_width_zero_gives_zeros():
    c = W.make_sparse(2, 8, 1, 128, 100, 8, 2, 0, seed=45, device=DEV)
    c.sel = c.sel[:, :0].contiguous()
    out = torch.full(c.out_shape(), 3.0, dtype=torch.bfloat16, device=DEV)
    B_.run_case(c, out=out)
    assert torch.count_nonzero(out).item() == 0


def test_sparse_named_workload():
    """The full sparse_selected workload, every output row against the oracle, and the same call
    with each sequence's pads removed is bit-identical."""
    c = W.make("sparse_selected", device=DEV)
    out = B_.run_case(c)
    torch.cuda.synchronize()
    host = W.SparseCase(c.q.cpu(), c.k_pool.cpu(), c.v_pool.cpu(), c.sel.cpu(), c.scale, c.B,
                        c.Hq, c.Hkv, c.D, c.pool_rows, c.n_valid_host)
    assert_close(out_f64(out), oracle_for(host), "sparse_selected")
    for b in (0, 7, 31):
        n = c.n_valid_host[b]
        sub = W.SparseCase(c.q[b:b + 1], c.k_pool[b:b + 1], c.v_pool[b:b + 1],
                           c.sel[b:b + 1, :n].contiguous(), c.scale, 1, c.Hq, c.Hkv, c.D,
                           c.pool_rows, [n])
        assert torch.equal(B_.run_case(sub), out[b:b + 1])


def test_no_device_error_recorded():
    assert B_.decode_attn_read_device_error() == 0
