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
    (1, 48, 1, 128, 5000, 2048, 128, 512),  # G = 48: tensor-core kernel, four chunks
    (2, 64, 1, 128, 9000, 5000, 128, 300),  # G = 64: tensor-core kernel, ten chunks
    (2, 48, 1, 64, 3000, 1500, 32, 100),    # G = 48 at D = 64: tensor-core kernel, three chunks
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


@pytest.mark.parametrize("G,Hkv,D", [(64, 1, 128), (8, 2, 128), (4, 4, 64), (16, 1, 128),
                                     (48, 1, 128), (64, 2, 128), (40, 1, 64)])
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


# ---- the tensor-core kernel (33..64 query heads per KV head at D = 128): CTA = (unit, chunk of
# 512 entries) with every head of the unit

TC_CASES = [
    # B, Hq, Hkv, pool_rows, width, window, max_pad
    (2, 64, 1, 2000, 1, 1, 0),        # one entry
    (2, 64, 1, 2000, 64, 8, 0),       # one full tile
    (2, 64, 1, 2000, 65, 8, 0),       # a tile and one row
    (2, 64, 1, 2000, 511, 16, 0),     # chunk - 1
    (2, 64, 1, 2000, 512, 16, 0),     # exactly one chunk
    (2, 64, 1, 2000, 513, 16, 0),     # chunk + 1: a second chunk of one row
    (3, 33, 1, 3000, 1100, 32, 90),   # G = 33: one live lane in the second softmax warp
    (2, 80, 2, 3000, 900, 32, 400),   # G = 40, two units per sequence
    (2, 128, 2, 4000, 1600, 64, 200), # G = 64, two units per sequence, four chunks
    (2, 64, 1, 8000, 2048, 16, 0),    # exactly four chunks: the last tc_merge case
    (2, 64, 1, 8000, 2049, 16, 0),    # five chunks: merge_unit
    (2, 64, 1, 8000, 3000, 32, 100),  # six chunks
    (1, 96, 2, 12000, 6000, 16, 300), # G = 48, twelve chunks
]


@pytest.mark.parametrize("cfg", TC_CASES, ids=lambda c: "B{}_Hq{}_Hkv{}_R{}_W{}".format(*c[:5]))
def test_sparse_tensor_core_kernel_matches_oracle(cfg):
    B, Hq, Hkv, R, width, window, max_pad = cfg
    c = W.make_sparse(B, Hq, Hkv, 128, R, width, window, max_pad, seed=500 + width, device=DEV,
                      poison_unselected=True)
    out = B_.run_case(c)
    assert_close(out_f64(out), oracle_for(c), f"tensor-core sparse {cfg}")


def test_sparse_tensor_core_growing_scores_rescale():
    """Scores that keep growing along the selection move the running maximum by far more than
    the rescale threshold many times inside a chunk (the accumulator is rescaled in TMEM)."""
    c = W.make_sparse(2, 64, 1, 128, 6000, 1500, 32, 0, seed=61, device=DEV)
    for b in range(c.B):
        n = c.n_valid_host[b]
        idx = c.sel[b, :n].long()
        f = (1.0 + torch.arange(n, device=DEV, dtype=torch.float32) / 24.0)[:, None]
        c.k_pool[b, 0, idx] = (c.k_pool[b, 0, idx].float() * f).to(torch.bfloat16)
    out = B_.run_case(c)
    assert_close(out_f64(out), oracle_for(c), "growing scores")


def test_sparse_tensor_core_pad_tiles_and_empty_chunk():
    """Whole tiles of -1 at the start and inside a chunk, and a chunk with no valid entry (its
    partial is empty and the merge skips it)."""
    c = W.make_sparse(2, 64, 1, 128, 4000, 1600, 16, 0, seed=62, device=DEV)
    sel = c.sel.clone()
    sel[0, 0:128] = -1            # the first two tiles of chunk 0
    sel[0, 300:364] = -1          # one tile inside chunk 0
    sel[1, 512:1024] = -1         # chunk 1 entirely
    sel[1, 1030] = 4000           # == pool_rows: skipped
    c.sel = sel
    out = B_.run_case(c)
    assert_close(out_f64(out), oracle_for(c), "pad tiles / empty chunk")


@pytest.mark.parametrize("G,D", [(64, 128), (40, 64)])
def test_pads_bit_identical_across_the_two_merges(G, D):
    """Up to four chunks merge in tc_merge (rows fetched by bulk copies), more in merge_unit; both
    perform the same operations in the same order, so a selection padded from four chunks to ten
    gives the bits of the call without the pads."""
    c = W.make_sparse(3, G, 1, D, 8000, 2000, 64, 500, seed=70 + G, device=DEV,
                      poison_unselected=True)
    ref = B_.run_case(c)                        # up to four chunks: tc_merge
    more = torch.cat([c.sel, torch.full((c.B, 3000), -1, dtype=torch.int32, device=DEV)], dim=1)
    wide = W.SparseCase(c.q, c.k_pool, c.v_pool, more.contiguous(), c.scale, c.B, c.Hq, c.Hkv,
                        c.D, c.pool_rows, c.n_valid_host)
    out = B_.run_case(wide)                     # ten chunks: merge_unit
    assert torch.equal(out, ref)
    assert_close(out_f64(out), oracle_for(c), f"G={G} D={D}")


@pytest.mark.parametrize("width", [2000, 1600, 6000])
def test_sparse_tensor_core_counters_return_to_zero(width):
    """Every call leaves the workspace's merge counters (one word per unit) at zero, and a second
    call on the same workspace gives the same bits."""
    c = W.make_sparse(4, 64, 1, 128, 8000, width, 32, 200, seed=80 + width, device=DEV)
    ws = B_.new_workspace(B_.decode_attn_workspace_size(2, c.B, c.Hq, c.Hkv, c.D, c.width), DEV)
    a = B_.run_case(c, workspace=ws)
    b = B_.run_case(c, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert torch.count_nonzero(ws[: 4 * c.B * c.Hkv]).item() == 0
    assert_close(out_f64(a), oracle_for(c), f"width {width}")


@pytest.mark.parametrize("limit", [0, 1, 5, 7])
def test_sparse_warp_mma_counters_return_to_zero(limit):
    """The warp-MMA kernel's merge counters (one word per unit) are zero after every call,
    whether a CTA computed all of a unit (merged without its counter: every unit with one CTA,
    some with five or seven) or the unit was split across CTAs (counted, then reset by the
    merging CTA: every unit with the full grid of one item per CTA, the others with five or
    seven); a second call on the same workspace gives the same bits, which match the oracle."""
    c = W.make_sparse(3, 32, 2, 128, 3000, 2000, 32, 300, seed=170 + limit, device=DEV)
    ws = B_.new_workspace(B_.decode_attn_workspace_size(2, c.B, c.Hq, c.Hkv, c.D, c.width), DEV)
    B_.decode_attn_set_grid_limit(limit)
    try:
        a = B_.run_case(c, workspace=ws)
        b = B_.run_case(c, workspace=ws)
    finally:
        B_.decode_attn_set_grid_limit(0)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert torch.count_nonzero(ws[: 4 * c.B * c.Hkv]).item() == 0
    assert_close(out_f64(a), oracle_for(c), f"grid limit {limit}")


@pytest.mark.parametrize("limit", [1, 2, 5, 7])
def test_sparse_warp_mma_persistent_grid_is_assignment_free(limit):
    """The warp-MMA sparse kernel runs a persistent grid: with 1..7 CTAs each takes a contiguous
    range of whole (unit, chunk) items, finishing one while gathering the next, and merges units
    split across CTAs.  Every item is computed the same way whichever CTA takes it, so the output
    is bit-identical to the full grid's, and it matches the oracle."""
    c = W.make_sparse(3, 32, 2, 128, 3000, 1700, 32, 400, seed=90 + limit, device=DEV,
                      poison_unselected=True)
    B_.decode_attn_set_grid_limit(0)
    ref = B_.run_case(c)
    B_.decode_attn_set_grid_limit(limit)
    try:
        out = B_.run_case(c)
    finally:
        B_.decode_attn_set_grid_limit(0)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    assert_close(out_f64(out), oracle_for(c), f"grid limit {limit}")


def test_sparse_width_zero_gives_zeros():
    c = W.make_sparse(2, 8, 1, 128, 100, 8, 2, 0, seed=45, device=DEV)
    c.sel = c.sel[:, :0].contiguous()
    out = torch.full(c.out_shape(), 3.0, dtype=torch.bfloat16, device=DEV)
    B_.run_case(c, out=out)
    assert torch.count_nonzero(out).item() == 0


@pytest.mark.parametrize("name", ["sparse_selected", "sparse_selected_g16"])
def test_sparse_named_workload(name):
    """The full sparse workloads (64 query heads per KV head: the tensor-core kernel; 16: the
    warp-MMA kernel), every output row against the oracle, and for every sequence the same call
    with its pads removed is bit-identical."""
    c = W.make(name, device=DEV)
    out = B_.run_case(c)
    torch.cuda.synchronize()
    host = W.SparseCase(c.q.cpu(), c.k_pool.cpu(), c.v_pool.cpu(), c.sel.cpu(), c.scale, c.B,
                        c.Hq, c.Hkv, c.D, c.pool_rows, c.n_valid_host)
    assert_close(out_f64(out), oracle_for(host), name)
    for b in range(c.B):
        n = c.n_valid_host[b]
        sub = W.SparseCase(c.q[b:b + 1], c.k_pool[b:b + 1], c.v_pool[b:b + 1],
                           c.sel[b:b + 1, :n].contiguous(), c.scale, 1, c.Hq, c.Hkv, c.D,
                           c.pool_rows, [n])
        assert torch.equal(B_.run_case(sub), out[b:b + 1]), f"{name}: pads of b={b} not neutral"


def test_no_device_error_recorded():
    assert B_.decode_attn_read_device_error() == 0


@pytest.mark.parametrize("B,Hkv,width", [(80, 1, 1100), (48, 2, 700)])
def test_sparse_tensor_core_kernel_several_waves(B, Hkv, width):
    """More CTAs than SMs (240 and 192 CTAs of one per SM): later CTAs allocate tensor memory on
    SMs whose earlier CTAs have freed it; every output row against the oracle."""
    c = W.make_sparse(B, 64 * Hkv, Hkv, 128, 1500, width, 16, 150, seed=600 + B, device=DEV,
                      poison_unselected=True)
    out = B_.run_case(c)
    assert_close(out_f64(out), oracle_for(c), f"tensor-core sparse, {B} sequences")
    assert B_.decode_attn_read_device_error() == 0


TC64_CASES = [
    # B, Hq, Hkv, pool_rows, width, window, max_pad  (head dim 64)
    (2, 64, 1, 2000, 1, 1, 0),
    (2, 64, 1, 2000, 65, 8, 0),
    (2, 64, 1, 2000, 513, 16, 0),
    (3, 33, 1, 3000, 1100, 32, 90),
    (2, 128, 2, 4000, 1600, 64, 200),
    (60, 40, 1, 1500, 1100, 16, 150),   # 180 CTAs: more than one wave
]


@pytest.mark.parametrize("cfg", TC64_CASES, ids=lambda c: "B{}_Hq{}_Hkv{}_R{}_W{}".format(*c[:5]))
def test_sparse_tensor_core_kernel_d64_matches_oracle(cfg):
    B, Hq, Hkv, R, width, window, max_pad = cfg
    c = W.make_sparse(B, Hq, Hkv, 64, R, width, window, max_pad, seed=700 + width, device=DEV,
                      poison_unselected=True)
    out = B_.run_case(c)
    assert_close(out_f64(out), oracle_for(c), f"tensor-core sparse D=64 {cfg}")


def test_sparse_tensor_core_d64_growing_scores_rescale():
    c = W.make_sparse(2, 48, 1, 64, 6000, 1500, 32, 0, seed=63, device=DEV)
    for b in range(c.B):
        n = c.n_valid_host[b]
        idx = c.sel[b, :n].long()
        f = (1.0 + torch.arange(n, device=DEV, dtype=torch.float32) / 16.0)[:, None]
        c.k_pool[b, 0, idx] = (c.k_pool[b, 0, idx].float() * f).to(torch.bfloat16)
    out = B_.run_case(c)
    assert_close(out_f64(out), oracle_for(c), "growing scores, D=64")
