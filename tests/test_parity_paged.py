"""GPU paged decode attention against the fp64 oracle ("DflashScratch",
option_b_indirect_args_dev: kv_len read on the device, rows gathered through a block table)."""
import numpy as np
import pytest
import torch

from token_decode_attention_split_gb300 import binding as B_
from token_decode_attention_split_gb300 import workloads as W

from helpers import assert_close, oracle_for, out_f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(autouse=True)
def _reset_grid():
    B_.decode_attn_set_grid_limit(0)
    yield
    B_.decode_attn_set_grid_limit(0)


CASES = [
    # B, Hq, Hkv, D, page_size, num_pages, kv_min, kv_max, stride
    (4, 32, 8, 128, 16, 512, 1, 600, 1),
    (5, 8, 2, 64, 8, 1024, 1, 500, 3),
    (3, 16, 2, 128, 32, 256, 30, 700, 3),
    (3, 8, 1, 128, 64, 64, 60, 700, 1),
    (2, 64, 8, 128, 128, 64, 100, 900, 1),
    (2, 16, 16, 128, 256, 32, 200, 1000, 3),
    (3, 64, 1, 128, 16, 300, 1, 800, 1),
    (3, 32, 8, 128, 8, 2048, 1, 700, 1),    # 8-row pages: eight KV heads (32 columns) per unit
    (2, 24, 8, 64, 16, 600, 5, 900, 3),     # G = 3, D = 64: four KV heads per unit
    (2, 64, 8, 128, 8, 1024, 1, 500, 1),    # G = 8, 8-row pages: eight KV heads, 64 columns
    (2, 32, 2, 128, 64, 200, 1, 700, 1),    # G = 16: one KV head (16 columns) per unit
    (2, 64, 2, 64, 128, 100, 1, 800, 3),    # G = 32, D = 64: one KV head (32 columns) per unit
]


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: "B{}_Hq{}_Hkv{}_D{}_P{}_np{}_{}-{}_s{}".format(*c))
def test_paged_matches_oracle(cfg):
    B, Hq, Hkv, D, P, npages, lo, hi, stride = cfg
    c = W.make_paged(B, Hq, Hkv, D, P, npages, lo, hi, seed=200 + P, device=DEV,
                     kv_len_stride=stride)
    out = B_.run_case(c)
    assert_close(out_f64(out), oracle_for(c), f"paged {cfg}")


@pytest.mark.parametrize("limit", [1, 2, 5, 13])
def test_paged_forced_split_merge(limit):
    B_.decode_attn_set_grid_limit(limit)
    c = W.make_paged(6, 32, 8, 128, 16, 600, 1, 1500, seed=31, device=DEV)
    out = B_.run_case(c)
    assert_close(out_f64(out), oracle_for(c), f"grid limit {limit}")


def test_paged_edge_lengths():
    """kv_len 0 (zero row), 1, page_size - 1, page_size, page_size + 1, and a length past
    max_pages * page_size (clamped)."""
    lens = [0, 1, 15, 16, 17, 64, 65, 10_000]
    c = W.make_paged(len(lens), 16, 4, 128, 16, 256, 0, 0, seed=32, device=DEV, max_pages=8,
                     kv_lens=lens)
    out = B_.run_case(c)
    got = out_f64(out)
    assert np.all(got[0] == 0.0)
    assert_close(got, oracle_for(c), "edge lengths")


def test_paged_out_of_range_pages_are_skipped():
    c = W.make_paged(3, 8, 2, 128, 16, 64, 40, 60, seed=33, device=DEV, max_pages=4,
                     kv_lens=[60, 50, 64], poison_unused=False)
    bt = c.block_table.clone()
    bt[0, 1] = -3
    bt[1, 0] = 1 << 30
    bt[2, 3] = 64                      # == num_pages
    c.block_table = bt
    out = B_.run_case(c)
    assert_close(out_f64(out), oracle_for(c), "out-of-range pages")


def test_paged_matches_dense_on_the_same_rows():
    """Scatter a dense cache into random pages; both paths agree within the tolerance."""
    B, Hq, Hkv, D, P, L = 3, 32, 4, 128, 16, 700
    d = W.make_dense(B, Hq, Hkv, D, L, L, seed=34, device=DEV)
    maxp = L // P + 1
    npages = B * maxp + 5
    perm = torch.randperm(npages, generator=torch.Generator().manual_seed(1))[:B * maxp]
    bt = perm.reshape(B, maxp).to(torch.int32)
    kp = torch.zeros(npages, Hkv, P, D, dtype=torch.bfloat16, device=DEV)
    vp = torch.zeros_like(kp)
    for b in range(B):
        for j0 in range(0, L, P):
            n = min(P, L - j0)
            kp[bt[b, j0 // P], :, :n] = d.k[b, :, j0:j0 + n]
            vp[bt[b, j0 // P], :, :n] = d.v[b, :, j0:j0 + n]
    lens = torch.tensor([L, 333, 17], dtype=torch.int32)
    pc = W.PagedCase(d.q, kp, vp, bt.to(DEV), lens.to(DEV), 1, lens.tolist(), d.scale, B, Hq, Hkv,
                     D, P, npages)
    out_p = out_f64(B_.run_case(pc))
    for b, n in enumerate(lens.tolist()):
        dc = W.DenseCase(d.q[b:b + 1], d.k[b:b + 1], d.v[b:b + 1], n, d.scale, 1, Hq, Hkv, D, L)
        assert_close(out_p[b:b + 1], out_f64(B_.run_case(dc)), f"paged vs dense b={b}")


def test_paged_graph_replay_reads_lengths_on_device():
    """Capture one call in a CUDA graph, rewrite the length words in place, replay: the output
    follows the new lengths (the host never passes them)."""
    c = W.make_paged(4, 16, 4, 128, 16, 256, 50, 400, seed=35, device=DEV, kv_len_stride=3,
                     max_pages=25, poison_unused=False)
    ws = B_.new_workspace(B_.decode_attn_workspace_size(1, c.B, c.Hq, c.Hkv, c.D), DEV)
    out = torch.empty(c.out_shape(), dtype=torch.bfloat16, device=DEV)
    B_.run_case(c, out=out, workspace=ws)          # warm-up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.graph(g, stream=s):
        B_.run_case(c, out=out, workspace=ws, stream=s)
    for new in ([10, 200, 1, 399], [400, 0, 64, 65]):
        args = c.kv_args.view(c.B, 3).clone()
        args[:, 0] = torch.tensor(new, dtype=torch.int32, device=DEV)
        c.kv_args.copy_(args.reshape(-1))
        c.kv_lens_host = new
        g.replay()
        torch.cuda.synchronize()
        got = out_f64(out)
        assert np.all(got[[i for i, n in enumerate(new) if n == 0]] == 0.0)
        assert_close(got, oracle_for(c), f"replay {new}")


@pytest.mark.parametrize("name", ["paged_ragged", "paged_ragged_p64"])
def test_paged_named_workload(name):
    """The full paged workloads (16-row pages: units of four KV heads; 64-row pages: one KV head
    per unit), in the launch configuration the benchmark times: every sequence's every row
    against the oracle, on a compact host copy of the pages the sequences use."""
    c = W.make(name, device=DEV)
    out = B_.run_case(c)
    torch.cuda.synchronize()
    got = out_f64(out)
    assert np.all(np.isfinite(got))
    lens = c.live_lengths()
    bt = c.block_table.cpu()
    npg = [-(-n // c.page_size) for n in lens]
    first = np.concatenate([[0], np.cumsum(npg)[:-1]]).astype(np.int64)
    pages = torch.cat([bt[b, :npg[b]].long() for b in range(c.B)]).to(DEV)
    kp = c.k_pool.index_select(0, pages).cpu()
    vp = c.v_pool.index_select(0, pages).cpu()
    table = torch.zeros((c.B, max(npg)), dtype=torch.int32)
    for b in range(c.B):
        table[b, :npg[b]] = torch.arange(first[b], first[b] + npg[b], dtype=torch.int32)
    host = W.PagedCase(c.q.cpu(), kp, vp, table, torch.tensor(lens, dtype=torch.int32), 1, lens,
                       c.scale, c.B, c.Hq, c.Hkv, c.D, c.page_size, int(pages.numel()))
    assert_close(got, oracle_for(host), name)


def test_no_device_error_recorded():
    assert B_.decode_attn_read_device_error() == 0
