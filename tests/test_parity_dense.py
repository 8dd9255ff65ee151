"""GPU dense decode attention against the fp64 oracle ("DecodeFlashSpec", fields q / k / v /
k_len / softmax_scale): every output element within 1e-2 + 1e-2 |ref|."""
import numpy as np
import pytest
import torch

from token_decode_attention_split_gb300 import binding as B_
from token_decode_attention_split_gb300 import workloads as W

from helpers import assert_close, bits, oracle_for, out_f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(autouse=True)
def _reset_grid():
    B_.decode_attn_set_grid_limit(0)
    yield
    B_.decode_attn_set_grid_limit(0)


SHAPES = [
    # B, Hq, Hkv, D, capacity, k_len   (several 64-row tiles, ragged tails, every group size)
    (1, 8, 2, 64, 512, 300),
    (2, 8, 8, 128, 300, 257),      # G = 1
    (3, 4, 2, 64, 200, 129),       # G = 2
    (2, 32, 8, 128, 700, 640),     # G = 4, exact multiple of the tile
    (2, 64, 8, 128, 1000, 777),    # G = 8
    (1, 32, 2, 128, 500, 333),     # G = 16
    (2, 32, 1, 64, 400, 190),      # G = 32
    (2, 64, 1, 128, 300, 201),     # G = 64
    (1, 12, 2, 128, 100, 65),      # G = 6 (padded group)
    (1, 40, 1, 128, 100, 99),      # G = 40 (padded group)
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B{}_Hq{}_Hkv{}_D{}_cap{}_k{}".format(*s))
def test_dense_matches_oracle(shape):
    B, Hq, Hkv, D, cap, k_len = shape
    c = W.make_dense(B, Hq, Hkv, D, cap, k_len, seed=100 + k_len, device=DEV, k_scale=2.0,
                     poison_tail=True)
    out = B_.run_case(c)
    assert_close(out_f64(out), oracle_for(c), f"dense {shape}")


@pytest.mark.parametrize("limit", [1, 2, 3, 7, 19])
def test_dense_forced_split_merge(limit):
    """Few CTAs: each (b, kv-head) is cut into several segments merged by log-sum-exp."""
    B_.decode_attn_set_grid_limit(limit)
    c = W.make_dense(2, 16, 2, 128, 1100, 1037, seed=7, device=DEV, k_scale=2.0, poison_tail=True)
    out = B_.run_case(c)
    assert_close(out_f64(out), oracle_for(c), f"grid limit {limit}")


def test_klen_one_returns_v0_exactly():
    c = W.make_dense(2, 16, 2, 128, 64, 1, seed=8, device=DEV, poison_tail=True)
    out = B_.run_case(c)
    v0 = c.v[:, :, 0:1, :].repeat_interleave(8, dim=1)          # [B, Hq, 1, D]
    assert torch.equal(out, v0)


def test_klen_zero_gives_zeros():
    c = W.make_dense(2, 8, 2, 64, 32, 0, seed=9, device=DEV)
    out = torch.full(c.out_shape(), 7.0, dtype=torch.bfloat16, device=DEV)
    B_.run_case(c, out=out)
    assert torch.count_nonzero(out).item() == 0


def test_identical_keys_give_mean_of_v():
    c = W.make_dense(2, 32, 4, 128, 600, 555, seed=10, device=DEV)
    c.k[:] = c.k[:, :, :1, :]
    out = B_.run_case(c)
    mean = c.v[:, :, :c.k_len].double().mean(dim=2).repeat_interleave(8, dim=1)
    assert_close(out_f64(out), mean.cpu().numpy(), "identical keys")


def test_deterministic_and_stream_ordered():
    c = W.make_dense(2, 64, 8, 128, 2000, 1999, seed=11, device=DEV)
    s = torch.cuda.Stream()
    ws = B_.new_workspace(B_.decode_attn_workspace_size(0, c.B, c.Hq, c.Hkv, c.D), DEV)
    B_.decode_attn_set_grid_limit(5)
    with torch.cuda.stream(s):
        a = B_.run_case(c, workspace=ws, stream=s)
        b = B_.run_case(c, workspace=ws, stream=s)
    s.synchronize()
    assert torch.equal(a, b)
    assert torch.count_nonzero(ws[: 4 * c.B * c.Hkv]).item() == 0   # counters back at zero


def test_workspace_too_small_is_rejected():
    c = W.make_dense(1, 8, 2, 64, 64, 64, seed=12, device=DEV)
    need = B_.decode_attn_workspace_size(0, c.B, c.Hq, c.Hkv, c.D)
    ws = B_.new_workspace(need, DEV)
    out = torch.empty(c.out_shape(), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(B_.DecodeAttnError) as e:
        B_.decode_attn_dense(c.q, c.k, c.v, out, c.k_len, c.scale, ws[: need - 16])
    assert e.value.status == 3


@pytest.mark.parametrize("name", ["dense_tiny", "dense_batched", "dense_long"])
def test_dense_named_workloads(name):
    """Full sizes, in the launch configuration the benchmark times: every (b, h) row against the
    oracle (the stream-K schedule splits units at points that depend on the totals, so every
    row's split and merge path is checked), and every row inside the per-column range of the
    attended V rows."""
    c = W.make(name, device=DEV)
    out = B_.run_case(c)
    torch.cuda.synchronize()
    got = out_f64(out)
    host = W.DenseCase(c.q.cpu(), c.k.cpu(), c.v.cpu(), c.k_len, c.scale, c.B, c.Hq, c.Hkv, c.D,
                       c.capacity)
    assert_close(got, oracle_for(host), name)
    assert np.all(np.isfinite(got))
    G = c.Hq // c.Hkv
    live = c.v[:, :, :c.k_len].float()
    lo = live.amin(dim=2).repeat_interleave(G, dim=1).double().cpu().numpy()
    hi = live.amax(dim=2).repeat_interleave(G, dim=1).double().cpu().numpy()
    slack = 1e-2 * np.maximum(np.abs(lo), np.abs(hi)) + 1e-3
    assert np.all(got >= lo - slack) and np.all(got <= hi + slack)


def test_no_device_error_recorded():
    assert B_.decode_attn_read_device_error() == 0


def _dev_len_call(c, k_len_word, out=None, ws=None, stream=None):
    out = torch.empty(c.out_shape(), dtype=torch.bfloat16, device=DEV) if out is None else out
    ws = B_.new_workspace(B_.decode_attn_workspace_size(0, c.B, c.Hq, c.Hkv, c.D), DEV) if ws is None else ws
    return B_.decode_attn_dense_device_len(c.q, c.k, c.v, out, k_len_word, c.scale, ws, stream)


@pytest.mark.parametrize("n", [0, 1, 63, 64, 65, 700, 1000, 5000])
def test_device_len_matches_oracle(n):
    """The live length read from device memory ("DecodeFlashSpec", k_len as a symbol bound each
    token), clamped to the capacity of 1000 rows."""
    c = W.make_dense(2, 32, 4, 128, 1000, 1000, seed=90, device=DEV, k_scale=2.0)
    word = torch.tensor([n], dtype=torch.int32, device=DEV)
    out = _dev_len_call(c, word)
    ref_case = W.DenseCase(c.q, c.k, c.v, min(n, 1000), c.scale, c.B, c.Hq, c.Hkv, c.D, 1000)
    assert_close(out_f64(out), oracle_for(ref_case), f"device k_len {n}")


def test_device_len_graph_replay_follows_the_length_word():
    c = W.make_dense(3, 16, 2, 128, 2048, 2048, seed=91, device=DEV)
    word = torch.tensor([100], dtype=torch.int32, device=DEV)
    out = torch.empty(c.out_shape(), dtype=torch.bfloat16, device=DEV)
    ws = B_.new_workspace(B_.decode_attn_workspace_size(0, c.B, c.Hq, c.Hkv, c.D), DEV)
    _dev_len_call(c, word, out, ws)           # warm-up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.graph(g, stream=s):
        _dev_len_call(c, word, out, ws, s)
    for n in (1, 777, 2048, 64, 0):
        word.fill_(n)
        g.replay()
        torch.cuda.synchronize()
        ref_case = W.DenseCase(c.q, c.k, c.v, n, c.scale, c.B, c.Hq, c.Hkv, c.D, 2048)
        assert_close(out_f64(out), oracle_for(ref_case), f"replay with k_len {n}")


def test_named_device_len_workload():
    """dense_device_len at full size: the length word on the device, every row vs the oracle."""
    c = W.make("dense_device_len", device=DEV)
    out = B_.run_case(c)
    torch.cuda.synchronize()
    host = W.DenseCase(c.q.cpu(), c.k.cpu(), c.v.cpu(), c.k_len, c.scale, c.B, c.Hq, c.Hkv, c.D,
                       c.capacity)
    assert_close(out_f64(out), oracle_for(host), "dense_device_len")


def test_spec_wrapper_matches_the_plain_call():
    """decode_attn_dense_spec (gate passed: causal only) gives the plain call's output bit for
    bit; a softcap is refused before anything runs."""
    c = W.make_dense(2, 16, 4, 128, 600, 555, seed=160, device=DEV, k_scale=2.0)
    ws = B_.new_workspace(B_.decode_attn_workspace_size(0, c.B, c.Hq, c.Hkv, c.D), DEV)
    ref = B_.decode_attn_dense(c.q, c.k, c.v, torch.empty(c.out_shape(), dtype=torch.bfloat16, device=DEV),
                               c.k_len, c.scale, ws)
    spec = B_.DecodeAttnSpec(causal=1, softmax_scale=c.scale)
    a = B_.decode_attn_dense_spec(spec, c.q, c.k, c.v, torch.empty_like(ref), c.k_len, ws)
    torch.cuda.synchronize()
    assert torch.equal(a, ref)
    with pytest.raises(B_.DecodeAttnError) as e:
        B_.decode_attn_dense_spec(B_.DecodeAttnSpec(has_softcap=1, softmax_scale=c.scale),
                                  c.q, c.k, c.v, torch.empty_like(ref), c.k_len, ws)
    assert e.value.status == 2
