"""Which rows a call reads, and how many times: bit-exact on the GPU.

Every attended key is the same vector, so every live row gets the same score and the softmax
weights are exactly equal (the weight exp2(0) = 1 in the kernels); the output is then the plain
mean of the V rows read, with multiplicity.  Each V row carries a one-hot code of its row id
inside a window of D rows (column c = row - D * window), and zeros outside the window, so

    out[c] = (times row D * window + c was read) / (rows read in total),

and round(out * n) recovers every count exactly (a count below 256 survives bf16 rounding).  A
row dropped, read twice, read from the wrong page or selection entry, or a masked entry that was
let through changes a count.  The live scores are -16 (q = 1, k = -1/8, scale 1: every partial
sum exact); a masked row that slipped into the softmax would arrive zero-filled with score 0 and
outweigh all live rows together by e^16, so a weight given to a masked row shows up too.  Rows
that must never be read hold NaN.

The pages fix the counts: "AttnV41", decode_fixed_topk (each selection entry adds its own term,
-1 adds nothing); "DflashScratch", option_b_indirect_args_dev (rows [0, kv_len) through the block
table); "DecodeFlashSpec", k_len (rows [0, k_len)).  Rows out of range are skipped (the reading
this library takes of device-resident values it never validates).
"""
import numpy as np
import pytest
import torch

from token_decode_attention_split_gb300 import binding as B_
from token_decode_attention_split_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"
K_LIVE = -0.125        # q = 1: q.k = -D / 8 (exact), times scale 1


@pytest.fixture(autouse=True)
def _reset_grid():
    B_.decode_attn_set_grid_limit(0)
    yield
    B_.decode_attn_set_grid_limit(0)


def onehot_rows(rows: np.ndarray, window: int, D: int) -> torch.Tensor:
    """bf16 [len(rows), D]: row r gets a 1 in column r - D * window when it lies in the window."""
    v = torch.zeros((len(rows), D), dtype=torch.float32)
    rel = rows - D * window
    inside = np.nonzero((rel >= 0) & (rel < D))[0]
    v[torch.from_numpy(inside), torch.from_numpy(rel[inside])] = 1.0
    return v.to(torch.bfloat16)


def recovered_counts(out: torch.Tensor, n: np.ndarray) -> np.ndarray:
    """[B, Hq, D] counts from a [B, Hq, 1, D] bf16 output and the rows read per sequence."""
    o = out.float().cpu().numpy()[:, :, 0, :].astype(np.float64)
    assert np.all(np.isfinite(o)), "non-finite output"
    return np.rint(o * n.reshape(-1, 1, 1)).astype(np.int64)


def expected_counts(reads, windows, B, Hq, Hkv, D):
    """reads[b]: the multiset (array) of row ids unit b reads (shared by its KV heads);
    windows[b][g]: the window unit (b, g) shows."""
    G = Hq // Hkv
    exp = np.zeros((B, Hq, D), dtype=np.int64)
    for b in range(B):
        ids, cnt = np.unique(np.asarray(reads[b], dtype=np.int64), return_counts=True)
        for g in range(Hkv):
            rel = ids - D * windows[b][g]
            m = (rel >= 0) & (rel < D)
            row = np.zeros(D, dtype=np.int64)
            row[rel[m]] = cnt[m]
            exp[b, g * G:(g + 1) * G] = row
    return exp


def check(out, reads, windows, B, Hq, Hkv, D, what):
    n = np.array([len(r) for r in reads], dtype=np.float64)
    got = recovered_counts(out, np.maximum(n, 1))
    exp = expected_counts(reads, windows, B, Hq, Hkv, D)
    if not np.array_equal(got, exp):
        b, h, c = np.argwhere(got != exp)[0]
        raise AssertionError(f"{what}: row {int(c)} of the window of (b={b}, head {h}) read "
                             f"{got[b, h, c]} times, expected {exp[b, h, c]}")
    # with a power-of-two total the mean itself is exact in bf16
    for b in range(B):
        if len(reads[b]) and (len(reads[b]) & (len(reads[b]) - 1)) == 0:
            want = torch.from_numpy(exp[b] / len(reads[b])).to(torch.bfloat16)
            assert torch.equal(out[b, :, 0, :].cpu(), want), f"{what}: b={b} mean not exact"


# ------------------------------------------------------------------------------------ dense

def dense_case(B, Hq, Hkv, D, cap, k_len, seed, device_len=False):
    c = W.make_dense(B, Hq, Hkv, D, cap, k_len, seed=seed, device=DEV, poison_tail=True,
                     scale=1.0, device_len=device_len)
    nwin = max(1, -(-k_len // D))
    windows = [[(b + g) % nwin for g in range(Hkv)] for b in range(B)]
    c.q.fill_(1.0)
    c.k[:, :, :k_len].fill_(K_LIVE)
    rows = np.arange(k_len)
    for b in range(B):
        for g in range(Hkv):
            c.v[b, g, :k_len] = onehot_rows(rows, windows[b][g], D).to(DEV)
    return c, [rows] * B, windows


@pytest.mark.parametrize("k_len", [1, 63, 64, 65, 127, 128, 129, 640, 1000])
@pytest.mark.parametrize("limit", [0, 3, 7])
def test_dense_rows_read_exactly_once(k_len, limit):
    """Dense tails around the 64-row tile and the 128-row window, with the default grid and with
    3 or 7 CTAs (units cut into segments merged across CTAs)."""
    B_.decode_attn_set_grid_limit(limit)
    B, Hq, Hkv, D = 2, 32, 8, 128
    c, reads, windows = dense_case(B, Hq, Hkv, D, 1024, k_len, seed=300 + k_len)
    out = B_.run_case(c)
    check(out, reads, windows, B, Hq, Hkv, D, f"dense k_len={k_len} grid={limit}")


@pytest.mark.parametrize("k_len", [63, 64, 65, 500])
def test_dense_rows_read_head_dim_64(k_len):
    B, Hq, Hkv, D = 3, 16, 8, 64
    c, reads, windows = dense_case(B, Hq, Hkv, D, 600, k_len, seed=320 + k_len)
    out = B_.run_case(c)
    check(out, reads, windows, B, Hq, Hkv, D, f"dense D=64 k_len={k_len}")


@pytest.mark.parametrize("k_len", [1, 64, 65, 999])
def test_dense_device_len_rows_read(k_len):
    """The length read from a device word: the rows past it in the last tile are fetched but
    must not count."""
    B, Hq, Hkv, D = 2, 32, 8, 128
    c, reads, windows = dense_case(B, Hq, Hkv, D, 1000, k_len, seed=340 + k_len, device_len=True)
    out = B_.run_case(c)
    check(out, reads, windows, B, Hq, Hkv, D, f"device k_len={k_len}")


# ------------------------------------------------------------------------------------ paged

def paged_case(B, Hq, Hkv, D, P, lens, max_pages, seed, bad=()):
    """bad: (b, page index) block-table entries replaced by an out-of-range page id."""
    num_pages = B * max_pages + 7
    c = W.make_paged(B, Hq, Hkv, D, P, num_pages, 1, 1, seed=seed, device=DEV, kv_lens=lens,
                     max_pages=max_pages, scale=1.0)
    bt = c.block_table.cpu().numpy().copy()
    for i, (b, j) in enumerate(bad):
        bt[b, j] = num_pages + 3 if i % 2 == 0 else -5
    c.block_table.copy_(torch.from_numpy(bt))
    c.q.fill_(1.0)
    cap = max_pages * P
    reads, windows = [], []
    nwin = max(1, -(-min(max(lens), cap) // D))
    for b in range(B):
        n = min(lens[b], cap)
        j = np.arange(n)
        keep = (bt[b, j // P] >= 0) & (bt[b, j // P] < num_pages)
        j = j[keep]
        reads.append(j)
        windows.append([(b + g) % nwin for g in range(Hkv)])
        if len(j) == 0:
            continue
        pages = torch.from_numpy(bt[b, j // P].astype(np.int64)).to(DEV)
        slots = torch.from_numpy(j % P).to(DEV)
        for g in range(Hkv):
            c.k_pool[pages, g, slots] = torch.full((len(j), D), K_LIVE, dtype=torch.bfloat16,
                                                   device=DEV)
            c.v_pool[pages, g, slots] = onehot_rows(j, windows[b][g], D).to(DEV)
    return c, reads, windows


@pytest.mark.parametrize("P", [16, 64])
@pytest.mark.parametrize("limit", [0, 5, 13])
def test_paged_rows_read_exactly_once(P, limit):
    """Lengths at page boundaries (one row before, on, after), one page, a length clamped to the
    block table's reach, and out-of-range page ids (those pages' rows are skipped); 16-row pages
    run units of four KV heads, 64-row pages units of one."""
    B_.decode_attn_set_grid_limit(limit)
    B, Hq, Hkv, D = 8, 32, 8, 128
    max_pages = -(-1000 // P)
    lens = [P - 1, P, P + 1, 4 * P + 1, 999, 1, 5000, 3 * P]
    bad = [(4, 1), (6, 2)]
    c, reads, windows = paged_case(B, Hq, Hkv, D, P, lens, max_pages, seed=400 + P, bad=bad)
    out = B_.run_case(c)
    check(out, reads, windows, B, Hq, Hkv, D, f"paged P={P} grid={limit}")


@pytest.mark.parametrize("P", [8, 32, 128, 256])
def test_paged_rows_read_other_page_sizes(P):
    """Pages of 8 and 32 rows (units of eight and two KV heads) and of 128 and 256 rows."""
    B, Hq, Hkv, D = 4, 16, 8, 128
    max_pages = -(-700 // P)
    lens = [P + 1, 700, 2 * P - 1, 1]
    c, reads, windows = paged_case(B, Hq, Hkv, D, P, lens, max_pages, seed=420 + P)
    out = B_.run_case(c)
    check(out, reads, windows, B, Hq, Hkv, D, f"paged P={P}")


# ----------------------------------------------------------------------------------- sparse

def selection(width, pool_rows, n_valid_target, rng, extras=True):
    """width entries: ring slots, random rows (some duplicated), an interior -1, a negative
    entry, an entry past the pool (those three when extras), then trailing -1 pads; at most
    n_valid_target entries are not pads."""
    body = list(range(min(16, n_valid_target)))
    pool = rng.permutation(np.arange(16, pool_rows))
    k = 0
    while len(body) < n_valid_target:
        if extras and len(body) % 97 == 50:
            body.append(body[-7])                        # a duplicate
        elif extras and len(body) == n_valid_target // 2:
            body.extend([-1, -7, pool_rows + 5][: n_valid_target - len(body)])
        else:
            body.append(int(pool[k % len(pool)]))
            k += 1
    sel = np.full(width, -1, dtype=np.int32)
    sel[:len(body)] = body[:width]
    return sel


def sparse_case(B, Hq, Hkv, D, pool_rows, sel_row):
    """Every sequence gets the same selection; unit (b, g) shows window (b * Hkv + g) % nwin;
    pool rows no valid entry names hold NaN."""
    valid = sel_row[(sel_row >= 0) & (sel_row < pool_rows)].astype(np.int64)
    rows = np.unique(valid)
    nwin = -(-pool_rows // D)
    windows = [[(b * Hkv + g) % nwin for g in range(Hkv)] for b in range(B)]
    q = torch.ones((B, Hq, 1, D), dtype=torch.bfloat16, device=DEV)
    k_pool = torch.full((B, Hkv, pool_rows, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    v_pool = torch.full_like(k_pool, float("nan"))
    rows_t = torch.from_numpy(rows).to(DEV)
    for b in range(B):
        for g in range(Hkv):
            k_pool[b, g, rows_t] = K_LIVE
            v_pool[b, g, rows_t] = onehot_rows(rows, windows[b][g], D).to(DEV)
    sel = torch.from_numpy(np.tile(sel_row, (B, 1))).to(DEV)
    c = W.SparseCase(q, k_pool, v_pool, sel, 1.0, B, Hq, Hkv, D, pool_rows, [len(valid)] * B)
    return c, [valid] * B, windows


SPARSE_KERNELS = [
    # Hq, Hkv, D: the tensor-core kernel (33..64 heads per KV head) and the warp-MMA kernel
    (64, 1, 128), (64, 1, 64), (48, 1, 128), (32, 1, 128), (32, 2, 128), (8, 2, 64),
]


@pytest.mark.parametrize("Hq,Hkv,D", SPARSE_KERNELS, ids=lambda x: str(x))
@pytest.mark.parametrize("width,n_sel", [(511, 511), (512, 512), (513, 513), (1024, 700),
                                         (1100, 1025), (2048, 1536)])
def test_sparse_rows_read_with_multiplicity(Hq, Hkv, D, width, n_sel):
    """Chunk edges (511 / 512 / 513 entries, chunks of 512), several chunks merged, duplicates
    counted once per entry, interior -1, other negatives and entries past the pool skipped,
    trailing pads."""
    rng = np.random.default_rng(width * 7 + n_sel)
    pool_rows = 1024
    sel_row = selection(width, pool_rows, n_sel, rng)
    B = -(-pool_rows // D) // Hkv
    c, reads, windows = sparse_case(B, Hq, Hkv, D, pool_rows, sel_row)
    out = B_.run_case(c)
    check(out, reads, windows, B, Hq, Hkv, D, f"sparse G={Hq // Hkv} D={D} width={width}")


@pytest.mark.parametrize("limit", [1, 3])
@pytest.mark.parametrize("Hq,Hkv,D", [(32, 2, 128), (8, 2, 64)], ids=lambda x: str(x))
def test_sparse_rows_read_on_few_ctas(Hq, Hkv, D, limit):
    """The warp-MMA sparse kernel with 1 or 3 CTAs, each taking many (unit, chunk) items in a row:
    every item still reads exactly its own rows."""
    B_.decode_attn_set_grid_limit(limit)
    rng = np.random.default_rng(limit * 31 + D)
    pool_rows = 1024
    sel_row = selection(1100, pool_rows, 1025, rng)
    B = -(-pool_rows // D) // Hkv
    c, reads, windows = sparse_case(B, Hq, Hkv, D, pool_rows, sel_row)
    out = B_.run_case(c)
    check(out, reads, windows, B, Hq, Hkv, D, f"sparse G={Hq // Hkv} D={D} grid={limit}")


@pytest.mark.parametrize("name", ["sparse_selected", "sparse_selected_g16"])
def test_sparse_named_workload_rows_read(name):
    """At the named workloads' full shape (width 2048, 65536 pool rows, the launch the benchmark
    times): all sequences take sequence 0's selection (its ring slots, distinct random rows and
    trailing pads); over 16 calls every window of the pool is shown by one unit, so every pool
    row's count is checked."""
    c = W.make(name, device=DEV)
    B, Hq, Hkv, D, R = c.B, c.Hq, c.Hkv, c.D, c.pool_rows
    sel_row = c.sel[0].cpu().numpy().copy()
    c.sel.copy_(torch.from_numpy(np.tile(sel_row, (B, 1))))
    c.q.fill_(1.0)
    c.scale = 1.0
    valid = sel_row[sel_row >= 0].astype(np.int64)
    rows_t = torch.from_numpy(valid).to(DEV)
    c.k_pool.fill_(float("nan"))
    c.k_pool[:, :, rows_t] = K_LIVE
    nwin = R // D
    units = B * Hkv
    for call in range(-(-nwin // units)):
        windows = [[(call * units + b * Hkv + g) % nwin for g in range(Hkv)] for b in range(B)]
        c.v_pool.fill_(float("nan"))
        for b in range(B):
            for g in range(Hkv):
                c.v_pool[b, g, rows_t] = onehot_rows(valid, windows[b][g], D).to(DEV)
        out = B_.run_case(c)
        check(out, [valid] * B, windows, B, Hq, Hkv, D, f"{name} call {call}")


def test_no_device_error_recorded():
    assert B_.decode_attn_read_device_error() == 0
