"""Seeded synthetic inputs for single-query decode attention.

This module only draws inputs (q, K/V caches, block tables, length buffers, selections) and
counts the bytes a call must move.  It holds none of the attention arithmetic, so the fp64
oracle used by the tests and the CUDA library can both be fed from it without sharing code.

Recipe (every value comes from ``torch.Generator(...).manual_seed(seed)``):
  * q, K, V: float32 N(0, 1) rounded to bfloat16 (round-to-nearest-even); K optionally scaled
    before rounding to sharpen the softmax.
  * dense: rows past ``k_len`` of K and V optionally set to NaN, so that reading them shows up.
  * paged: ``kv_len[b]`` uniform integers in [kv_min, kv_max]; the block table gives sequence b
    the consecutive slice ``perm[b*max_pages:(b+1)*max_pages]`` of one random permutation of the
    page ids (the identity with ``shuffle_pages=False``), so no two sequences share a page; every
    page no sequence uses, and every slot past
    ``kv_len`` in a sequence's last page, is NaN.  The length buffer holds u32 words, either one
    per sequence (stride 1) or the ``{kv_len, q_offset, q_rope_pos}`` triple (stride 3).
  * sparse: each sequence's selection of ``width`` int32 entries is the ring-window slots
    ``0..window-1``, then distinct uniform pool rows from ``[window, pool_rows)``, then a seeded
    number in ``[0, max_pad]`` of trailing -1 pads.

The named workloads (``CONFIGS``) are the decode steps the attention kernels are measured on: the
five decode configurations of the scope statement, two variants that route the same recipe
through the other kernel instantiations (64-row pages, 16 query heads per KV head), the
device-length and 4-token verify forms of the batched dense step, and the KV append.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

BF16 = torch.bfloat16

CONFIGS = {
    # dense decode over a capacity buffer's live prefix
    "dense_tiny": dict(kind="dense", B=1, Hq=8, Hkv=2, D=64, capacity=512, k_len=300, seed=1001),
    "dense_batched": dict(kind="dense", B=16, Hq=32, Hkv=8, D=128, capacity=8192, k_len=4096,
                          poison_tail=True, seed=1002),
    "dense_long": dict(kind="dense", B=4, Hq=64, Hkv=8, D=128, capacity=131072, k_len=131071,
                       k_scale=2.0, seed=1003),
    # the batched dense step with its length read on the device (a captured graph replays it
    # for every token), and a 4-token verify step with causal masking inside the new tail
    "dense_device_len": dict(kind="dense", B=16, Hq=32, Hkv=8, D=128, capacity=8192, k_len=4096,
                             poison_tail=True, device_len=True, seed=1007),
    "dense_verify4": dict(kind="dense", B=16, Hq=32, Hkv=8, D=128, capacity=8192, k_len=4096,
                          poison_tail=True, sq=4, causal=1, seed=1008),
    # paged, per-sequence lengths in a device args buffer
    "paged_ragged": dict(kind="paged", B=64, Hq=32, Hkv=8, D=128, page_size=16, num_pages=160000,
                         kv_min=128, kv_max=32768, seed=1004),
    # the same paged step with 64-row pages: one KV head per unit (the single-head paged kernel)
    "paged_ragged_p64": dict(kind="paged", B=64, Hq=32, Hkv=8, D=128, page_size=64,
                             num_pages=40000, kv_min=128, kv_max=32768, seed=1009),
    # sparse, fixed-width int32 selection with trailing -1 pads
    "sparse_selected": dict(kind="sparse", B=32, Hq=64, Hkv=1, D=128, pool_rows=65536, width=2048,
                            window=128, max_pad=512, seed=1005),
    # the same selection recipe with 4 KV heads of 16 query heads each (the warp-MMA sparse kernel)
    "sparse_selected_g16": dict(kind="sparse", B=32, Hq=64, Hkv=4, D=128, pool_rows=65536,
                                width=2048, window=128, max_pad=512, seed=1010),
    # KV append into the paged cache (the step before paged decode): a ctx window of new rows
    "append_paged": dict(kind="append", T=8192, Hkv=8, D=128, page_size=16, num_pages=160000,
                         seed=1006),
}


def _normal_bf16(shape, gen: torch.Generator, device, mult: float = 1.0, chunk_rows: int = 1 << 25):
    """N(0,1) float32 draws (times ``mult``) rounded to bf16, drawn in leading-dim chunks so the
    float32 temporary stays bounded; the draw order (and so the values) does not depend on
    ``chunk_rows`` as long as whole leading-dim slices are drawn in order."""
    out = torch.empty(shape, dtype=BF16, device=device)
    n0 = shape[0]
    inner = math.prod(shape[1:]) if len(shape) > 1 else 1
    step = max(1, chunk_rows // max(1, inner))
    for s in range(0, n0, step):
        e = min(n0, s + step)
        t = torch.randn((e - s,) + tuple(shape[1:]), generator=gen, device=device,
                        dtype=torch.float32)
        if mult != 1.0:
            t.mul_(mult)
        out[s:e].copy_(t)
        del t
    return out


def _gens(seed: int, device, value_seed=None):
    """Generators of one case: float values from ``value_seed`` (default ``seed``) on the device,
    integer structure (lengths, pages, selections, slots) from ``seed`` on the CPU, so two cases
    with one ``seed`` and different ``value_seed`` share their structure and byte counts."""
    dev = torch.device(device)
    g_dev = torch.Generator(device=dev)
    g_dev.manual_seed(seed if value_seed is None else value_seed)
    g_cpu = torch.Generator()
    g_cpu.manual_seed(seed + 7919)
    return dev, g_dev, g_cpu


@dataclass
class DenseCase:
    q: torch.Tensor            # [B, Hq, 1, D] bf16
    k: torch.Tensor            # [B, Hkv, capacity, D] bf16
    v: torch.Tensor            # [B, Hkv, capacity, D] bf16
    k_len: int
    scale: float
    B: int
    Hq: int
    Hkv: int
    D: int
    capacity: int
    kind: str = "dense"
    sq: int = 1                            # query tokens per sequence (q, out [B, Hq, sq, D])
    causal: int = 0                        # sq > 1: token i attends rows [0, k_len - sq + i]
    k_len_dev: torch.Tensor | None = None  # set: the length is read from this device word

    def algorithmic_bytes(self) -> int:
        """Live K/V rows + q + out (bf16), + the length word when it is read on the device."""
        kv = 2 * self.B * self.Hkv * self.k_len * self.D * 2
        return kv + 2 * self.B * self.Hq * self.sq * self.D * 2 + (4 if self.k_len_dev is not None else 0)

    def out_shape(self):
        return (self.B, self.Hq, self.sq, self.D)


@dataclass
class PagedCase:
    q: torch.Tensor            # [B, Hq, 1, D] bf16
    k_pool: torch.Tensor       # [num_pages, Hkv, page_size, D] bf16
    v_pool: torch.Tensor
    block_table: torch.Tensor  # [B, max_pages] int32
    kv_args: torch.Tensor      # int32 words holding u32 values; kv_len of b at b * kv_len_stride
    kv_len_stride: int
    kv_lens_host: list         # the lengths, for byte counting and test bookkeeping
    scale: float
    B: int
    Hq: int
    Hkv: int
    D: int
    page_size: int
    num_pages: int
    kind: str = "paged"

    @property
    def max_pages(self) -> int:
        return self.block_table.shape[1]

    def live_lengths(self):
        cap = self.max_pages * self.page_size
        return [min(int(x), cap) for x in self.kv_lens_host]

    def algorithmic_bytes(self) -> int:
        """Live K/V rows + block-table words read + length words + q + out."""
        lens = self.live_lengths()
        rows = sum(lens)
        pages = sum((n + self.page_size - 1) // self.page_size for n in lens)
        return (2 * rows * self.Hkv * self.D * 2 + pages * 4 + self.B * 4
                + 2 * self.B * self.Hq * self.D * 2)

    def out_shape(self):
        return (self.B, self.Hq, 1, self.D)


@dataclass
class SparseCase:
    q: torch.Tensor            # [B, Hq, 1, D] bf16
    k_pool: torch.Tensor       # [B, Hkv, pool_rows, D] bf16
    v_pool: torch.Tensor
    sel: torch.Tensor          # [B, width] int32
    scale: float
    B: int
    Hq: int
    Hkv: int
    D: int
    pool_rows: int
    n_valid_host: list = field(default_factory=list)
    kind: str = "sparse"

    @property
    def width(self) -> int:
        return self.sel.shape[1]

    def algorithmic_bytes(self) -> int:
        """Selected K/V rows + selection words + q + out."""
        rows = sum(self.n_valid_host)
        return (2 * rows * self.Hkv * self.D * 2 + self.B * self.width * 4
                + 2 * self.B * self.Hq * self.D * 2)

    def out_shape(self):
        return (self.B, self.Hq, 1, self.D)


@dataclass
class AppendCase:
    k_new: torch.Tensor        # [T, Hkv, D] bf16
    v_new: torch.Tensor
    k_pool: torch.Tensor       # [num_pages, Hkv, page_size, D] bf16
    v_pool: torch.Tensor
    slot_mapping: torch.Tensor  # [T] int64
    T: int
    Hkv: int
    D: int
    page_size: int
    num_pages: int
    kind: str = "append"

    def algorithmic_bytes(self) -> int:
        """New rows read + written (K and V, valid slots) + slot words."""
        valid = int(((self.slot_mapping >= 0) &
                     (self.slot_mapping < self.num_pages * self.page_size)).sum())
        return 2 * 2 * valid * self.Hkv * self.D * 2 + self.T * 8


def make_append(T, Hkv, D, page_size, num_pages, seed, device="cpu", pad_every=0,
                value_seed=None) -> AppendCase:
    """T new rows to distinct random slots of a paged pool; with pad_every = n, every n-th slot
    is -1 (a padding row)."""
    dev, g, gc = _gens(seed, device, value_seed)
    if T > num_pages * page_size:
        raise ValueError("more rows than slots")
    slots = torch.randperm(num_pages * page_size, generator=gc)[:T].to(torch.int64)
    if pad_every:
        slots[::pad_every] = -1
    k_new = _normal_bf16((T, Hkv, D), g, dev)
    v_new = _normal_bf16((T, Hkv, D), g, dev)
    k_pool = _normal_bf16((num_pages, Hkv, page_size, D), g, dev)
    v_pool = _normal_bf16((num_pages, Hkv, page_size, D), g, dev)
    return AppendCase(k_new, v_new, k_pool, v_pool, slots.to(dev), T, Hkv, D, page_size, num_pages)


def make_dense(B, Hq, Hkv, D, capacity, k_len, seed, device="cpu", k_scale=1.0,
               poison_tail=False, scale=None, sq=1, causal=0, device_len=False,
               value_seed=None) -> DenseCase:
    """sq > 1: several query tokens per sequence (q [B, Hq, sq, D]); device_len: the length is
    also stored as one u32 word in device memory, for the call that reads it there."""
    dev, g, _ = _gens(seed, device, value_seed)
    q = _normal_bf16((B, Hq, sq, D), g, dev)
    k = _normal_bf16((B, Hkv, capacity, D), g, dev, mult=k_scale)
    v = _normal_bf16((B, Hkv, capacity, D), g, dev)
    if poison_tail and k_len < capacity:
        k[:, :, k_len:, :] = float("nan")
        v[:, :, k_len:, :] = float("nan")
    word = torch.tensor([int(k_len)], dtype=torch.int32, device=dev) if device_len else None
    return DenseCase(q, k, v, int(k_len), scale if scale is not None else 1.0 / math.sqrt(D),
                     B, Hq, Hkv, D, capacity, sq=int(sq), causal=int(causal), k_len_dev=word)


def make_paged(B, Hq, Hkv, D, page_size, num_pages, kv_min, kv_max, seed, device="cpu",
               kv_len_stride=1, max_pages=None, kv_lens=None, poison_unused=True,
               shuffle_pages=True, scale=None, value_seed=None) -> PagedCase:
    dev, g, gc = _gens(seed, device, value_seed)
    if kv_lens is None:
        kv_lens = torch.randint(kv_min, kv_max + 1, (B,), generator=gc).tolist()
    kv_lens = [int(x) for x in kv_lens]
    if max_pages is None:
        max_pages = max(1, -(-max(kv_lens + [kv_max]) // page_size))
    if B * max_pages > num_pages:
        raise ValueError("pool too small for distinct pages per sequence")
    perm = torch.randperm(num_pages, generator=gc)
    if not shuffle_pages:
        perm = torch.arange(num_pages)   # sequence b owns pages [b*max_pages, (b+1)*max_pages)
    bt = perm[: B * max_pages].reshape(B, max_pages).to(torch.int32)
    q = _normal_bf16((B, Hq, 1, D), g, dev)
    k_pool = _normal_bf16((num_pages, Hkv, page_size, D), g, dev)
    v_pool = _normal_bf16((num_pages, Hkv, page_size, D), g, dev)
    if poison_unused:
        used = torch.zeros(num_pages, dtype=torch.bool)
        for b, n in enumerate(kv_lens):
            n = min(n, max_pages * page_size)
            used[bt[b, : -(-n // page_size)].long()] = True
        unused = torch.nonzero(~used).flatten().to(dev)
        if unused.numel():
            k_pool.index_fill_(0, unused, float("nan"))
            v_pool.index_fill_(0, unused, float("nan"))
        for b, n in enumerate(kv_lens):
            n = min(n, max_pages * page_size)
            if n % page_size:
                last = int(bt[b, n // page_size])
                k_pool[last, :, n % page_size:, :] = float("nan")
                v_pool[last, :, n % page_size:, :] = float("nan")
    args = torch.zeros((B, kv_len_stride), dtype=torch.int32)
    args[:, 0] = torch.tensor(kv_lens, dtype=torch.int32)
    if kv_len_stride >= 3:
        # q_offset and q_rope_pos of the {kv_len, q_offset, q_rope_pos} record: the new token
        # sits at position kv_len - 1; seq_q = 1 never reads these words.
        args[:, 1] = torch.tensor([max(0, n - 1) for n in kv_lens], dtype=torch.int32)
        args[:, 2] = args[:, 1]
    return PagedCase(q, k_pool, v_pool, bt.to(dev), args.reshape(-1).to(dev), kv_len_stride,
                     kv_lens, scale if scale is not None else 1.0 / math.sqrt(D), B, Hq, Hkv, D,
                     page_size, num_pages)


def make_sparse(B, Hq, Hkv, D, pool_rows, width, window, max_pad, seed, device="cpu",
                poison_unselected=False, scale=None, value_seed=None) -> SparseCase:
    dev, g, gc = _gens(seed, device, value_seed)
    if window > width or window > pool_rows:
        raise ValueError("window larger than the selection or the pool")
    sel = torch.full((B, width), -1, dtype=torch.int32)
    n_valid = []
    for b in range(B):
        npad = int(torch.randint(0, max_pad + 1, (1,), generator=gc))
        npad = min(npad, width - window)
        nrand = width - window - npad
        if nrand > pool_rows - window:
            raise ValueError("pool too small for distinct selected rows")
        rand = torch.randperm(pool_rows - window, generator=gc)[:nrand] + window
        sel[b, :window] = torch.arange(window, dtype=torch.int32)
        sel[b, window:window + nrand] = rand.to(torch.int32)
        n_valid.append(window + nrand)
    q = _normal_bf16((B, Hq, 1, D), g, dev)
    k_pool = _normal_bf16((B, Hkv, pool_rows, D), g, dev)
    v_pool = _normal_bf16((B, Hkv, pool_rows, D), g, dev)
    if poison_unselected:
        for b in range(B):
            keep = torch.zeros(pool_rows, dtype=torch.bool)
            s = sel[b]
            keep[s[s >= 0].long()] = True
            drop = torch.nonzero(~keep).flatten().to(dev)
            k_pool[b].index_fill_(1, drop, float("nan"))
            v_pool[b].index_fill_(1, drop, float("nan"))
    return SparseCase(q, k_pool, v_pool, sel.to(dev), scale if scale is not None else
                      1.0 / math.sqrt(D), B, Hq, Hkv, D, pool_rows, n_valid)


def make(name: str, device="cpu", **overrides):
    """Builds one of the named workloads (``CONFIGS``), with optional field overrides."""
    cfg = dict(CONFIGS[name])
    cfg.update(overrides)
    kind = cfg.pop("kind")
    if kind == "dense":
        return make_dense(device=device, **cfg)
    if kind == "paged":
        return make_paged(device=device, **cfg)
    if kind == "sparse":
        return make_sparse(device=device, **cfg)
    if kind == "append":
        return make_append(device=device, **cfg)
    raise KeyError(kind)
