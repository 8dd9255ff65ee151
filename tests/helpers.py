"""Shared helpers for the parity tests: oracle calls for workload objects and the tolerance."""
import numpy as np
import torch

import oracle

RTOL = 1e-2
ATOL = 1e-2


def out_f64(out: torch.Tensor) -> np.ndarray:
    """bf16 [B,Hq,1,D] device output -> fp64 [B,Hq,D] host array."""
    return out.float().cpu().numpy()[:, :, 0, :].astype(np.float64)


def oracle_for(case, pairs=None):
    if case.kind == "dense":
        return oracle.dense(case.q, case.k, case.v, case.k_len, case.scale, pairs=pairs)
    if case.kind == "paged":
        return oracle.paged(case.q, case.k_pool, case.v_pool, case.block_table.cpu().numpy(),
                            case.kv_args.cpu().numpy().view(np.uint32), case.scale,
                            kv_len_stride=case.kv_len_stride, pairs=pairs)
    return oracle.sparse(case.q, case.k_pool, case.v_pool, case.sel.cpu().numpy(), case.scale,
                         pairs=pairs)


def assert_close(got: np.ndarray, ref: np.ndarray, what: str = ""):
    """|got - ref| <= 1e-2 + 1e-2 |ref| elementwise (bf16 I/O, fp32 accumulation)."""
    assert got.shape == ref.shape, (got.shape, ref.shape)
    bad = ~(np.abs(got - ref) <= ATOL + RTOL * np.abs(ref))
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; first at "
                             f"{tuple(i)}: got {got[tuple(i)]!r} ref {ref[tuple(i)]!r}")


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy()
