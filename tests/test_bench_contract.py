"""The benchmark's reference arm on the CPU: `bench.py --impl reference` times the fp64 oracle and
prints one JSON line with the fields the native arm prints (metric, unit, config of the same
workload, e2e and cpu_baseline describing the run)."""
import json
import os
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_reference(workload):
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", workload,
                          "--steps", "3", "--warmup", "3", "--cpu-budget", "0.5"],
                         cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    return json.loads(lines[0])


@pytest.mark.parametrize("workload", ["dense_tiny", "append_paged", "dense_verify4"])
def test_reference_line(workload):
    import bench
    from token_decode_attention_split_gb300 import workloads as W
    d = run_reference(workload)
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3
    assert d["value"] > 0 and d["e2e"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    cfg = d["config"]
    assert cfg["workload"] == workload
    for k, v in W.CONFIGS[workload].items():
        if k != "seed":
            assert cfg[k] == v
    assert cfg["algorithmic_bytes_per_call"] > 0


@pytest.mark.parametrize("workload", ["dense_tiny", "append_paged"])
def test_both_arms_build_the_same_config(workload):
    """The native arm's config (the same workload fields, per-call bytes, L2 note and
    parallelism, built from input copy 0 of rank 0) equals the reference arm's."""
    import bench
    ref = run_reference(workload)["config"]
    if workload == "append_paged":
        alg, dev = bench.append_shape_bytes(workload)
        native = bench.workload_config(workload, algorithmic_bytes_per_call=int(alg),
                                       l2=bench.l2_note_bytes(alg, dev), parallelism="replicas x1")
    else:
        c0 = bench.make_case(workload, "cpu")
        native = bench.workload_config(workload, algorithmic_bytes_per_call=int(c0.algorithmic_bytes()),
                                       l2=bench.l2_note(c0), parallelism="replicas x1")
    assert native == ref


def test_input_copies_share_structure():
    """Input copies of one rank share their integer structure (so their byte counts are equal)
    and differ in values."""
    import bench
    a = bench.make_case("dense_tiny", "cpu", copy=0)
    b = bench.make_case("dense_tiny", "cpu", copy=1)
    assert a.algorithmic_bytes() == b.algorithmic_bytes()
    assert not torch.equal(a.q.view(torch.int16), b.q.view(torch.int16))
    from token_decode_attention_split_gb300 import workloads as W
    s0 = W.make_sparse(3, 8, 1, 64, 500, 300, 16, 100, seed=5)
    s1 = W.make_sparse(3, 8, 1, 64, 500, 300, 16, 100, seed=5, value_seed=105)
    assert torch.equal(s0.sel, s1.sel) and s0.n_valid_host == s1.n_valid_host
    assert not torch.equal(s0.k_pool.view(torch.int16), s1.k_pool.view(torch.int16))


def test_kernel_kind_follows_the_library_dispatch():
    """The kernel whose sources key a workload's DRAM-traffic record: the sparse workload (64
    query heads per KV head at D = 128) runs the tensor-core sparse kernel, whose hash covers
    sparse_tc.cu as well as the shared headers."""
    import bench
    from token_decode_attention_split_gb300 import workloads as W
    kinds = {name: bench.kernel_kind(cfg) for name, cfg in W.CONFIGS.items()}
    assert kinds["sparse_selected"] == "sparse_tc"
    assert kinds["append_paged"] == "append"
    assert all(k == "decode" for n, k in kinds.items() if n.startswith(("dense", "paged")))
    assert bench.kernel_kind(dict(kind="sparse", Hq=32, Hkv=1, D=128)) == "decode"   # G = 32
    assert bench.kernel_kind(dict(kind="sparse", Hq=64, Hkv=1, D=64)) == "sparse_tc"
    assert bench.kernel_kind(dict(kind="sparse", Hq=33, Hkv=1, D=128)) == "sparse_tc"
    assert any("sparse_tc.cu" in f for f in bench.KERNEL_SOURCES["sparse_tc"])
    assert bench.kernel_label(W.CONFIGS["sparse_selected"]) == "sparse_tc_kernel"
    assert len({bench.kernel_sha(k) for k in bench.KERNEL_SOURCES}) == 3


def test_committed_traffic_records_match_the_kernel_sources():
    """profiles/dram_traffic.json holds, for every named workload but the launch-bound tiny one,
    the DRAM bytes of an ncu capture of the kernel code as it stands (bench.py reports a record
    as roofline.traffic only while the hash of the timed kernel's sources agrees)."""
    import bench
    from token_decode_attention_split_gb300 import workloads as W
    stale = [n for n in W.CONFIGS if n != "dense_tiny" and bench.traffic_record(n) is None]
    assert not stale, f"recapture the profiles of {stale}"
