"""Decode-attention benchmark: achieved HBM GB/s (and % of the measured GB300 copy peak) and
µs per call, on one of the named synthetic workloads (default: paged_ragged, the largest).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]
                    [--min-seconds S]

A step is one decode-attention call over the whole workload (one kernel launch; inputs resident
in HBM).  K steps are captured in one CUDA graph; after W warm-up steps and about a second of
untimed replays (steady clocks), the graph is replayed R times between two CUDA events on the
launching stream, R chosen so the timed region lasts about S seconds (default 4), and the line
reports the mean per call.  Several independent input copies (same lengths and selections,
different values) are alternated call by call, as many as it takes for their live bytes to exceed
the L2 three times over, so no call reads what the previous ones left in L2.  With N > 1
(torchrun), every rank runs its own replica of the workload with its own seed; the job value is
the bytes of all ranks over the slowest rank's time.  ``--impl reference`` times the fp64 CPU
oracle on the host cores instead (a bounded sample of the same workload).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from token_decode_attention_split_gb300 import workloads as W  # noqa: E402

METRIC = "decode-attention achieved HBM GB/s (% of GB300 peak) and µs per call"
NOMINAL_HBM_GBS = 8000.0     # the ~8 TB/s nominal HBM3e figure of a GB300, context only
DEFAULT_WORKLOAD = "paged_ragged"
L2_BYTES = 129 * 10**6       # GB300 L2 (bytes)
COPY_BUDGET_BYTES = 48 * 10**9   # device memory the alternated input copies may take
KERNEL_SOURCES = {
    "decode": ["token_decode_attention_split_gb300/csrc/decode_kernel.cuh",
               "token_decode_attention_split_gb300/csrc/ptx.cuh"],
    "sparse_tc": ["token_decode_attention_split_gb300/csrc/sparse_tc.cu",
                  "token_decode_attention_split_gb300/csrc/decode_kernel.cuh",
                  "token_decode_attention_split_gb300/csrc/ptx.cuh"],
    "append": ["token_decode_attention_split_gb300/csrc/append.cu",
               "token_decode_attention_split_gb300/csrc/ptx.cuh"],
}


def kernel_kind(cfg: dict) -> str:
    """Which kernel a workload's timed call runs: "append", "sparse_tc" (sparse calls with 33..64
    query heads per KV head go to the tensor-core kernel, as the library dispatches them) or
    "decode" (the mma.sync decode kernel)."""
    if cfg["kind"] == "append":
        return "append"
    if cfg["kind"] == "sparse" and 32 < cfg["Hq"] // cfg["Hkv"] <= 64:
        return "sparse_tc"
    return "decode"


def kernel_label(cfg: dict) -> str:
    k = kernel_kind(cfg)
    return {"append": "append_kernel", "sparse_tc": "sparse_tc_kernel"}.get(
        k, f"decode_attn_kernel<{cfg['kind']}>")


def code_only(src: str) -> str:
    """C/C++ source without comments, whitespace runs collapsed (string literals kept)."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            i = src.find("\n", i)
            i = n if i < 0 else i
        elif src.startswith("/*", i):
            i = src.find("*/", i + 2)
            i = n if i < 0 else i + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_sha(kind: str = "decode") -> str:
    """First 16 hex digits of the sha256 of the code (comments and layout aside) of the sources
    of the kernel a workload times (kind: a kernel_kind())."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, f), encoding="utf-8") as fh:
            h.update(code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def traffic_record(workload: str):
    """DRAM bytes per launch from the committed ncu summary, or None when it was taken on other
    kernel sources than the ones built now."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        rec = d.get(workload)
        if rec and rec.get("kernel_sha") == kernel_sha(kernel_kind(W.CONFIGS[workload])):
            return float(rec["bytes_per_launch"])
    except Exception:
        pass
    return None


def gpu_selector(dev) -> str:
    """nvidia-smi -i argument for the torch device: its UUID when torch reports one."""
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(dev.index or 0)


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: str):
        self.gpu = gpu
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": float(max(smax)) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


OVERRIDES = {}


def make_case(name: str, device, rank: int = 0, copy: int = 0):
    """Input copy `copy` of rank `rank`'s replica: every copy of a rank shares the integer
    structure (lengths, pages, selection: the seed) and draws its own values (the value seed)."""
    cfg = dict(W.CONFIGS[name])
    cfg.update(OVERRIDES)
    seed = cfg["seed"] + 1000 * rank
    return W.make(name, device=device, **{**OVERRIDES, "seed": seed, "value_seed": seed + 100 * copy})


def case_device_bytes(case) -> int:
    """Bytes of every tensor of a case (what one input copy holds on the device)."""
    n = 0
    for v in vars(case).values():
        if isinstance(v, torch.Tensor):
            n += v.numel() * v.element_size()
    return n


def copies_for(alg: int, device_bytes: int) -> int:
    """Input copies to alternate: enough that their live bytes exceed the L2 three times over
    (2 at least, 16 at most), within COPY_BUDGET_BYTES of device memory."""
    want = max(2, min(16, -(-3 * L2_BYTES // max(1, alg))))
    fit = max(2, COPY_BUDGET_BYTES // max(1, device_bytes))
    return int(min(want, fit))


def input_copies(case) -> int:
    return copies_for(case.algorithmic_bytes(), case_device_bytes(case))


def l2_note(case) -> str:
    return l2_note_bytes(case.algorithmic_bytes(), case_device_bytes(case))


def parse_overrides(items):
    out = {}
    for it in items or []:
        k, v = it.split("=", 1)
        try:
            out[k] = int(v)
        except ValueError:
            out[k] = float(v)
    return out


def case_bytes_copied(case):
    """Host->device bytes of one end-to-end step: the buffers the step reads."""
    if case.kind == "append":
        return 2 * case.k_new.numel() * 2 + case.slot_mapping.numel() * 8
    if case.kind == "dense":
        live = 2 * case.B * case.Hkv * case.k_len * case.D * 2
        return case.q.numel() * 2 + live
    if case.kind == "paged":
        return (case.q.numel() * 2 + 2 * case.k_pool.numel() * 2 + case.block_table.numel() * 4
                + case.kv_args.numel() * 4)
    return case.q.numel() * 2 + 2 * case.k_pool.numel() * 2 + case.sel.numel() * 4


class HostCopy:
    """Pinned host copies of one case's inputs and the per-step H2D / D2H copies of the
    end-to-end measurement (dense: the live rows of each (b, kv-head) as one strided copy)."""

    def __init__(self, case):
        self.case = case
        import ctypes
        self.rt = ctypes.CDLL("libcudart.so.13")
        self.rt.cudaMemcpy2DAsync.restype = ctypes.c_int
        self.rt.cudaMemcpy2DAsync.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
                                              ctypes.c_size_t, ctypes.c_size_t, ctypes.c_size_t,
                                              ctypes.c_int, ctypes.c_void_p]
        c = case
        if c.kind == "append":
            self.kn = c.k_new.cpu().pin_memory()
            self.vn = c.v_new.cpu().pin_memory()
            self.sm = c.slot_mapping.cpu().pin_memory()
            self.out = None
            return
        if c.kind == "dense":
            self.q = c.q.cpu().pin_memory()
            self.k = c.k[:, :, :c.k_len].contiguous().cpu().pin_memory()
            self.v = c.v[:, :, :c.k_len].contiguous().cpu().pin_memory()
        elif c.kind == "paged":
            self.q = c.q.cpu().pin_memory()
            self.k = c.k_pool.cpu().pin_memory()
            self.v = c.v_pool.cpu().pin_memory()
            self.bt = c.block_table.cpu().pin_memory()
            self.kl = c.kv_args.cpu().pin_memory()
        else:
            self.q = c.q.cpu().pin_memory()
            self.k = c.k_pool.cpu().pin_memory()
            self.v = c.v_pool.cpu().pin_memory()
            self.sel = c.sel.cpu().pin_memory()
        self.out = torch.empty(c.out_shape(), dtype=torch.bfloat16).pin_memory()

    def h2d(self, stream, dst=None):
        """Copies the pinned inputs into `dst` (a case of the same shapes; default: the source
        case's own device buffers)."""
        c = self.case if dst is None else dst
        s = stream.cuda_stream
        if c.kind == "append":
            c.k_new.copy_(self.kn, non_blocking=True)
            c.v_new.copy_(self.vn, non_blocking=True)
            c.slot_mapping.copy_(self.sm, non_blocking=True)
            return
        c.q.copy_(self.q, non_blocking=True)
        if c.kind == "dense":
            rows = c.B * c.Hkv
            width = c.k_len * c.D * 2
            pitch = c.capacity * c.D * 2
            for dst, src in ((c.k, self.k), (c.v, self.v)):
                rc = self.rt.cudaMemcpy2DAsync(dst.data_ptr(), pitch, src.data_ptr(), width,
                                               width, rows, 1, s)
                if rc != 0:
                    raise RuntimeError(f"cudaMemcpy2DAsync failed ({rc})")
        elif c.kind == "paged":
            c.k_pool.copy_(self.k, non_blocking=True)
            c.v_pool.copy_(self.v, non_blocking=True)
            c.block_table.copy_(self.bt, non_blocking=True)
            c.kv_args.copy_(self.kl, non_blocking=True)
        else:
            c.k_pool.copy_(self.k, non_blocking=True)
            c.v_pool.copy_(self.v, non_blocking=True)
            c.sel.copy_(self.sel, non_blocking=True)

    def d2h(self, out):
        if self.out is not None:      # append: the result is the device cache itself
            self.out.copy_(out, non_blocking=True)


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if (args.impl == "native" and torch.cuda.is_available()) else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def dist_max(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def oracle_sample_run(case_host, budget_s: float):
    """Runs the oracle on as many (b, h) rows of the workload as fit in about ``budget_s``
    seconds (whole passes when they fit); returns (rows, seconds, threads)."""
    import oracle
    n = case_host.B * case_host.Hq
    threads = os.cpu_count() or 1
    # size the sample from a short probe
    probe = np.arange(min(n, max(1, threads)), dtype=np.int64)
    t0 = time.perf_counter()
    done = _run_oracle(case_host, probe, threads)
    dt = max(time.perf_counter() - t0, 1e-6)
    per_row = dt / done
    rows = int(max(1, min(n, budget_s / per_row)))
    pairs = np.linspace(0, n - 1, rows).round().astype(np.int64)
    pairs = np.unique(pairs)
    # a sample shorter than the budget is repeated (whole passes) to fill about half of it
    passes, done, t0 = 0, 0, time.perf_counter()
    while True:
        done += _run_oracle(case_host, pairs, threads)
        passes += 1
        el = time.perf_counter() - t0
        if el >= budget_s / 2 or passes >= 1000:
            break
    return done, el, threads


def _run_oracle(c, pairs, threads):
    """The oracle on the (b, h) rows `pairs` of a host case; returns the rows it computed (for
    several query tokens, every head of each sequence that `pairs` touches)."""
    import oracle
    if c.kind == "dense" and c.sq > 1:
        bs = np.unique(np.asarray(pairs) // c.Hq)
        oracle.dense_mq(c.q[bs], c.k[bs], c.v[bs], c.k_len, c.scale, causal=bool(c.causal),
                        nthreads=threads)
        return len(bs) * c.Hq
    if c.kind == "dense":
        oracle.dense(c.q, c.k, c.v, c.k_len, c.scale, pairs=pairs, nthreads=threads)
    elif c.kind == "paged":
        oracle.paged(c.q, c.k_pool, c.v_pool, c.block_table.numpy(),
                     c.kv_args.numpy().view(np.uint32), c.scale,
                     kv_len_stride=c.kv_len_stride, pairs=pairs, nthreads=threads)
    else:
        oracle.sparse(c.q, c.k_pool, c.v_pool, c.sel.numpy(), c.scale, pairs=pairs,
                      nthreads=threads)
    return len(pairs)


def cpu_case(name):
    """The workload built on the host (seeded like the GPU run; for the large pools the host
    draw is slow, so it is drawn on the GPU when one is present and copied back)."""
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    c = make_case(name, dev)
    if dev == "cpu":
        return c
    for f in ("q", "k", "v", "k_pool", "v_pool", "block_table", "kv_args", "sel"):
        if hasattr(c, f):
            setattr(c, f, getattr(c, f).cpu())
    torch.cuda.empty_cache()
    return c


def append_cpu_sample(name: str, budget_s: float):
    """The oracle's append on the host: rows of the workload written into a host pool sized for
    them, as many as take about budget_s; returns (bytes of that sample, seconds, threads)."""
    import oracle
    cfg = {**W.CONFIGS[name], **OVERRIDES}
    T, Hkv, D, P = cfg["T"], cfg["Hkv"], cfg["D"], cfg["page_size"]
    rows = min(T, 512)
    while True:
        pages = max(1, 2 * rows // P + 1)
        c = W.make_append(rows, Hkv, D, P, pages, seed=cfg["seed"])
        kp = c.k_pool.view(torch.int16).numpy().view(np.uint16).copy()
        vp = c.v_pool.view(torch.int16).numpy().view(np.uint16).copy()
        t0 = time.perf_counter()
        oracle.append_paged(c.k_new, c.v_new, kp, vp, c.slot_mapping.numpy(), inplace=True)
        secs = time.perf_counter() - t0
        if secs * 4 > budget_s or rows >= T:
            return c.algorithmic_bytes(), secs, 1, rows
        rows = min(T, rows * 4)


def cpu_baseline(name: str, budget_s: float = 15.0):
    if W.CONFIGS[name]["kind"] == "append":
        nbytes, secs, threads, rows = append_cpu_sample(name, budget_s)
        return {"value": round(nbytes / secs / 1e9, 4), "unit": "GB/s", "cores": threads,
                "kind": "oracle", "sample": f"{rows} appended rows of {name} in {secs:.3f} s"}
    c = cpu_case(name)
    rows, secs, threads = oracle_sample_run(c, budget_s)
    frac = rows / (c.B * c.Hq)
    gbs = c.algorithmic_bytes() * frac / secs / 1e9
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{rows} (b, h) rows of {name} (of {c.B * c.Hq} per call; repeated passes "
                      f"when shorter) in {secs:.2f} s; value = the matching share of the "
                      f"workload's algorithmic bytes / time"}


def workload_config(name: str, **extra):
    """The line's `config`: the workload's name and fields (with any overrides) plus `extra`;
    both arms build it from the same workload, so their configs are equal."""
    return {"workload": name + ("" if not OVERRIDES else " (overridden)"),
            **{k: v for k, v in {**W.CONFIGS[name], **OVERRIDES}.items() if k != "seed"},
            **extra}


def append_shape_bytes(name: str):
    """(algorithmic bytes per call, device bytes per input copy) of an append workload, from its
    fields alone (every slot of the workload is valid)."""
    cfg = {**W.CONFIGS[name], **OVERRIDES}
    T, H, D, P, N = cfg["T"], cfg["Hkv"], cfg["D"], cfg["page_size"], cfg["num_pages"]
    alg = 2 * 2 * T * H * D * 2 + T * 8
    dev = 2 * T * H * D * 2 + T * 8 + 2 * N * H * P * D * 2
    return alg, dev


def l2_note_bytes(alg: int, device_bytes: int) -> str:
    n = copies_for(alg, device_bytes)
    live = n * alg
    where = ("exceed the {:.0f} MB L2" if live > L2_BYTES else
             "fit in the {:.0f} MB L2 (a launch-bound small case)").format(L2_BYTES / 1e6)
    return (f"{n} input copies alternated call by call; their live bytes ({live / 1e6:.1f} MB) "
            f"{where}")


def run_reference(args, world, rank):
    if rank != 0:
        return
    name = args.workload
    threads = os.cpu_count() or 1
    if W.CONFIGS[name]["kind"] == "append":
        times = []
        rows = 0
        for i in range(args.warmup + args.steps):
            nbytes, secs, _, rows = append_cpu_sample(name, 2.0)
            if i >= args.warmup:
                times.append(secs / nbytes)
        per_byte = float(np.mean(times))
        total, dev_bytes = append_shape_bytes(name)
        gbs = 1.0 / per_byte / 1e9
        ms = total * per_byte * 1e3
        cores, dtype = 1, "bf16 copy"
        sample = f"{rows} appended rows per step, scaled to the whole workload"
        cfg = workload_config(name, algorithmic_bytes_per_call=int(total),
                              l2=l2_note_bytes(total, dev_bytes), parallelism=f"replicas x{world}")
    else:
        c = cpu_case(name)
        per_step = max(0.2, 4.0 * args.cpu_budget / max(1, args.steps + args.warmup))
        times = []
        rows_used = 0
        for i in range(args.warmup + args.steps):
            rows, secs, threads = oracle_sample_run(c, per_step)
            if i >= args.warmup:
                times.append(secs / rows)
                rows_used = rows
        per_row = float(np.mean(times))
        secs_full = per_row * c.B * c.Hq
        gbs = c.algorithmic_bytes() / secs_full / 1e9
        ms = secs_full * 1e3
        cores, dtype = threads, "f64"
        sample = (f"{rows_used} (b, h) row computations per step (a call has {c.B * c.Hq} rows; "
                  f"a shorter sample is repeated in whole passes), scaled to the whole workload")
        cfg = workload_config(name, algorithmic_bytes_per_call=int(c.algorithmic_bytes()),
                              l2=l2_note(c), parallelism=f"replicas x{world}")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": dtype, "data": "synthetic", "config": cfg,
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "run": {"executor": "the fp64 oracle on the host cores, as it stands"},
    }
    print(json.dumps(line), flush=True)


def run_native(args, world, rank, local):
    from token_decode_attention_split_gb300 import binding as B_
    B_.load_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    name = args.workload
    c0 = make_case(name, dev, rank=rank, copy=0)
    ncopies = args.copies if args.copies > 0 else input_copies(c0)
    cases = [c0] + [make_case(name, dev, rank=rank, copy=k) for k in range(1, ncopies)]
    if c0.kind == "append":
        ws = None
        outs = [c.k_pool for c in cases]
    else:
        var = {"dense": 0, "paged": 1, "sparse": 2}[c0.kind]
        ws = B_.new_workspace(B_.decode_attn_workspace_size(
            var, c0.B, c0.Hq * getattr(c0, "sq", 1), c0.Hkv, c0.D, getattr(c0, "width", 0)), dev)
        outs = [torch.empty(c.out_shape(), dtype=torch.bfloat16, device=dev) for c in cases]
    stream = torch.cuda.Stream(dev)
    alg = [c.algorithmic_bytes() for c in cases]
    assert len(set(alg)) == 1, "input copies must share their structure"
    bytes_call = float(alg[0])

    def step(i):
        B_.run_case(cases[i % ncopies], out=outs[i % ncopies], workspace=ws, stream=stream)

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i)
    stream.synchronize()

    # ---- K back-to-back calls captured in one CUDA graph (host launch cost stays out of the
    # device number); replayed R times between events on the launching stream
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(args.steps):
            step(i)
    e_a = torch.cuda.Event(enable_timing=True)
    e_b = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        graph.replay()                      # untimed: sizes R
        e_a.record(stream)
        graph.replay()
        e_b.record(stream)
    stream.synchronize()
    per_replay_s = max(e_a.elapsed_time(e_b) * 1e-3, 1e-6)
    replays = int(max(1, math.ceil(args.min_seconds / per_replay_s)))
    if world > 1:
        replays = int(dist_max(float(replays), world, dev))
    warm = int(max(1, math.ceil(min(1.0, args.min_seconds / 4) / per_replay_s)))
    with torch.cuda.stream(stream):
        for _ in range(warm):               # untimed: clocks settle under this load
            graph.replay()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(gpu_selector(dev))
    clocks.start()
    dist_barrier(world)
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(replays):
            graph.replay()
        ev1.record(stream)
    stream.synchronize()
    dist_barrier(world)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall
    clk = clocks.stop()
    calls = args.steps * replays
    total_ms = ev0.elapsed_time(ev1)
    step_ms = dist_max(total_ms / calls, world, dev)
    launch_ms = total_ms / calls            # one kernel launch per call

    # ---- end to end: pinned host inputs copied in and the output copied back every step
    hc = HostCopy(c0)
    h2d = case_bytes_copied(c0)
    d2h = 0 if c0.kind == "append" else outs[0].numel() * 2
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    e2e_steps = max(3, min(args.steps, 20))
    with torch.cuda.stream(stream):
        hc.h2d(stream, cases[0])
        B_.run_case(cases[0], out=outs[0], workspace=ws, stream=stream)
        hc.d2h(outs[0])
    stream.synchronize()
    dist_barrier(world)
    with torch.cuda.stream(stream):
        e_start.record(stream)
        for i in range(e2e_steps):
            j = i % 2
            hc.h2d(stream, cases[j])
            B_.run_case(cases[j], out=outs[j], workspace=ws, stream=stream)
            hc.d2h(outs[j])
        e_end.record(stream)
    stream.synchronize()
    e2e_ms = dist_max(e_start.elapsed_time(e_end) / e2e_steps, world, dev)
    del hc

    peak, peak_kind = measured_peak()
    value = world * bytes_call / (step_ms * 1e-3) / 1e9
    achieved = bytes_call / (launch_ms * 1e-3) / 1e9
    traffic = traffic_record(name)
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_ms, 5),
        "us_per_call": round(step_ms * 1e3, 2),
        "pct_of_peak": round(100.0 * value / world / peak, 2),
        "pct_of_nominal_8tbs": round(100.0 * value / world / NOMINAL_HBM_GBS, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": workload_config(name, algorithmic_bytes_per_call=int(bytes_call),
                                  l2=l2_note(c0) if args.copies <= 0 else
                                  f"{ncopies} input copies alternated (set by --copies)",
                                  parallelism=f"replicas x{world}"),
        "timing": {"graph_calls": args.steps, "replays": replays, "calls_timed": calls,
                   "timed_ms": round(total_ms, 3), "untimed_warm_replays": warm,
                   "input_copies": ncopies},
        "e2e": {"value": round(world * bytes_call / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "ms_per_step": round(e2e_ms, 4)},
        "gpu_launches": calls,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": traffic, "peak_source": f"{peak_kind} hbm_gbs (burst copy)",
                     "kernel": kernel_label({**W.CONFIGS[name], **OVERRIDES}),
                     "timing": f"cuda graph of {args.steps} calls replayed {replays} times",
                     "launch_us": round(launch_ms * 1e3, 3)},
        "clocks": clk,
        "wall_s_timed_region": round(wall, 4),
    }
    if c0.kind == "append":
        line["roofline"]["traffic_note"] = (
            "DRAM reads and the writes that left L2 before the captured launch ended; the "
            "scattered pool writes are mostly still dirty in L2 then, so this is about the reads")
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(name, args.cpu_budget)
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(W.CONFIGS))
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--copies", type=int, default=0,
                    help="input copies to alternate (default: enough to exceed the L2 three "
                         "times over); a small number keeps a profiler capture's memory small")
    ap.add_argument("--min-seconds", type=float, default=4.0,
                    help="length of the timed region (the K-call graph is replayed to fill it)")
    ap.add_argument("--override", action="append", metavar="KEY=VALUE",
                    help="change one field of the workload (e.g. B=8) for a smaller profiling case")
    args = ap.parse_args()
    OVERRIDES.update(parse_overrides(args.override))
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_native(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
