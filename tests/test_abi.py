"""The C ABI on the host, no GPU needed: every symbol the header declares is exported, and
arguments the calls must reject are rejected before anything touches the device."""
import ctypes
import math
import os
import re
import subprocess

import pytest

from token_decode_attention_split_gb300 import binding, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "decode_attn.h")
OK, INVALID, UNSUPPORTED = 0, 1, 2
FAKE = 0x10000          # an aligned non-null address the rejected calls never dereference


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load_library()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(decode_attn_\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("decode_attn_dense", "decode_attn_paged", "decode_attn_sparse",
              "decode_attn_workspace_size", "decode_attn_abi_version"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", binding.library_path()],
                         capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_version_and_status_strings(lib):
    src = open(HEADER).read()
    ver = int(re.search(r"#define DECODE_ATTN_ABI_VERSION (\d+)", src).group(1))
    assert lib.decode_attn_abi_version() == ver
    for s in range(5):
        assert lib.decode_attn_status_string(s)
    assert lib.decode_attn_status_string(99) == b"unknown status"


def dense(lib, q=FAKE, k=FAKE, v=FAKE, out=FAKE, B=1, Hq=8, Hkv=2, D=128, cap=16, k_len=8,
          scale=0.1, ws=FAKE, ws_bytes=1 << 20):
    return lib.decode_attn_dense(q, k, v, out, B, Hq, Hkv, D, cap, k_len, scale, ws, ws_bytes, None)


def paged(lib, B=2, Hq=8, Hkv=2, D=128, P=16, maxp=4, npages=16, stride=1, bt=FAKE, kl=FAKE,
          q=FAKE, scale=0.1):
    return lib.decode_attn_paged(q, FAKE, FAKE, FAKE, bt, maxp, P, npages, kl, stride, B, Hq, Hkv,
                                 D, scale, FAKE, 1 << 20, None)


def sparse(lib, B=2, Hq=8, Hkv=1, D=128, R=100, width=10, sel=FAKE, scale=0.1):
    return lib.decode_attn_sparse(FAKE, FAKE, FAKE, FAKE, R, sel, width, B, Hq, Hkv, D, scale, FAKE,
                                  1 << 20, None)


def test_dense_rejects(lib):
    assert dense(lib, q=None) == INVALID
    assert dense(lib, k=None) == INVALID
    assert dense(lib, ws=None) == INVALID
    assert dense(lib, q=FAKE + 2) == INVALID            # misaligned
    assert dense(lib, Hq=6, Hkv=4) == INVALID            # Hq % Hkv != 0
    assert dense(lib, k_len=17) == INVALID               # k_len > capacity
    assert dense(lib, k_len=-1) == INVALID
    assert dense(lib, cap=0, k_len=0) == INVALID
    assert dense(lib, scale=math.nan) == INVALID
    assert dense(lib, scale=math.inf) == INVALID
    assert dense(lib, D=96) == UNSUPPORTED               # fail closed
    assert dense(lib, D=256) == UNSUPPORTED
    assert dense(lib, Hq=128, Hkv=1) == UNSUPPORTED      # group of 128 heads
    assert dense(lib, cap=1 << 31, k_len=5) == UNSUPPORTED
    assert dense(lib, B=0) == OK                         # empty batch: nothing to do


def test_paged_rejects(lib):
    assert paged(lib, bt=None) == INVALID
    assert paged(lib, kl=None) == INVALID
    assert paged(lib, kl=FAKE + 2) == INVALID
    assert paged(lib, stride=2) == INVALID
    assert paged(lib, maxp=0) == INVALID
    assert paged(lib, npages=0) == INVALID
    assert paged(lib, P=12) == UNSUPPORTED
    assert paged(lib, P=4) == UNSUPPORTED
    assert paged(lib, P=512) == UNSUPPORTED
    assert paged(lib, B=1025) == UNSUPPORTED
    assert paged(lib, D=80) == UNSUPPORTED
    assert paged(lib, B=0) == OK


def test_sparse_rejects(lib):
    assert sparse(lib, width=-1) == INVALID
    assert sparse(lib, R=0) == INVALID
    assert sparse(lib, sel=None) == INVALID
    assert sparse(lib, sel=FAKE + 1) == INVALID
    assert sparse(lib, R=1 << 31) == UNSUPPORTED
    assert sparse(lib, Hq=65, Hkv=1) == UNSUPPORTED
    assert sparse(lib, B=0) == OK


def test_misc_host_calls(lib):
    assert lib.decode_attn_set_grid_limit(-1) == INVALID
    assert lib.decode_attn_set_grid_limit(0) == OK
    assert lib.decode_attn_workspace_init(None, 0, None) == OK
    assert lib.decode_attn_workspace_init(None, 16, None) == INVALID
    assert lib.decode_attn_read_device_error(None) == INVALID
    assert lib.decode_attn_check_wait_timeout(0, None) == INVALID
    assert lib.decode_attn_check_wait_timeout(1000001, None) == INVALID
    # sizes the calls would reject have no workspace size
    assert lib.decode_attn_workspace_size(0, 1, 6, 4, 128, 0) == 0
    assert lib.decode_attn_workspace_size(2, 1, 8, 1, 96, 10) == 0
    assert lib.decode_attn_workspace_size(7, 1, 8, 1, 128, 10) == 0


def test_append_rejects(lib):
    def ap(k=FAKE, sm=FAKE, T=4, Hkv=2, D=128, P=16, npages=8):
        return lib.decode_attn_append_paged(k, FAKE, FAKE, FAKE, sm, T, Hkv, D, P, npages, None)

    def ar(pos=FAKE, B=2, D=128, R=64, window=16):
        return lib.decode_attn_append_ring(FAKE, FAKE, FAKE, FAKE, pos, B, 2, D, R, window, None)

    assert ap(k=None) == INVALID
    assert ap(sm=None) == INVALID
    assert ap(sm=FAKE + 4) == INVALID          # slot words must be 8-byte aligned
    assert ap(T=-1) == INVALID
    assert ap(P=0) == INVALID
    assert ap(D=100) == UNSUPPORTED
    assert ap(T=0) == OK                      # nothing to write
    assert ar(window=0) == INVALID
    assert ar(window=65) == INVALID           # window larger than the pool
    assert ar(pos=None) == INVALID
    assert ar(B=0) == OK


Spec = binding.DecodeAttnSpec     # the ABI's decode_attn_spec layout


def test_flash_spec_gate(lib):
    """Which options disqualify the flash arm (tests/golden/flash_spec_gate.json)."""
    import json
    rule = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "flash_spec_gate.json")))
    lib.decode_attn_spec_check.restype = ctypes.c_int
    assert lib.decode_attn_spec_check(ctypes.byref(Spec(softmax_scale=0.125))) == OK
    for f in rule["accepted_and_ignored"]:
        s = Spec(softmax_scale=0.125)
        setattr(s, f, 1)
        assert lib.decode_attn_spec_check(ctypes.byref(s)) == OK, f
    for f in rule["disqualify"]:
        s = Spec(softmax_scale=0.125, causal=1)
        setattr(s, f, 1)
        assert lib.decode_attn_spec_check(ctypes.byref(s)) == UNSUPPORTED, f
    assert lib.decode_attn_spec_check(None) == INVALID
    assert lib.decode_attn_spec_check(ctypes.byref(Spec(softmax_scale=math.nan))) == INVALID
    # the spec entry point refuses before touching any (here fake) device pointer
    lib.decode_attn_dense_spec.restype = ctypes.c_int
    s = Spec(softmax_scale=0.1, has_softcap=1)
    assert lib.decode_attn_dense_spec(ctypes.byref(s), FAKE, FAKE, FAKE, FAKE, 1, 8, 2, 128,
                                      ctypes.c_int64(16), ctypes.c_int64(8), FAKE,
                                      ctypes.c_size_t(1 << 20), None) == UNSUPPORTED


def test_dense_device_len_rejects(lib):
    lib.decode_attn_dense_device_len.restype = ctypes.c_int
    call = lambda kl, cap=16: lib.decode_attn_dense_device_len(
        FAKE, FAKE, FAKE, FAKE, 1, 8, 2, 128, ctypes.c_int64(cap), kl, ctypes.c_float(0.1), FAKE,
        ctypes.c_size_t(1 << 20), None)
    assert call(None) == INVALID
    assert call(FAKE + 2) == INVALID        # the length word must be 4-byte aligned
    assert call(FAKE, cap=0) == INVALID


def test_multitoken_rejects(lib):
    lib.decode_attn_dense_mq.restype = ctypes.c_int
    call = lambda Hq, Hkv, Sq: lib.decode_attn_dense_mq(
        FAKE, FAKE, FAKE, FAKE, 1, Hq, Hkv, 128, Sq, 1, ctypes.c_int64(64), ctypes.c_int64(32),
        ctypes.c_float(0.1), FAKE, ctypes.c_size_t(1 << 20), None)
    assert call(8, 2, 0) == INVALID          # no query token
    assert call(64, 2, 3) == UNSUPPORTED     # 32 heads x 3 tokens > 64 columns per unit


def test_binding_has_every_declared_call():
    """The Python binding exposes each C entry point under the same name."""
    for name in declared_functions():
        assert hasattr(binding, name), name


def test_binding_spec_gate_without_gpu(lib):
    S = binding.DecodeAttnSpec
    assert binding.decode_attn_spec_check(S(softmax_scale=0.125)) == OK
    assert binding.decode_attn_spec_check(S(causal=1, softmax_scale=0.125)) == OK
    for field in ("has_alibi", "has_window_left", "has_window_right", "has_softcap"):
        assert binding.decode_attn_spec_check(S(softmax_scale=0.125, **{field: 1})) == UNSUPPORTED
    assert binding.decode_attn_spec_check(S(softmax_scale=math.inf)) == INVALID
    assert binding.decode_attn_status_string(UNSUPPORTED)


def test_sparse_workspace_size_formula(lib):
    """Sparse calls need no device to size their workspace: one u32 counter per unit (B * Hkv),
    then the LSEs and the fp32 partial rows of units * ceil(width / 512) segments of G heads
    (the chunk of 512 selection entries is the same for both sparse kernels and depends on
    nothing else), each region starting on a 256-byte boundary."""
    def expect(B, Hq, Hkv, D, width):
        G, units = Hq // Hkv, B * Hkv
        segs = units * -(-width // 512)
        up = lambda x: -(-x // 256) * 256
        lse = up(units * 4)
        o = lse + up(segs * G * 4)
        return max(o + segs * G * D * 4, 256)
    for B, Hq, Hkv, D, width in [(32, 64, 1, 128, 2048),   # the sparse workload: 4 MB of rows
                                 (3, 48, 1, 64, 700), (2, 16, 2, 128, 1), (5, 8, 8, 64, 513),
                                 (1, 64, 2, 128, 0)]:
        assert lib.decode_attn_workspace_size(2, B, Hq, Hkv, D, width) == expect(B, Hq, Hkv, D, width)
    assert lib.decode_attn_workspace_size(2, 32, 64, 1, 128, 2048) > 4 * 2 ** 20
