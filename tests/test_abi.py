"""The C-ABI library on the CPU: it builds, loads, exports every declared
symbol, and its host-only paths (validation, planning, sizing) behave.

No call here launches a kernel: every call either is pure host arithmetic
or fails validation before anything touches the device.
"""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from paged_kv_decode_np_gb300 import build_lib
    path = build_lib.build()
    import paged_kv_decode_np_gb300 as npg
    return npg.load(path)


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names |= set(re.findall(r"^[A-Za-z_][\w\s\*]*?\b(np_\w+)\s*\(", src, flags=re.M))
    return sorted(names)


def test_header_declares_the_calls():
    names = _declared()
    for must in ("np_kv_append", "np_paged_decode", "np_paged_decode_reduce",
                 "np_paged_decode_workspace_bytes", "np_paged_decode_plan",
                 "np_paged_decode_split_len", "np_status_string", "np_abi_version"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_abi_version_and_status_strings(lib):
    hdr = open(os.path.join(ROOT, "include", "np_paged.h")).read()
    ver = int(re.search(r"#define NP_ABI_VERSION (\d+)", hdr).group(1))
    assert lib.np_abi_version() == ver
    for code, name in [(0, "NP_OK"), (1, "NP_ERR_INVALID_ARG"), (2, "NP_ERR_UNSUPPORTED"),
                       (3, "NP_ERR_WORKSPACE"), (4, "NP_ERR_OUT_OF_RANGE"), (5, "NP_ERR_CUDA"),
                       (99, "NP_ERR_UNKNOWN")]:
        assert lib.np_status_string(code).decode() == name


def _decode(lib, **kw):
    a = dict(out=None, q=None, k=None, v=None, dtype=0, nb=16, bs=16, hk=2, d=128, bt=None,
             mb=4, cl=None, rows=2, qlen=1, hq=4, scale=0.1, splits=1, ws=None, wsb=0, err=None)
    a.update(kw)
    return lib.np_paged_decode(a["out"], a["q"], a["k"], a["v"], a["dtype"], a["nb"], a["bs"],
                               a["hk"], a["d"], a["bt"], a["mb"], a["cl"], a["rows"], a["qlen"],
                               a["hq"], a["scale"], a["splits"], a["ws"], a["wsb"], a["err"], None)


FAKE = 0x10000  # a 16-byte aligned address that is never dereferenced


def test_decode_validation(lib):
    ok_ptrs = dict(out=FAKE, q=FAKE, k=FAKE, v=FAKE, bt=FAKE, cl=FAKE)
    assert _decode(lib, hq=3, **ok_ptrs) == 1          # q_heads % kv_heads
    assert _decode(lib, d=48, **ok_ptrs) == 2          # head_dim not compiled
    assert _decode(lib, hk=1, hq=9, **ok_ptrs) == 2    # fp32: group > 8
    # fp32: any group <= 8 passes validation (without a GPU the launch then
    # fails with NP_ERR_CUDA)
    assert _decode(lib, hk=1, hq=3, **ok_ptrs) in (0, 5)
    assert _decode(lib, hk=1, hq=17, dtype=1, **ok_ptrs) == 2  # bf16: group > 16
    # bf16: any group <= 16 passes validation (on a machine without a GPU the
    # launch itself then fails with NP_ERR_CUDA)
    assert _decode(lib, hk=1, hq=3, dtype=1, **ok_ptrs) in (0, 5)
    assert _decode(lib, dtype=7, **ok_ptrs) == 2       # dtype
    assert _decode(lib, scale=float("nan"), **ok_ptrs) == 1
    assert _decode(lib, splits=-1, **ok_ptrs) == 1
    assert _decode(lib, splits=0, **ok_ptrs) == 3            # balanced read: needs workspace
    assert _decode(lib, splits=0, dtype=1, hk=6, hq=12, **ok_ptrs) == 3  # any kv heads
    assert _decode(lib, splits=0, dtype=1, hk=1, hq=8, bs=4, **ok_ptrs) == 2  # box x heads % 8
    assert _decode(lib, splits=0, dtype=1, hk=4, hq=8, bs=3, **ok_ptrs) == 2  # bf16 4 heads: odd bs
    assert _decode(lib, splits=0, dtype=1, hk=4, hq=8, nb=16, **ok_ptrs) == 3  # no workspace
    assert _decode(lib, splits=0, dtype=1, hk=8, hq=16, nb=16, **ok_ptrs) == 3  # no workspace
    assert _decode(lib, bs=0, **ok_ptrs) == 1
    assert _decode(lib, nb=0, **ok_ptrs) == 1
    assert _decode(lib, rows=-1, **ok_ptrs) == 1
    assert _decode(lib) == 1                           # null pointers
    assert _decode(lib, rows=0) == 0                   # nothing to do
    assert _decode(lib, **dict(ok_ptrs, q=FAKE + 4)) == 1   # misaligned
    assert _decode(lib, **dict(ok_ptrs, out=None)) == 1     # out needed unsplit
    assert _decode(lib, splits=4, **ok_ptrs) == 3            # no workspace
    assert _decode(lib, splits=4, ws=FAKE, wsb=100, **ok_ptrs) == 3
    assert _decode(lib, nb=2**62, **ok_ptrs) == 4            # pool bytes overflow
    assert _decode(lib, qlen=0, **ok_ptrs) == 1              # no query token
    assert _decode(lib, qlen=2, **ok_ptrs) in (0, 5)         # fp32: 4 rows on the split grid
    assert _decode(lib, qlen=5, **ok_ptrs) == 2              # fp32: g*query_len > 8
    assert _decode(lib, mb=2**20, bs=2**12, **ok_ptrs) == 2  # fp32: positions past int32
    assert _decode(lib, qlen=2, splits=0, hk=8, hq=16, **ok_ptrs) == 3  # balanced: needs workspace
    assert _decode(lib, qlen=5, splits=0, hk=8, hq=16, **ok_ptrs) == 2  # fp32: g*query_len > 8
    assert _decode(lib, qlen=9, dtype=1, **ok_ptrs) == 2     # bf16: g*query_len > 16
    assert _decode(lib, qlen=8, dtype=1, splits=4, **ok_ptrs) == 3   # workspace missing


def _noalloc(lib, **kw):
    a = dict(out=FAKE, q=FAKE, k=FAKE, v=FAKE, dtype=1, nb=16, bs=16, hk=8, d=128, bt=FAKE,
             mb=4, cl=FAKE, rows=2, qlen=1, hq=16, scale=0.1, splits=4, err=None)
    a.update(kw)
    return lib.np_paged_decode_noalloc(a["out"], a["q"], a["k"], a["v"], a["dtype"], a["nb"],
                                       a["bs"], a["hk"], a["d"], a["bt"], a["mb"], a["cl"],
                                       a["rows"], a["qlen"], a["hq"], a["scale"], a["splits"],
                                       a["err"], None)


def test_noalloc_validation_precedes_the_scratch_check(lib):
    """Sizes np_paged_decode refuses get its codes from the no-allocation
    entry point too -- never NP_ERR_WORKSPACE -- and rows * query_len is
    never formed for them; only valid shapes reach the scratch-size check.
    Every call here returns before touching the device."""
    assert _noalloc(lib, rows=70000) == 2                   # rows past the grid limit
    assert _noalloc(lib, rows=2**31 - 1, qlen=16) == 2      # the product would overflow int32
    assert _noalloc(lib, qlen=17) == 2
    assert _noalloc(lib, qlen=0) == 1
    assert _noalloc(lib, rows=-1) == 1
    assert _noalloc(lib, splits=-1) == 1
    assert _noalloc(lib, splits=70000) == 1
    assert _noalloc(lib, hq=0) == 1
    assert _noalloc(lib, d=0) == 1
    assert _noalloc(lib, rows=0) == 0                       # nothing to do
    assert _noalloc(lib, out=None) == 1                     # out is always written
    assert _noalloc(lib, out=FAKE + 4) == 1
    # a valid shape whose partials exceed the array
    per = 2 * 16 * 4 * 129
    assert _noalloc(lib, splits=(32 << 20) // per + 1) == 3
    assert _noalloc(lib, splits=1, hq=17) == 1              # one split: np_paged_decode's checks


def test_append_validation(lib):
    f = lib.np_kv_append
    assert f(FAKE, FAKE, 0, 16, 16, 2, 128, FAKE, FAKE, FAKE, 0, None, None) == 0  # no tokens
    assert f(None, FAKE, 0, 16, 16, 2, 128, FAKE, FAKE, FAKE, 3, None, None) == 1
    assert f(FAKE, FAKE, 5, 16, 16, 2, 128, FAKE, FAKE, FAKE, 3, None, None) == 2
    assert f(FAKE, FAKE, 1, 16, 16, 1, 3, FAKE, FAKE, FAKE, 3, None, None) == 2   # row % 16
    assert f(FAKE, FAKE, 0, 16, 16, 2, 128, FAKE + 8, FAKE, FAKE, 3, None, None) == 1
    assert f(FAKE, FAKE, 0, 16, 16, 2, 128, FAKE, FAKE, FAKE, -1, None, None) == 1
    assert f(FAKE, FAKE, 0, 2**62, 16, 2, 128, FAKE, FAKE, FAKE, 3, None, None) == 4


def test_reduce_validation(lib):
    f = lib.np_paged_decode_reduce
    assert f(FAKE, 0, FAKE, 10**6, 2, 4, 128, 1, None) == 1      # one split: nothing to merge
    assert f(FAKE, 0, None, 0, 2, 4, 128, 4, None) == 3
    assert f(FAKE, 0, FAKE, 8, 2, 4, 128, 4, None) == 3
    assert f(FAKE, 0, FAKE, 10**6, 2, 4, 100, 4, None) == 2
    assert f(FAKE, 9, FAKE, 10**6, 2, 4, 128, 4, None) == 2
    assert f(FAKE, 0, FAKE, 10**6, 0, 4, 128, 4, None) == 0


def test_workspace_bytes(lib):
    f = lib.np_paged_decode_workspace_bytes
    assert f(4, 8, 128, 1) == 0
    assert f(4, 8, 128, 0) > 0  # the balanced read's partials and counters
    n_o = 4 * 8 * 3 * 128 * 4
    n_l = 4 * 8 * 3 * 4
    assert f(4, 8, 128, 3) == (n_o + 255) // 256 * 256 + (n_l + 255) // 256 * 256


@pytest.mark.parametrize("bs,mb,s", [(16, 128, 1), (16, 128, 3), (8, 2048, 26), (32, 4096, 128),
                                     (1, 7, 2), (100, 3, 2), (128, 64, 5)])
def test_split_len_covers_the_table(lib, bs, mb, s):
    sl = lib.np_paged_decode_split_len(bs, mb, s)
    cap = bs * mb
    assert sl * s >= cap
    assert sl % (bs if bs > 64 else 64) == 0
    assert (s - 1) * sl < cap + sl


def test_plan_is_static_and_sane(lib):
    import paged_kv_decode_np_gb300 as npg
    import workloads as wl
    for w in wl.WORKLOADS.values():
        s = npg.np_paged_decode_plan(w.rows, w.q_heads, w.kv_heads, w.head_dim, w.block_size,
                                     w.max_blocks_per_row, w.torch_dtype, num_sms=152)
        cap = w.max_blocks_per_row * w.block_size
        if s == 0:  # the balanced read: head_dim % 64 (bf16) or % 32 (fp32), <= 256
            assert w.head_dim <= 256
            assert w.head_dim % (64 if w.dtype == "bf16" else 32) == 0
            continue
        sl = npg.np_paged_decode_split_len(w.block_size, w.max_blocks_per_row, s)
        assert s >= 1 and sl * s >= cap
        if s > 1:  # each split reads at least 64 tokens' worth of every head group
            assert sl >= 64
    for name in ("bf16-mqa", "bf16-kv2", "llama-fp32-kv16"):  # any kv head count
        w = wl.WORKLOADS[name]
        assert npg.np_paged_decode_plan(w.rows, w.q_heads, w.kv_heads, w.head_dim, w.block_size,
                                        w.max_blocks_per_row, w.torch_dtype, num_sms=152) == 0
    # same shapes, same plan (no hidden state)
    a = npg.np_paged_decode_plan(16, 64, 8, 128, 32, 4096, "bf16", num_sms=152)
    assert a == npg.np_paged_decode_plan(16, 64, 8, 128, 32, 4096, "bf16", num_sms=152)


def test_binding_refuses_cpu_tensors():
    import torch

    import paged_kv_decode_np_gb300 as npg
    q = torch.zeros(2, 4, 128)
    kp = torch.zeros(4, 16, 2, 128)
    with pytest.raises(ValueError, match="CUDA"):
        npg.np_paged_decode(torch.zeros_like(q), q, kp, kp, torch.zeros(2, 4, dtype=torch.int32),
                            torch.zeros(2, dtype=torch.int32), 0.1)


def test_product_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "paged_kv_decode_np_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"(import\s+oracle|from\s+oracle|np_oracle|npo_)", src), f
