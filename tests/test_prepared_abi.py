"""PreparedStep passes the C library exactly the arguments the checked
binding passes (pointer, integer and float types included), with a stub
library built here by gcc in place of the CUDA one: each stub entry point
prints its arguments as it received them, and the two paths' records must
match.  CPU only; the GPU parity of PreparedStep is in test_parity_gpu.py.
"""
import ctypes
import os
import shutil
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import paged_kv_decode_np_gb300 as npg  # noqa: E402

STUB = r"""
#include <stdint.h>
#include <stddef.h>
#include <stdio.h>
static char rec[4096];
const char* stub_last(void) { return rec; }
const char* np_status_string(int s) { (void)s; return "stub"; }
int32_t np_abi_version(void) { return 0; }
int np_kv_append(void) { return 0; }
int np_paged_decode_plan(void) { return 0; }
int64_t np_paged_decode_split_len(void) { return 0; }
size_t np_paged_decode_workspace_bytes(void) { return 0; }
int np_paged_decode(void) { return 0; }
int np_paged_decode_noalloc(void) { return 0; }
int np_selftest_bounded_wait(void) { return 0; }
int np_paged_append_decode(void* out, const void* q, const void* kn, const void* vn,
                           const int64_t* sm, void* kp, void* vp, int dtype, int64_t nb,
                           int32_t bs, int32_t hk, int32_t d, const int32_t* bt, int32_t mb,
                           const int32_t* cl, int32_t rows, int32_t qn, int32_t hq,
                           float scale, int32_t ns, void* ws, size_t wsb, int32_t* err,
                           void* stream) {
  snprintf(rec, sizeof rec,
           "append_decode %p %p %p %p %p %p %p %d %lld %d %d %d %p %d %p %d %d %d %.9g %d %p "
           "%zu %p %p",
           out, q, kn, vn, (const void*)sm, kp, vp, dtype, (long long)nb, bs, hk, d,
           (const void*)bt, mb, (const void*)cl, rows, qn, hq, (double)scale, ns, ws, wsb,
           (void*)err, stream);
  return 0;
}
int np_paged_decode_reduce(void* out, int dtype, const void* ws, size_t wsb, int32_t rows,
                           int32_t hq, int32_t d, int32_t ns, void* stream) {
  snprintf(rec, sizeof rec, "reduce %p %d %p %zu %d %d %d %d %p", out, dtype, ws, wsb, rows,
           hq, d, ns, stream);
  return 0;
}
"""


@pytest.fixture()
def stub(tmp_path, monkeypatch):
    if shutil.which("gcc") is None:
        pytest.skip("gcc is needed to build the stub library")
    src = tmp_path / "stub.c"
    src.write_text(STUB)
    so = tmp_path / "libstub.so"
    subprocess.check_call(["gcc", "-O1", "-shared", "-fPIC", "-o", str(so), str(src)])
    lib = npg.load(str(so))
    lib.stub_last.restype = ctypes.c_char_p
    monkeypatch.setattr(npg, "_LIB", lib)
    # CPU tensors stand in for device ones: only their addresses are passed
    monkeypatch.setattr(npg, "_dev", lambda t, name, cur: t.data_ptr())
    monkeypatch.setattr(npg, "_stream", lambda s: 0x5151)
    return lib


def _tensors(splits):
    rows, hq, hk, d, bs, nb, mb = 3, 8, 2, 64, 16, 40, 12
    q = torch.randn(rows, hq, d)
    return dict(out=torch.empty_like(q), q=q, k_new=torch.randn(rows, hk, d),
                v_new=torch.randn(rows, hk, d), slot_mapping=torch.arange(rows) * 7,
                k_pool=torch.randn(nb, bs, hk, d), v_pool=torch.randn(nb, bs, hk, d),
                block_tables=torch.zeros(rows, mb, dtype=torch.int32),
                context_lens=torch.tensor([5, 100, 17], dtype=torch.int32),
                scale=0.123456789, num_splits=splits,
                workspace=torch.empty(4096, dtype=torch.uint8),
                err_word=torch.zeros(1, dtype=torch.int32))


@pytest.mark.parametrize("splits", [0, 1, 4])
def test_prepared_step_passes_the_same_arguments(stub, splits):
    t = _tensors(splits)
    order = ["q", "k_new", "v_new", "slot_mapping", "k_pool", "v_pool", "block_tables",
             "context_lens", "scale", "num_splits", "workspace", "err_word"]
    out_arg = t["out"] if splits <= 1 else None
    npg.np_paged_append_decode(out_arg, *[t[k] for k in order], None)
    direct = [stub.stub_last().decode()]
    if splits > 1:
        npg.np_paged_decode_reduce(t["out"], t["workspace"], splits, None)
        direct.append(stub.stub_last().decode())
    step = npg.PreparedStep(t["out"], *[t[k] for k in order], None)
    prepared = []
    for name, fn, cargs in step._calls:  # one call at a time, as launch() makes them
        assert fn(*cargs) == 0
        prepared.append(stub.stub_last().decode())
    assert prepared == direct
    assert "0.123456791" in direct[0]  # the scale reached C as a float
    assert step.launch() == (2 if splits == 0 else 1) + (1 if splits > 1 else 0)
