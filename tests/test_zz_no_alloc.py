"""np_paged_decode_noalloc: the split read for callers that cannot allocate.

Some callers are handed only their input and output buffers and a stream
(a host framework calling this library as a plugin without exposing its
allocator, or a serving loop that must not call cudaMalloc once it runs), so
they cannot supply the split workspace.  This entry point keeps the split
partials in a fixed array inside the library instead.  The tests drive it
through the C ABI and check every output element against the oracle at the
parity tolerance, and against the workspace entry points
(np_paged_decode + np_paged_decode_reduce, or the balanced read with a caller
workspace), on calls in a row with different shapes -- the shared array
keeps the previous call's contents, so a stale-data bug would show on the
later calls.

The file name sorts last so that a run stopping at the first failure has
already run every other test; it also passes alone in a fresh process.
"""
import pytest
import torch

import workloads as wl
from step_helpers import assert_parity, host_inputs, oracle_step

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _case(contexts, q_heads, kv_heads, block_size, dtype, seed, query_len=1, head_dim=128):
    # every slot holds finite values: this entry point reads, it does not
    # append, so the rows' newest positions are read as they are
    w = wl.Workload(f"noalloc-{seed}", rows=len(contexts), q_heads=q_heads, kv_heads=kv_heads,
                    head_dim=head_dim, block_size=block_size, dtype=dtype,
                    ctx=("fixed", tuple(contexts)), pool=("spare", 2), seed=seed,
                    query_len=query_len)
    inp = wl.make_inputs(w, device=DEV, poison=False)
    bt, cl = inp.block_tables.to(DEV), inp.context_lens.to(DEV)
    return w, inp, bt, cl


def _oracle(w, inp):
    ref, _ = oracle_step(host_inputs(inp), w.softmax_scale, append=False)
    return ref


def _with_workspace(npg, w, inp, bt, cl, splits):
    ws = npg.workspace(w.rows, w.q_heads, w.head_dim, splits, device=DEV,
                       query_len=w.query_len)
    out = torch.empty_like(inp.q)
    if splits == 0:
        npg.np_paged_decode(out, inp.q, inp.k_pool, inp.v_pool, bt, cl, w.softmax_scale, 0, ws)
    else:
        npg.np_paged_decode(None, inp.q, inp.k_pool, inp.v_pool, bt, cl, w.softmax_scale,
                            splits, ws)
        npg.np_paged_decode_reduce(out, ws, splits)
    torch.cuda.synchronize()
    return out


def _noalloc(npg, w, inp, bt, cl, splits):
    out = torch.full_like(inp.q, float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    npg.np_paged_decode_noalloc(out, inp.q, inp.k_pool, inp.v_pool, bt, cl, w.softmax_scale,
                                splits, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return out


def test_noalloc_split_read_against_the_oracle_calls_in_a_row(nplib):
    """Split reads (bf16 and fp32, one and two query tokens per row) one
    after another through the shared array: each matches the oracle, and
    the workspace entry points' result bit for bit (the same kernels)."""
    cases = [
        (_case([33, 2000, 700, 5, 1500], 40, 8, 32, "bf16", seed=81), 7),
        (_case([900, 1, 64, 3100], 32, 8, 16, "f32", seed=82), 12),
        (_case([2, 300, 4100, 77], 32, 8, 16, "bf16", seed=87, query_len=2), 5),
        (_case([33, 2000, 700, 5, 1500], 40, 8, 32, "bf16", seed=81), 3),
    ]
    for (w, inp, bt, cl), splits in cases:
        ref = _oracle(w, inp)
        out = _noalloc(nplib, w, inp, bt, cl, splits)
        assert_parity(out, ref, w.dtype, f"noalloc {w.name} splits={splits}")
        assert torch.equal(out, _with_workspace(nplib, w, inp, bt, cl, splits))


def test_noalloc_rejects_partials_larger_than_its_scratch(nplib):
    w, inp, bt, cl = _case([100, 200], 64, 8, 32, "bf16", seed=83)
    per_split = nplib.np_paged_decode_workspace_bytes(w.rows, w.q_heads, w.head_dim, 1000)
    assert per_split > nplib.NP_NOALLOC_SCRATCH_BYTES // 2
    too_many = 1 + nplib.NP_NOALLOC_SCRATCH_BYTES // (w.rows * w.q_heads * 4 * (w.head_dim + 1))
    out = torch.full_like(inp.q, float("nan"))
    with pytest.raises(nplib.NPError) as e:
        nplib.np_paged_decode_noalloc(out, inp.q, inp.k_pool, inp.v_pool, bt, cl,
                                      w.softmax_scale, too_many)
    assert e.value.status == nplib.NP_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.isnan(out.float()).all()  # refused before anything ran


def test_noalloc_balanced_read(nplib):
    """num_splits = 0: the balanced read keeps its cut-row partials in the
    library's array (head_dim 128 fits, 256 does not); matches the oracle
    and the same read with a caller workspace, bit for bit."""
    for (w, inp, bt, cl) in (_case([33, 2000, 700, 5, 1500], 40, 8, 32, "bf16", seed=84),
                             _case([900, 1, 64, 3100], 32, 8, 16, "f32", seed=85),
                             _case([5000, 3, 260], 32, 8, 16, "bf16", seed=88, query_len=3)):
        ref = _oracle(w, inp)
        out = _noalloc(nplib, w, inp, bt, cl, 0)
        assert_parity(out, ref, w.dtype, f"noalloc balanced {w.name}")
        assert torch.equal(out, _with_workspace(nplib, w, inp, bt, cl, 0))
    w, inp, bt, cl = _case([40, 70], 16, 8, 16, "bf16", seed=86, head_dim=256)
    with pytest.raises(nplib.NPError) as e:
        nplib.np_paged_decode_noalloc(torch.empty_like(inp.q), inp.q, inp.k_pool, inp.v_pool,
                                      bt, cl, w.softmax_scale, 0)
    assert e.value.status == nplib.NP_ERR_WORKSPACE
