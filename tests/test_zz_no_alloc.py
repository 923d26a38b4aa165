"""np_paged_decode_noalloc: the split read for callers that cannot allocate.

Some callers are handed only their input and output buffers and a stream
(a host framework calling this library as a plugin without exposing its
allocator, or a serving loop that must not call cudaMalloc once it runs), so
they cannot supply the split workspace.  This entry point keeps the split
partials in a fixed array inside the library instead.  The test drives it
through the C ABI and checks it against the workspace entry points
(np_paged_decode + np_paged_decode_reduce) at the parity tolerance, on two
calls in a row with different shapes -- the shared array keeps the previous
call's contents, so a stale-data bug would show on the second call.

The file name sorts last so that a run stopping at the first failure has
already run every other test; it also passes alone in a fresh process.
"""
import pytest
import torch

import workloads as wl
from step_helpers import assert_parity

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _case(contexts, q_heads, kv_heads, block_size, dtype, seed, poison=True):
    w = wl.Workload(f"noalloc-{seed}", rows=len(contexts), q_heads=q_heads, kv_heads=kv_heads,
                    head_dim=128, block_size=block_size, dtype=dtype,
                    ctx=("fixed", tuple(contexts)), pool=("spare", 2), seed=seed)
    inp = wl.make_inputs(w, device=DEV, poison=poison)
    bt, cl = inp.block_tables.to(DEV), inp.context_lens.to(DEV)
    return w, inp, bt, cl


def _with_workspace(npg, w, inp, bt, cl, splits):
    ws = npg.workspace(w.rows, w.q_heads, w.head_dim, splits, device=DEV)
    out = torch.empty_like(inp.q)
    npg.np_paged_decode(None, inp.q, inp.k_pool, inp.v_pool, bt, cl, w.softmax_scale,
                        splits, ws)
    npg.np_paged_decode_reduce(out, ws, splits)
    torch.cuda.synchronize()
    return out


def test_noalloc_matches_workspace_entry_points_two_calls(nplib):
    cases = [
        (_case([33, 2000, 700, 5, 1500], 40, 8, 32, "bf16", seed=81), 7),
        (_case([900, 1, 64, 3100], 32, 8, 16, "f32", seed=82), 12),
    ]
    for (w, inp, bt, cl), splits in cases:
        ref = _with_workspace(nplib, w, inp, bt, cl, splits)
        out = torch.full_like(inp.q, float("nan"))
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        nplib.np_paged_decode_noalloc(out, inp.q, inp.k_pool, inp.v_pool, bt, cl,
                                      w.softmax_scale, splits, err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_parity(out, ref.double().cpu().numpy(), w.dtype, f"noalloc {w.name}")


def test_noalloc_rejects_partials_larger_than_its_scratch(nplib):
    w, inp, bt, cl = _case([100, 200], 64, 8, 32, "bf16", seed=83)
    per_split = nplib.np_paged_decode_workspace_bytes(w.rows, w.q_heads, w.head_dim, 1000)
    assert per_split > nplib.NP_NOALLOC_SCRATCH_BYTES // 2
    too_many = 1 + nplib.NP_NOALLOC_SCRATCH_BYTES // (w.rows * w.q_heads * 4 * (w.head_dim + 1))
    out = torch.empty_like(inp.q)
    with pytest.raises(nplib.NPError) as e:
        nplib.np_paged_decode_noalloc(out, inp.q, inp.k_pool, inp.v_pool, bt, cl,
                                      w.softmax_scale, too_many)
    assert e.value.status == nplib.NP_ERR_WORKSPACE


def test_noalloc_balanced_read(nplib):
    """num_splits = 0: the balanced read keeps its cut-row partials in the
    library's array (head_dim 128 fits, 256 does not)."""
    for (w, inp, bt, cl) in (_case([33, 2000, 700, 5, 1500], 40, 8, 32, "bf16", seed=84,
                                   poison=False),
                             _case([900, 1, 64, 3100], 32, 8, 16, "f32", seed=85,
                                   poison=False)):
        ws = nplib.workspace(w.rows, w.q_heads, w.head_dim, 0, device=DEV)
        ref = torch.empty_like(inp.q)
        nplib.np_paged_decode(ref, inp.q, inp.k_pool, inp.v_pool, bt, cl, w.softmax_scale, 0, ws)
        out = torch.full_like(inp.q, float("nan"))
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        nplib.np_paged_decode_noalloc(out, inp.q, inp.k_pool, inp.v_pool, bt, cl,
                                      w.softmax_scale, 0, err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert torch.isfinite(out.float()).all()
        assert torch.equal(out, ref)  # the same launches, bit for bit
    w = wl.Workload("noalloc-d256", rows=2, q_heads=16, kv_heads=8, head_dim=256, block_size=16,
                    dtype="bf16", ctx=("fixed", (40, 70)), pool=("spare", 2), seed=86)
    inp = wl.make_inputs(w, device=DEV)
    with pytest.raises(nplib.NPError) as e:
        nplib.np_paged_decode_noalloc(torch.empty_like(inp.q), inp.q, inp.k_pool, inp.v_pool,
                                      inp.block_tables.to(DEV), inp.context_lens.to(DEV),
                                      w.softmax_scale, 0)
    assert e.value.status == nplib.NP_ERR_WORKSPACE
