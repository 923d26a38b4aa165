"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle.

Every test here drives libnp_paged.so through the Python binding and
compares element by element with the oracle on the same seeded bytes:
fp32 within atol 1e-5 + rtol 1e-4, bf16 within atol 2e-2, appends bit for bit.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import golden_cases
import oracle
import workloads as wl
from step_helpers import (assert_parity, assert_pool_equal, gpu_step, host_inputs, oracle_append,
                          oracle_step, oracle_step_in_place, to64)

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _custom(contexts, q_heads, kv_heads, head_dim, block_size, dtype, seed=11, spare=3,
            scale=None, query_len=1):
    return wl.Workload(f"custom-{seed}", rows=len(contexts), q_heads=q_heads,
                       kv_heads=kv_heads, head_dim=head_dim, block_size=block_size,
                       dtype=dtype, ctx=("fixed", tuple(contexts)), pool=("spare", spare),
                       seed=seed, scale=scale, query_len=query_len)


def _full_parity(npg, w, num_splits=None, append=True, device=DEV, fused=True):
    """The step (append + read [+ reduce]) against the oracle; by default the
    append runs fused in the read's launch, fused=False uses np_kv_append.
    The pools after the step must equal the oracle's append bit for bit."""
    inp = wl.make_inputs(w, device="cpu")
    host = wl.full_host(inp)
    dinp = wl.Inputs(w, inp.md, *(t.to(device) for t in
                                  (inp.q, inp.k_pool, inp.v_pool, inp.k_new, inp.v_new)))
    out, s, _ = gpu_step(npg, dinp, num_splits=num_splits, append=append, fused=fused)
    ref, _ = oracle_step(host, w.softmax_scale, append=append)
    if append:
        rk, rv = host["k_pool"].copy(), host["v_pool"].copy()
        oracle_append(rk, rv, host)
        assert wl.host_array(dinp.k_pool).tobytes() == rk.tobytes(), "K pool after the step"
        assert wl.host_array(dinp.v_pool).tobytes() == rv.tobytes(), "V pool after the step"
    return assert_parity(out, ref, w.dtype, f"{w.name} splits={s} fused={fused}"), s


# ------------------------------------------------------------------ golden --
def _pad_dim(a, d_new):
    pad = [(0, 0)] * (a.ndim - 1) + [(0, d_new - a.shape[-1])]
    return np.pad(a, pad)


def test_golden_read_three_tokens(nplib):
    g = golden_cases.load("read_three_tokens_gqa.json")
    D = 16  # smallest compiled head_dim; zero padding leaves scores unchanged
    q = torch.from_numpy(_pad_dim(g["q"], D)).to(DEV)
    kp = torch.from_numpy(_pad_dim(g["k_pool"], D).astype(np.float32)).to(DEV)
    vp = torch.from_numpy(_pad_dim(g["v_pool"], D).astype(np.float32)).to(DEV)
    for s in (1, 2):
        out = torch.empty_like(q)
        ws = nplib.workspace(1, 2, D, s)
        bt = torch.from_numpy(g["block_tables"]).to(DEV)
        cl = torch.from_numpy(g["context_lens"]).to(DEV)
        nplib.decode_step(out, q, kp, vp, bt, cl, g["scale"], num_splits=s, workspace=ws)
        torch.cuda.synchronize()
        o = to64(out)
        np.testing.assert_allclose(o[..., :2], g["expected_out"], rtol=0, atol=g["atol"])
        assert np.all(o[..., 2:] == 0)


def test_golden_append_then_read(nplib):
    g = golden_cases.load("append_then_read.json")
    D = 16
    kp = torch.from_numpy(_pad_dim(g["k_pool"], D).astype(np.float32)).to(DEV)
    vp = torch.from_numpy(_pad_dim(g["v_pool"], D).astype(np.float32)).to(DEV)
    kn = torch.from_numpy(_pad_dim(g["k_new"], D).astype(np.float32)).to(DEV)
    vn = torch.from_numpy(_pad_dim(g["v_new"], D).astype(np.float32)).to(DEV)
    sm = torch.from_numpy(g["slot_mapping"]).to(DEV)
    q = torch.from_numpy(_pad_dim(g["q"], D)).to(DEV)
    out = torch.empty_like(q)
    nplib.decode_step(out, q, kp, vp, torch.from_numpy(g["block_tables"]).to(DEV),
                      torch.from_numpy(g["context_lens"]).to(DEV), g["scale"], k_new=kn[:1],
                      v_new=vn[:1], slot_mapping=sm[:1])
    nplib.np_kv_append(kp, vp, kn[1:], vn[1:], sm[1:])  # the padding token: skipped
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to64(kp)[..., :1], g["expected_k_pool"])
    np.testing.assert_array_equal(to64(vp)[..., :1], g["expected_v_pool"])
    np.testing.assert_allclose(to64(out)[..., :1], g["expected_out"], rtol=0, atol=g["atol"])


# --------------------------------------------------------- the workloads ---
@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("name", ["tiny-fp32", "llama-fp32"])
def test_workload_full_parity(nplib, name, fused):
    w = wl.WORKLOADS[name]
    _full_parity(nplib, w, fused=fused)
    _full_parity(nplib, w, num_splits=1, fused=fused)


# Every configuration at full size: the pools drawn on the GPU, the launch
# the bench times (the plan's schedule, the append fused into the read), every
# output of every row against the oracle, and both pools after the step
# against the oracle's append, byte for byte.
FULL_SIZE = ["tiny-fp32", "llama-fp32", "llama-fp32-kv16", "bf16-gqa4", "bf16-long",
             "bf16-ragged-bs8", "bf16-ragged-bs32", "bf16-gqa4-q4"]


@pytest.mark.parametrize("name", FULL_SIZE)
def test_workload_full_size_every_row(nplib, name):
    _full_size(nplib, name, fused=True)


@pytest.mark.parametrize("name", ["bf16-long", "bf16-ragged-bs8"])
def test_workload_full_size_unfused_append(nplib, name):
    """The same steps with the append as its own launch (np_kv_append)."""
    _full_size(nplib, name, fused=False)


def _full_size(nplib, name, fused):
    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w, device=DEV)
    host = host_inputs(inp)                      # copied before any kernel runs
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, s, _ = gpu_step(nplib, inp, err=err, fused=fused)
    assert int(err.item()) == 0
    assert torch.isfinite(out.float()).all()
    ref, _ = oracle_step_in_place(host, w.softmax_scale)
    st = assert_parity(out, ref, w.dtype, f"{name} splits={s} fused={fused}")
    print(f"parity-margin {name} fused={int(fused)} schedule={s}: max|err| {st['max_abs']:.3e}"
          f" = {st['max_frac_of_tol']:.3f} of the gate, p99.9 {st['p999_abs']:.3e},"
          f" {st['n']} outputs")
    assert_pool_equal(inp.k_pool, host["k_pool"], f"{name}: K pool after the step")
    assert_pool_equal(inp.v_pool, host["v_pool"], f"{name}: V pool after the step")


# ------------------------------------------------------------ split-K ----
@pytest.mark.parametrize("splits", [1, 2, 3, 5, 16, 32])
def test_split_counts_fp32(nplib, splits):
    _full_parity(nplib, wl.WORKLOADS["llama-fp32"], num_splits=splits)


@pytest.mark.parametrize("splits", [1, 2, 7, 40])
def test_split_counts_bf16(nplib, splits):
    w = _custom([1, 63, 64, 65, 700, 2500, 333], 40, 8, 128, 16, "bf16", seed=5)
    _full_parity(nplib, w, num_splits=splits)


def test_partials_match_oracle_splits(nplib):
    """The workspace holds, per split, the normalised output and natural-log lse."""
    w = _custom([5, 64, 130, 640, 1000], 16, 4, 64, 16, "f32", seed=6)
    inp = wl.make_inputs(w)
    host = wl.full_host(inp)
    d = wl.Inputs(w, inp.md, *(t.to(DEV) for t in
                               (inp.q, inp.k_pool, inp.v_pool, inp.k_new, inp.v_new)))
    S = 9
    out, _, ws = gpu_step(nplib, d, num_splits=S)
    sl = nplib.np_paged_decode_split_len(w.block_size, w.max_blocks_per_row, S)
    n_o = w.rows * w.q_heads * S * w.head_dim
    wsf = ws.view(torch.float32)
    o = wsf[:n_o].view(w.rows, w.q_heads, S, w.head_dim)
    off = (n_o * 4 + 255) // 256 * 256 // 4
    lse = wsf[off:off + w.rows * w.q_heads * S].view(w.rows, w.q_heads, S)
    ro, rl = oracle_step(host, w.softmax_scale, split_len=sl, num_splits=S)
    lse_g = to64(lse)
    assert np.array_equal(np.isinf(lse_g), np.isinf(rl))
    fin = np.isfinite(rl)
    np.testing.assert_allclose(lse_g[fin], rl[fin], rtol=1e-5, atol=1e-5)
    og = to64(o)
    assert_parity(og[fin], ro[fin], "f32", "partials")
    full, _ = oracle_step(host, w.softmax_scale)
    assert_parity(out, full, "f32", "reduced")


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_reduce_alone(nplib, out_dtype):
    R, H, S, D = 5, 6, 7, 128
    g = torch.Generator().manual_seed(3)
    o = torch.randn(R, H, S, D, generator=g, dtype=torch.float32)
    lse = torch.randn(R, H, S, generator=g, dtype=torch.float32) * 4
    lse[0, :, 3] = -float("inf")
    o[0, :, 3] = float("nan")            # an empty split's o is never read
    lse[1, 2, :] = -float("inf")         # every split empty -> zeros
    o[1, 2, :] = float("nan")
    ws = nplib.workspace(R, H, D, S)
    wsf = ws.view(torch.float32)
    n_o = R * H * S * D
    wsf[:n_o] = o.reshape(-1).to(DEV)
    off = (n_o * 4 + 255) // 256 * 256 // 4
    wsf[off:off + R * H * S] = lse.reshape(-1).to(DEV)
    out = torch.empty(R, H, D, dtype=out_dtype, device=DEV)
    nplib.np_paged_decode_reduce(out, ws, S)
    torch.cuda.synchronize()
    ref = oracle.reduce(o.double().numpy(), lse.double().numpy())
    assert np.all(to64(out)[1, 2] == 0)
    if out_dtype == torch.float32:
        assert_parity(out, ref, "f32", "reduce")
    else:
        assert_parity(out, ref, "bf16", "reduce")


# --------------------------------------------------------------- append ---
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_append_bit_exact(nplib, dtype):
    w = _custom([3, 17, 40, 1, 0, 9], 8, 4, 128, 8, dtype, seed=8)
    inp = wl.make_inputs(w, poison=False)
    host = wl.full_host(inp)
    kp, vp = inp.k_pool.to(DEV), inp.v_pool.to(DEV)
    sm = inp.slot_mapping.clone()
    sm[1] = -1                                   # padding token
    nslots = inp.md.num_blocks * w.block_size
    sm[3] = nslots                               # past the pool: skipped, flagged
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    nplib.np_kv_append(kp, vp, inp.k_new.to(DEV), inp.v_new.to(DEV), sm.to(DEV), err)
    torch.cuda.synchronize()
    rk, rv = host["k_pool"].copy(), host["v_pool"].copy()
    rc = oracle.kv_append(rk, rv, host["k_new"], host["v_new"], sm.numpy())
    assert rc == oracle.BAD_BLOCK
    assert int(err.item()) == nplib.NP_FLAG_SLOT
    assert wl.host_array(kp).tobytes() == rk.tobytes()
    assert wl.host_array(vp).tobytes() == rv.tobytes()


def test_append_many_tokens_bit_exact(nplib):
    g = torch.Generator().manual_seed(4)
    nb, bs, hk, d, T = 64, 16, 8, 128, 300
    kp = torch.randn(nb, bs, hk, d, generator=g).to(torch.bfloat16)
    vp = torch.randn(nb, bs, hk, d, generator=g).to(torch.bfloat16)
    kn = torch.randn(T, hk, d, generator=g).to(torch.bfloat16)
    vn = torch.randn(T, hk, d, generator=g).to(torch.bfloat16)
    sm = torch.randperm(nb * bs, generator=g)[:T].to(torch.int64)
    dk, dv = kp.to(DEV), vp.to(DEV)
    nplib.np_kv_append(dk, dv, kn.to(DEV), vn.to(DEV), sm.to(DEV))
    torch.cuda.synchronize()
    rk, rv = wl.host_array(kp), wl.host_array(vp)
    oracle.kv_append(rk, rv, wl.host_array(kn), wl.host_array(vn), sm.numpy())
    assert wl.host_array(dk).tobytes() == rk.tobytes()
    assert wl.host_array(dv).tobytes() == rv.tobytes()


# ------------------------------------------------- every compiled variant --
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("head_dim", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("group", [1, 2, 4, 5, 8])
def test_every_head_dim_and_group(nplib, dtype, head_dim, group):
    w = _custom([1, 37, 200, 16], 2 * group, 2, head_dim, 16, dtype, seed=head_dim + group)
    _full_parity(nplib, w)
    _full_parity(nplib, w, num_splits=3)


@pytest.mark.parametrize("group,kv_heads,query_len", [
    (3, 8, 1), (6, 8, 2), (7, 8, 1), (7, 4, 2), (16, 8, 1), (3, 2, 5), (9, 1, 1), (12, 12, 1)])
def test_any_group_on_bf16(nplib, group, kv_heads, query_len):
    """bf16 pools take any GQA group up to 16 ((query token, head) rows <= 16):
    the tensor-core warps read the group at run time.  Balanced read where
    the kv heads allow it, and the split grid."""
    ctx = [1, query_len, 300, 2049, 64, 0, 900]
    ctx = [max(c, query_len) if c else 0 for c in ctx]
    w = _custom(ctx, kv_heads * group, kv_heads, 128, 16, "bf16",
                seed=300 + group * 7 + kv_heads + query_len, query_len=query_len)
    _full_parity(nplib, w, num_splits=0)
    _full_parity(nplib, w, num_splits=1)
    _full_parity(nplib, w, num_splits=3, fused=False)


@pytest.mark.parametrize("group,kv_heads,query_len,head_dim", [
    (3, 8, 1, 128), (6, 8, 1, 64), (7, 4, 1, 128), (3, 8, 2, 256), (6, 12, 1, 32),
    (3, 2, 1, 128), (7, 1, 1, 64), (3, 3, 2, 16), (6, 5, 1, 256)])
def test_other_groups_on_fp32(nplib, group, kv_heads, query_len, head_dim):
    """fp32 groups outside {1, 2, 4, 5, 8} (up to 8 (query token, head) rows)
    run on the FMA warp's layout with the group read at run time: on the
    balanced read where the kv heads allow it, and on the split grid, one
    split or several."""
    ctx = [1, 300, 2049, 64, 0, 900]
    ctx = [max(c, query_len) if c else 0 for c in ctx]
    w = _custom(ctx, kv_heads * group, kv_heads, head_dim, 16, "f32",
                seed=400 + group * 7 + kv_heads + query_len, query_len=query_len)
    if head_dim % 32 == 0:
        _full_parity(nplib, w, num_splits=0)
        _full_parity(nplib, w, num_splits=0, fused=False)
    _full_parity(nplib, w, num_splits=1)
    _full_parity(nplib, w, num_splits=3, fused=False)


@pytest.mark.parametrize("kv_heads", [1, 3, 5, 12, 16])
def test_kv_head_grouping(nplib, kv_heads):
    """kv_heads not a multiple of 8 and > 8 (several head groups per row)."""
    w = _custom([50, 129, 7], 2 * kv_heads, kv_heads, 64, 16, "bf16", seed=20 + kv_heads)
    _full_parity(nplib, w)
    _full_parity(nplib, w, num_splits=4)


@pytest.mark.parametrize("block_size", [1, 3, 8, 16, 24, 32, 64, 128])
def test_block_sizes(nplib, block_size):
    w = _custom([1, 31, 32, 33, 255, 513], 8, 2, 128, block_size, "f32", seed=30 + block_size)
    _full_parity(nplib, w)
    _full_parity(nplib, w, num_splits=5)
    _full_parity(nplib, w, num_splits=5, fused=False)


@pytest.mark.parametrize("kv_heads", [1, 8])
@pytest.mark.parametrize("block_size", [1, 3, 4, 8, 24, 32, 64])
def test_block_sizes_bf16(nplib, block_size, kv_heads):
    """bf16 staging: tiled TMA boxes of 1..16 tokens (one or several per
    chunk) and, where a box would not start on a swizzle boundary
    (box tokens x kv heads per CTA not a multiple of 8), per-token copies."""
    w = _custom([1, 15, 16, 17, 100, 700], 2 * kv_heads, kv_heads, 128, block_size, "bf16",
                seed=70 + block_size + kv_heads)
    _full_parity(nplib, w)
    _full_parity(nplib, w, num_splits=3)
    _full_parity(nplib, w, num_splits=3, fused=False)


def test_edge_contexts(nplib):
    """Empty rows, one token, exact chunk and split boundaries, full tables."""
    ctx = [0, 1, 2, 15, 16, 17, 63, 64, 65, 127, 128, 129, 512]
    w = _custom(ctx, 8, 8, 128, 16, "bf16", seed=40)
    for s in (1, 2, 8, 32):
        _full_parity(nplib, w, num_splits=s)
    w = _custom(ctx, 4, 2, 128, 16, "f32", seed=41)
    for s in (1, 3, 9):
        _full_parity(nplib, w, num_splits=s)


def test_zero_context_gives_zeros_and_single_token_gives_v(nplib):
    w = _custom([0, 1, 1], 8, 2, 128, 16, "f32", seed=42)
    inp = wl.make_inputs(w)
    d = wl.Inputs(w, inp.md, *(t.to(DEV) for t in
                               (inp.q, inp.k_pool, inp.v_pool, inp.k_new, inp.v_new)))
    for s in (1, 2):
        out, _, _ = gpu_step(nplib, d, num_splits=s)
        o = to64(out)
        assert np.all(o[0] == 0)
        vnew = to64(inp.v_new)                       # the only token is the new one
        np.testing.assert_array_equal(o[1], np.repeat(vnew[1], 4, axis=0))


def test_fused_append_refuses_a_slot_that_is_not_the_newest_position(nplib):
    """A slot-mapping entry that is not where the row's newest position lives
    is flagged and not written (the row then reads its pool as it was)."""
    w = _custom([40, 25, 64], 8, 2, 128, 16, "bf16", seed=55)
    inp = wl.make_inputs(w, poison=False)
    host = wl.full_host(inp)
    sm = inp.slot_mapping.clone()
    sm[1] = int(inp.slot_mapping[0])           # row 0's slot: not row 1's position
    md = wl.Metadata(inp.context_lens, inp.block_tables, sm, inp.md.num_blocks)
    d = wl.Inputs(w, md, *(t.to(DEV) for t in
                           (inp.q, inp.k_pool, inp.v_pool, inp.k_new, inp.v_new)))
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    for s in (1, 4):
        d.k_pool.copy_(inp.k_pool.to(DEV))
        d.v_pool.copy_(inp.v_pool.to(DEV))
        err.zero_()
        out, _, _ = gpu_step(nplib, d, num_splits=s, err=err)
        assert int(err.item()) == nplib.NP_FLAG_SLOT
        keep = np.array([0, 2])
        h2 = dict(host, slot_mapping=np.array([int(inp.slot_mapping[0]), -1,
                                               int(inp.slot_mapping[2])], dtype=np.int64))
        ref, _ = oracle_step(h2, w.softmax_scale)
        assert_parity(out, ref, "bf16", f"mismatched slot splits={s}")
        rk = host["k_pool"].copy()
        rv = host["v_pool"].copy()
        oracle.kv_append(rk, rv, host["k_new"][keep], host["v_new"][keep],
                         inp.slot_mapping.numpy()[keep])
        assert wl.host_array(d.k_pool).tobytes() == rk.tobytes()


# ------------------------------------------------- several query tokens ----
@pytest.mark.parametrize("group,query_len", [(1, 3), (1, 16), (2, 5), (4, 2), (4, 4), (5, 3),
                                             (8, 2)])
def test_multi_query_tokens(nplib, group, query_len):
    """Each row's last query_len positions attend causally (bf16, tensor cores),
    with the new tokens appended fused or separately, split or not; includes
    rows shorter than the query run and runs crossing split boundaries."""
    ctx = [1, query_len, query_len + 1, 63, 64, 65, 700, 1500]
    w = _custom(ctx, 2 * group, 2, 128, 16, "bf16", seed=90 + group * 7 + query_len,
                query_len=query_len)
    for s in (1, 5):
        _full_parity(nplib, w, num_splits=s)
    _full_parity(nplib, w, num_splits=5, fused=False)


@pytest.mark.parametrize("group,query_len,head_dim", [(1, 3, 128), (1, 8, 64), (2, 4, 128),
                                                       (4, 2, 128), (2, 3, 256), (1, 5, 32)])
def test_multi_query_tokens_fp32(nplib, group, query_len, head_dim):
    """fp32 pools: several query tokens per row on the balanced read (FMA
    warps, (query token, head) rows up to 8), fused append or separate."""
    ctx = [1, query_len, query_len + 1, 63, 64, 65, 700, 1500, 0]
    w = _custom(ctx, 8 * group, 8, head_dim, 16, "f32", seed=200 + group * 7 + query_len,
                query_len=query_len)
    _full_parity(nplib, w, num_splits=0)
    _full_parity(nplib, w, num_splits=0, fused=False)


@pytest.mark.parametrize("kv_heads,group,query_len,head_dim", [
    (1, 2, 3, 128), (2, 1, 5, 64), (3, 2, 4, 32), (11, 1, 3, 128)])
def test_multi_query_tokens_fp32_small_head_groups(nplib, kv_heads, group, query_len, head_dim):
    """fp32, several query tokens, head groups under 8 on the balanced read:
    several FMA warps per kv head, each on its slice of every stage (one
    head of 11: one copy per token, in rounds of 32 tokens)."""
    ctx = [1, query_len, query_len + 1, 63, 64, 65, 700, 1500, 0]
    w = _custom(ctx, kv_heads * group, kv_heads, head_dim, 16, "f32",
                seed=240 + kv_heads * 5 + group + query_len, query_len=query_len)
    _full_parity(nplib, w, num_splits=0)
    _full_parity(nplib, w, num_splits=0, fused=False)


@pytest.mark.parametrize("group,kv_heads,query_len,head_dim", [
    (2, 8, 2, 128), (1, 2, 5, 64), (4, 2, 2, 128), (2, 3, 3, 32), (1, 1, 8, 16)])
def test_multi_query_fp32_split_grid(nplib, group, kv_heads, query_len, head_dim):
    """Several query tokens per row on fp32 pools through the split grid (any
    kv head count, head_dim 16 included), one split and several, the append
    fused or separate."""
    ctx = [1, query_len, query_len + 1, 63, 64, 65, 700, 1500, 0]
    w = _custom(ctx, kv_heads * group, kv_heads, head_dim, 16, "f32",
                seed=210 + group * 7 + kv_heads + query_len, query_len=query_len)
    _full_parity(nplib, w, num_splits=1)
    _full_parity(nplib, w, num_splits=4)
    _full_parity(nplib, w, num_splits=4, fused=False)


@pytest.mark.parametrize("head_dim,block_size", [(64, 8), (256, 32), (32, 16)])
def test_multi_query_head_dims(nplib, head_dim, block_size):
    w = _custom([5, 80, 300], 16, 8, head_dim, block_size, "bf16", seed=130 + head_dim,
                query_len=2)
    _full_parity(nplib, w)
    _full_parity(nplib, w, num_splits=3)


def test_head_dim_256_with_eight_kv_heads(nplib):
    w = _custom([10, 700, 2500], 64, 8, 256, 32, "bf16", seed=140)
    _full_parity(nplib, w)
    _full_parity(nplib, w, num_splits=4)


# ------------------------------------------- the balanced streamed read ----
@pytest.mark.parametrize("kv_heads,group,head_dim,block_size,query_len", [
    (8, 4, 128, 16, 1), (8, 8, 128, 32, 1), (8, 5, 128, 8, 1), (16, 1, 64, 16, 1),
    (8, 2, 256, 32, 1), (8, 4, 128, 16, 3), (8, 8, 64, 64, 2), (16, 4, 128, 4, 1),
    (4, 4, 128, 16, 1), (4, 8, 128, 32, 2), (12, 2, 64, 8, 1), (4, 5, 256, 2, 1),
    (20, 1, 128, 16, 4), (1, 8, 128, 16, 1), (1, 16, 128, 32, 1), (2, 8, 128, 16, 2),
    (3, 4, 128, 8, 1), (6, 3, 64, 16, 1), (5, 2, 256, 16, 1), (7, 1, 128, 32, 3),
    (2, 4, 64, 8, 1), (10, 2, 128, 16, 1), (11, 2, 128, 16, 1), (9, 2, 128, 8, 1),
    (1, 8, 256, 16, 1), (2, 8, 64, 16, 1), (1, 4, 128, 8, 2),
    (1, 3, 128, 16, 1), (2, 5, 64, 16, 1), (1, 5, 128, 8, 3)])
def test_balanced_read(nplib, kv_heads, group, head_dim, block_size, query_len):
    """num_splits = 0: one CTA per SM, equal token shares; rows cut between
    CTAs are merged by the second kernel.  Small totals spread over 152
    CTAs cut most rows, so the merge path is exercised heavily.  Any kv head
    count: with fewer than 8 heads per CTA several warps read each head,
    each taking its slice of every stage's tokens, and merge their states at
    every row end."""
    ctx = [0, 1, 5, 16, 17, 300, 2049, 64, 0, 4000, 31, 7]
    ctx = [max(c, query_len if c else 0) for c in ctx]
    w = _custom(ctx, kv_heads * group, kv_heads, head_dim, block_size, "bf16",
                seed=150 + kv_heads + group + head_dim + block_size + query_len,
                query_len=query_len)
    _full_parity(nplib, w, num_splits=0)
    _full_parity(nplib, w, num_splits=0, fused=False)


@pytest.mark.parametrize("kv_heads,group,head_dim,block_size", [
    (8, 4, 128, 16), (8, 1, 128, 32), (8, 2, 64, 8), (8, 8, 32, 3), (8, 5, 256, 16),
    (16, 4, 128, 16), (16, 2, 256, 1), (8, 8, 128, 24), (8, 4, 32, 64),
    (4, 4, 128, 16), (12, 1, 256, 3), (4, 8, 64, 1), (1, 8, 128, 16), (2, 4, 128, 3),
    (3, 2, 64, 16), (6, 1, 256, 8), (5, 8, 32, 1), (11, 2, 128, 16), (13, 1, 32, 16),
    (1, 8, 256, 16), (2, 4, 64, 1), (1, 3, 64, 16), (2, 5, 128, 16), (1, 7, 32, 8)])
def test_balanced_read_fp32(nplib, kv_heads, group, head_dim, block_size):
    """fp32 pools on the balanced read (FMA consumers, 1-D bulk copies:
    whole block runs when the pool has just the CTA's kv heads, one copy per
    token otherwise, in rounds of 32 tokens when a stage holds more).  Odd
    groups with one or two kv heads: several warps per head whose row-end
    states hold an odd number of rows (16-byte vector stores)."""
    ctx = [0, 1, 5, 16, 17, 300, 2049, 64, 0, 4000, 31, 7]
    w = _custom(ctx, kv_heads * group, kv_heads, head_dim, block_size, "f32",
                seed=180 + kv_heads + group + head_dim + block_size)
    _full_parity(nplib, w, num_splits=0)
    _full_parity(nplib, w, num_splits=0, fused=False)


@pytest.mark.parametrize("dtype,ctx,block_size", [
    ("bf16", [20000], 16),                    # one row cut across every CTA
    ("f32", [9000], 16),
    ("bf16", [16] * 40 + [15] * 40, 16),      # many one-chunk rows: few cuts
    ("f32", [8] * 100 + [1] * 20, 8),
    ("bf16", [16 * 37, 16 * 5, 16 * 300, 16], 16),  # lengths whole chunks
    ("f32", [8 * 41, 8 * 3, 8 * 500, 8], 8),
    ("bf16", [0, 0, 0, 70000, 0], 32),        # empty rows around a long one
    ("bf16", [3, 3, 3], 4),                   # fewer chunks than 4 per SM: few CTAs
])
def test_balanced_read_partition_edges(nplib, dtype, ctx, block_size):
    """Partition edge cases of the balanced read: a row cut into as many
    pieces as there are CTAs (its merge tasks dealt over all of them), many
    rows of one chunk each, rows of whole chunks (boundaries on row ends),
    empty rows beside a long one, and a step too small for every SM."""
    w = _custom(ctx, 32, 8, 128, block_size, dtype, seed=700 + len(ctx) + block_size)
    _full_parity(nplib, w, num_splits=0)


def test_balanced_read_two_calls_one_workspace(nplib):
    """The workspace needs no zeroing: a NaN-filled one, reused by a second
    call with other lengths, must not leak stale partials."""
    ws = None
    for seed, ctx in ((160, [3000, 17, 900, 64, 1]), (161, [5, 5000, 2500, 0, 130])):
        w = _custom(ctx, 32, 8, 128, 16, "bf16", seed=seed)
        inp = wl.make_inputs(w)
        host = wl.full_host(inp)
        if ws is None:
            ws = nplib.workspace(w.rows, w.q_heads, w.head_dim, 0)
            ws.view(torch.float32).fill_(float("nan"))
        dev = [t.to(DEV) for t in (inp.q, inp.k_pool, inp.v_pool, inp.k_new, inp.v_new)]
        bt, cl, sm = (t.to(DEV) for t in (inp.block_tables, inp.context_lens, inp.slot_mapping))
        out = torch.full_like(dev[0], float("nan"))
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        nplib.np_paged_append_decode(out, dev[0], dev[3], dev[4], sm, dev[1], dev[2], bt, cl,
                                     w.softmax_scale, 0, ws, err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        ref, _ = oracle_step(host, w.softmax_scale)
        assert_parity(out, ref, "bf16", f"balanced call seed={seed}")


def test_balanced_read_graph_replay(nplib):
    w = _custom([700, 4096, 33, 1200, 2], 40, 8, 128, 32, "bf16", seed=170)
    inp = wl.make_inputs(w)
    host = wl.full_host(inp)
    q, kp, vp, kn, vn = (t.to(DEV) for t in (inp.q, inp.k_pool, inp.v_pool, inp.k_new, inp.v_new))
    bt, cl, sm = (t.to(DEV) for t in (inp.block_tables, inp.context_lens, inp.slot_mapping))
    ws = nplib.workspace(w.rows, w.q_heads, w.head_dim, 0)
    out = torch.empty_like(q)
    nplib.np_paged_append_decode(out, q, kn, vn, sm, kp, vp, bt, cl, w.softmax_scale, 0, ws)
    torch.cuda.synchronize()
    eager = out.clone()
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        nplib.np_paged_append_decode(out, q, kn, vn, sm, kp, vp, bt, cl, w.softmax_scale, 0, ws)
    for _ in range(3):
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager)
    ref, _ = oracle_step(host, w.softmax_scale)
    assert_parity(out, ref, "bf16", "balanced graph replay")


# ---------------------------------------------------------- robustness ----
def test_bad_block_id_is_flagged_not_faulted(nplib):
    w = _custom([40, 40], 8, 2, 128, 16, "f32", seed=50)
    inp = wl.make_inputs(w, poison=False)
    host = wl.full_host(inp)
    bt = inp.block_tables.clone()
    bt[0, 1] = inp.md.num_blocks + 1000                 # outside the pool
    d = wl.Inputs(w, wl.Metadata(inp.context_lens, bt, inp.slot_mapping, inp.md.num_blocks),
                  *(t.to(DEV) for t in (inp.q, inp.k_pool, inp.v_pool, inp.k_new, inp.v_new)))
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, _, _ = gpu_step(nplib, d, num_splits=1, err=err)
    assert int(err.item()) & nplib.NP_FLAG_BLOCK_ID
    ref, _ = oracle_step(host, w.softmax_scale)
    assert_parity(out[1:], ref[1:], "f32", "the untouched row")


def test_context_past_table_is_clamped_and_flagged(nplib):
    w = _custom([40, 64], 8, 2, 128, 16, "f32", seed=51)
    inp = wl.make_inputs(w)
    host = wl.full_host(inp)
    cl = inp.context_lens.clone()
    cl[0] = 10_000                                      # table holds 64
    dmd = wl.Metadata(cl, inp.block_tables, inp.slot_mapping, inp.md.num_blocks)
    d = wl.Inputs(w, dmd, *(t.to(DEV) for t in
                            (inp.q, inp.k_pool, inp.v_pool, inp.k_new, inp.v_new)))
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, _, _ = gpu_step(nplib, d, num_splits=1, err=err)
    assert int(err.item()) & nplib.NP_FLAG_CONTEXT
    ref, _ = oracle_step(host, w.softmax_scale)
    assert_parity(out[1:], ref[1:], "f32", "the untouched row")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_balanced_bad_block_id_is_flagged_not_faulted(nplib, dtype):
    """The balanced read walks several rows per thread block: a bad table
    entry is flagged and read as block 0, and only its own row is affected."""
    w = _custom([40, 300, 40, 1000], 32, 8, 128, 16, dtype, seed=53)
    inp = wl.make_inputs(w, poison=False)
    host = wl.full_host(inp)
    bt = inp.block_tables.clone()
    bt[0, 1] = inp.md.num_blocks + 1000                 # outside the pool
    bt[2, 0] = -5
    d = wl.Inputs(w, wl.Metadata(inp.context_lens, bt, inp.slot_mapping, inp.md.num_blocks),
                  *(t.to(DEV) for t in (inp.q, inp.k_pool, inp.v_pool, inp.k_new, inp.v_new)))
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, s, _ = gpu_step(nplib, d, num_splits=0, err=err)
    assert s == 0 and int(err.item()) & nplib.NP_FLAG_BLOCK_ID
    assert torch.isfinite(out.float()).all()
    ref, _ = oracle_step(host, w.softmax_scale)
    for r in (1, 3):
        assert_parity(out[r:r + 1], ref[r:r + 1], dtype, f"untouched row {r}")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_balanced_context_out_of_range_is_clamped_and_flagged(nplib, dtype):
    w = _custom([40, 64, 500, 7], 32, 8, 128, 16, dtype, seed=54)
    inp = wl.make_inputs(w)
    host = wl.full_host(inp)
    cl = inp.context_lens.clone()
    cl[0] = 10_000                                      # the table holds 512
    cl[3] = -3                                          # read as empty
    dmd = wl.Metadata(cl, inp.block_tables, inp.slot_mapping, inp.md.num_blocks)
    d = wl.Inputs(w, dmd, *(t.to(DEV) for t in
                            (inp.q, inp.k_pool, inp.v_pool, inp.k_new, inp.v_new)))
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, s, _ = gpu_step(nplib, d, num_splits=0, err=err)
    assert s == 0 and int(err.item()) & nplib.NP_FLAG_CONTEXT
    # row 0 reads table entries past its history (poisoned): its values are
    # not checked; the others are untouched and row 3 is empty
    assert torch.isfinite(out[1:].float()).all()
    assert torch.count_nonzero(out[3]) == 0
    ref, _ = oracle_step(host, w.softmax_scale)
    assert_parity(out[1:3], ref[1:3], dtype, "the untouched rows")


def test_balanced_read_at_the_row_limit(nplib):
    """4096 (row, 8-head group) pairs: the largest balanced launch (its row
    prefix takes 32 KB of shared memory, the ring drops to 2 stages); one more
    row is refused with NP_ERR_UNSUPPORTED and the plan picks the split grid."""
    g = torch.Generator().manual_seed(55)
    ctx = torch.randint(1, 48, (4096,), generator=g).tolist()
    w = _custom(ctx, 8, 8, 64, 16, "bf16", seed=55)
    _full_parity(nplib, w, num_splits=0)
    assert nplib.np_paged_decode_plan(4096, 8, 8, 64, 16, 3, "bf16") == 0
    assert nplib.np_paged_decode_plan(4097, 8, 8, 64, 16, 3, "bf16") >= 1
    w2 = _custom(ctx + [5], 8, 8, 64, 16, "bf16", seed=56)
    inp = wl.make_inputs(w2)
    d = [t.to(DEV) for t in (inp.q, inp.k_pool, inp.v_pool)]
    bt, cl = inp.block_tables.to(DEV), inp.context_lens.to(DEV)
    ws = nplib.workspace(w2.rows, w2.q_heads, w2.head_dim, 0)
    with pytest.raises(nplib.NPError) as e:
        nplib.np_paged_decode(torch.empty_like(d[0]), d[0], d[1], d[2], bt, cl, 0.1,
                              num_splits=0, workspace=ws)
    assert e.value.status == nplib.NP_ERR_UNSUPPORTED


def test_bounded_wait_gives_up_and_the_context_stays_usable(nplib):
    """The read's wait-timeout path, exercised without any fault: a wait that
    nothing completes gives up after ~1 ms, flags NP_FLAG_TIMEOUT, and the
    next read on the same context is correct."""
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    nplib.np_selftest_bounded_wait(err, 2_000_000)       # ~1 ms at 2 GHz
    torch.cuda.synchronize()
    assert int(err.item()) == nplib.NP_FLAG_TIMEOUT
    with pytest.raises(nplib.NPError):
        nplib.np_selftest_bounded_wait(err, 0)
    w = _custom([300, 5, 2000], 32, 8, 128, 16, "bf16", seed=57)
    _full_parity(nplib, w)


def test_tensors_off_the_current_device_are_refused(nplib, monkeypatch):
    """Kernels launch on the current device: a tensor on another GPU would be
    dereferenced there.  The binding refuses it before any launch (the
    current device is made to look like another one, so one GPU suffices)."""
    w = _custom([40, 70], 16, 8, 128, 16, "bf16", seed=59)
    inp = wl.make_inputs(w, poison=False)      # finite pools: compared with torch.equal
    q, kp, vp, kn, vn = (t.to(DEV) for t in (inp.q, inp.k_pool, inp.v_pool, inp.k_new, inp.v_new))
    bt, cl, sm = (t.to(DEV) for t in (inp.block_tables, inp.context_lens, inp.slot_mapping))
    ws = nplib.workspace(w.rows, w.q_heads, w.head_dim, 4)
    out = torch.full_like(q, float("nan"))
    kp0 = kp.clone()
    torch.cuda.synchronize()
    other = torch.cuda.current_device() + 1
    monkeypatch.setattr(nplib, "_current_device", lambda: other)
    calls = [
        lambda: nplib.np_paged_decode(out, q, kp, vp, bt, cl, 0.1, num_splits=1),
        lambda: nplib.np_paged_append_decode(out, q, kn, vn, sm, kp, vp, bt, cl, 0.1, 1),
        lambda: nplib.np_kv_append(kp, vp, kn, vn, sm),
        lambda: nplib.np_paged_decode_reduce(out, ws, 4),
        lambda: nplib.np_paged_decode_noalloc(out, q, kp, vp, bt, cl, 0.1, 4),
        lambda: nplib.PreparedStep(out, q, kn, vn, sm, kp, vp, bt, cl, 0.1, 1),
    ]
    for call in calls:
        with pytest.raises(ValueError, match="current device"):
            call()
    monkeypatch.undo()
    torch.cuda.synchronize()
    assert torch.isnan(out.float()).all()        # nothing was launched
    assert torch.equal(kp, kp0)


def test_validation_errors_return_before_launch(nplib):
    w = _custom([10], 8, 2, 128, 16, "f32", seed=52)
    inp = wl.make_inputs(w)
    d = [t.to(DEV) for t in (inp.q, inp.k_pool, inp.v_pool)]
    bt, cl = inp.block_tables.to(DEV), inp.context_lens.to(DEV)
    out = torch.empty_like(d[0])
    with pytest.raises(nplib.NPError) as e:
        nplib.np_paged_decode(out, d[0], d[1], d[2], bt, cl, float("inf"))
    assert e.value.status == nplib.NP_ERR_INVALID_ARG
    with pytest.raises(nplib.NPError) as e:
        nplib.np_paged_decode(None, d[0], d[1], d[2], bt, cl, 0.1, num_splits=4)
    assert e.value.status == nplib.NP_ERR_WORKSPACE
    small = torch.empty(16, dtype=torch.uint8, device=DEV)
    with pytest.raises(nplib.NPError) as e:
        nplib.np_paged_decode(None, d[0], d[1], d[2], bt, cl, 0.1, num_splits=4, workspace=small)
    assert e.value.status == nplib.NP_ERR_WORKSPACE


# ------------------------------------------------------ launch contexts ---
def test_cuda_graph_capture_planned_schedule(nplib):
    """The plan's schedule for a bf16 GQA-5 step with the fused append,
    captured in a CUDA graph: the replay equals the direct call bit for bit
    and matches the oracle."""
    w = _custom([100, 3000, 17, 1200], 40, 8, 128, 32, "bf16", seed=60)
    inp = wl.make_inputs(w)
    host = wl.full_host(inp)
    q, kp, vp, kn, vn = (t.to(DEV) for t in (inp.q, inp.k_pool, inp.v_pool, inp.k_new, inp.v_new))
    bt, cl, sm = (t.to(DEV) for t in (inp.block_tables, inp.context_lens, inp.slot_mapping))
    S = nplib.np_paged_decode_plan(w.rows, w.q_heads, w.kv_heads, w.head_dim, w.block_size,
                                   bt.shape[1], torch.bfloat16)
    ws = nplib.workspace(w.rows, w.q_heads, w.head_dim, S)
    out = torch.empty_like(q)
    # first call on the device outside capture (sets kernel attributes)
    nplib.decode_step(out, q, kp, vp, bt, cl, w.softmax_scale, k_new=kn, v_new=vn,
                      slot_mapping=sm, num_splits=S, workspace=ws)
    torch.cuda.synchronize()
    eager = out.clone()
    out.zero_()
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        nplib.decode_step(out, q, kp, vp, bt, cl, w.softmax_scale, k_new=kn, v_new=vn,
                          slot_mapping=sm, num_splits=S, workspace=ws)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)
    ref, _ = oracle_step(host, w.softmax_scale)
    assert_parity(out, ref, "bf16", "graph replay")


def test_concurrent_streams_from_two_host_threads(nplib):
    """Two decode steps in flight at once -- each on its own stream with its
    own workspace, issued from its own host thread, 20 times over (the fused
    append rewrites the same new token, so repeats are idempotent) -- both
    match the oracle and leave the pools as the oracle's append does."""
    import threading

    cases = [_custom([700, 4096, 33, 0, 1200], 40, 8, 128, 32, "bf16", seed=600),
             _custom([17, 900, 2500, 64], 32, 8, 128, 16, "f32", seed=601)]
    runs = []
    for w in cases:
        inp = wl.make_inputs(w)
        host = wl.full_host(inp)
        dinp = wl.Inputs(w, inp.md, *(t.to(DEV) for t in
                                      (inp.q, inp.k_pool, inp.v_pool, inp.k_new, inp.v_new)))
        runs.append((w, inp, host, dinp))
    outs, errs, failures = [None, None], [None, None], []

    def worker(i):
        try:  # no synchronisation inside: the two threads' steps overlap on the GPU
            w, inp, host, dinp = runs[i]
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                bt, cl, sm = (t.to(DEV) for t in (dinp.block_tables, dinp.context_lens,
                                                  dinp.slot_mapping))
                ws = nplib.workspace(w.rows, w.q_heads, w.head_dim, 0, device=DEV)
                out = torch.full_like(dinp.q, float("nan"))
                for _ in range(20):
                    nplib.decode_step(out, dinp.q, dinp.k_pool, dinp.v_pool, bt, cl,
                                      w.softmax_scale, k_new=dinp.k_new, v_new=dinp.v_new,
                                      slot_mapping=sm, num_splits=0, workspace=ws,
                                      err_word=errs[i], stream=s)
                outs[i] = out
        except Exception as e:  # reported on the main thread
            failures.append(e)

    for i in range(2):
        errs[i] = torch.zeros(1, dtype=torch.int32, device=DEV)
    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not failures, failures
    for i, (w, inp, host, dinp) in enumerate(runs):
        assert int(errs[i].item()) == 0
        ref, _ = oracle_step(host, w.softmax_scale)
        assert_parity(outs[i], ref, w.dtype, f"concurrent {w.name}")
        rk, rv = host["k_pool"].copy(), host["v_pool"].copy()
        oracle_append(rk, rv, host)
        assert wl.host_array(dinp.k_pool).tobytes() == rk.tobytes()
        assert wl.host_array(dinp.v_pool).tobytes() == rv.tobytes()


def test_non_default_stream_and_determinism(nplib):
    w = _custom([900, 50, 2048], 32, 8, 128, 16, "bf16", seed=61)
    inp = wl.make_inputs(w)
    d = wl.Inputs(w, inp.md, *(t.to(DEV) for t in
                               (inp.q, inp.k_pool, inp.v_pool, inp.k_new, inp.v_new)))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        a, _, _ = gpu_step(nplib, d, stream=s)
    b, _, _ = gpu_step(nplib, d)
    assert torch.equal(a, b)


@pytest.mark.parametrize("dtype,splits", [("bf16", 0), ("f32", 0), ("bf16", 4), ("f32", 1)])
def test_cuda_graph_capture_and_replay(nplib, dtype, splits):
    """A decode step captured in a CUDA graph and replayed: the replay equals
    the direct call bit for bit and matches the oracle; after q is rewritten
    in place, a replay reads the new q (the graph re-runs the kernels on the
    captured buffers rather than repeating a result)."""
    w = _custom([700, 4096, 33, 0, 1200, 5000], 32, 8, 128, 16, dtype, seed=610 + splits)
    inp = wl.make_inputs(w)
    host = wl.full_host(inp)
    d = wl.Inputs(w, inp.md, *(t.to(DEV) for t in
                               (inp.q, inp.k_pool, inp.v_pool, inp.k_new, inp.v_new)))
    bt, cl, sm = (t.to(DEV) for t in (d.block_tables, d.context_lens, d.slot_mapping))
    ws = nplib.workspace(w.rows, w.q_heads, w.head_dim, splits, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = torch.full_like(d.q, float("nan"))

    def step(s):
        nplib.decode_step(out, d.q, d.k_pool, d.v_pool, bt, cl, w.softmax_scale,
                          k_new=d.k_new, v_new=d.v_new, slot_mapping=sm, num_splits=splits,
                          workspace=ws, err_word=err, stream=s)

    step(torch.cuda.current_stream())
    torch.cuda.synchronize()
    direct = out.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step(s)
    out.fill_(float("nan"))
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(out, direct)
    ref, _ = oracle_step(host, w.softmax_scale)
    assert_parity(out, ref, w.dtype, f"graph replay {w.name}")

    q2 = torch.randn(d.q.shape, generator=torch.Generator().manual_seed(77)).to(d.q.dtype)
    d.q.copy_(q2.to(DEV))
    g.replay()
    torch.cuda.synchronize()
    host2 = dict(host, q=wl.host_array(d.q))
    ref2, _ = oracle_step(host2, w.softmax_scale)
    assert_parity(out, ref2, w.dtype, f"graph replay with a new q {w.name}")


@pytest.mark.parametrize("dtype,splits", [("bf16", 0), ("f32", 0), ("bf16", 4), ("f32", 1)])
def test_prepared_step(nplib, dtype, splits):
    """PreparedStep issues the same calls as decode_step: equal output bit
    for bit, the oracle's result, and a relaunch after q is rewritten in
    place reads the new q."""
    w = _custom([700, 4096, 33, 0, 1200, 5000], 32, 8, 128, 16, dtype, seed=630 + splits)
    inp = wl.make_inputs(w)
    host = wl.full_host(inp)
    d = wl.Inputs(w, inp.md, *(t.to(DEV) for t in
                               (inp.q, inp.k_pool, inp.v_pool, inp.k_new, inp.v_new)))
    bt, cl, sm = (t.to(DEV) for t in (d.block_tables, d.context_lens, d.slot_mapping))
    ws = nplib.workspace(w.rows, w.q_heads, w.head_dim, splits, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out_ref = torch.full_like(d.q, float("nan"))
    nplib.decode_step(out_ref, d.q, d.k_pool, d.v_pool, bt, cl, w.softmax_scale,
                      k_new=d.k_new, v_new=d.v_new, slot_mapping=sm, num_splits=splits,
                      workspace=ws, err_word=err)
    out = torch.full_like(d.q, float("nan"))
    ps = nplib.PreparedStep(out, d.q, d.k_new, d.v_new, sm, d.k_pool, d.v_pool, bt, cl,
                            w.softmax_scale, splits, ws, err)
    assert ps.launch() == (2 if splits == 0 else 1) + (1 if splits > 1 else 0)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(out, out_ref)
    ref, _ = oracle_step(host, w.softmax_scale)
    assert_parity(out, ref, w.dtype, f"prepared {w.name}")
    q2 = torch.randn(d.q.shape, generator=torch.Generator().manual_seed(78)).to(d.q.dtype)
    d.q.copy_(q2.to(DEV))
    ps.launch()
    torch.cuda.synchronize()
    ref2, _ = oracle_step(dict(host, q=wl.host_array(d.q)), w.softmax_scale)
    assert_parity(out, ref2, w.dtype, f"prepared relaunch {w.name}")
