"""The synthetic-input recipes (CPU only): shapes, tables, poison, the step."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as wl


@pytest.mark.parametrize("name", sorted(wl.WORKLOADS))
def test_metadata_is_a_valid_allocation(name):
    w = wl.WORKLOADS[name]
    md = wl.metadata(w)
    cl = md.context_lens
    assert cl.shape == (w.rows,) and cl.dtype == torch.int32
    kind = w.ctx[0]
    if kind != "fixed":
        assert int(cl.min()) >= w.ctx[1] and int(cl.max()) <= w.ctx[2]
    assert md.block_tables.shape == (w.rows, w.max_blocks_per_row)
    used = []
    for r in range(w.rows):
        n = -(-int(cl[r]) // w.block_size)
        row = md.block_tables[r]
        assert (row[:n] >= 0).all() and (row[:n] < md.num_blocks).all()
        assert (row[n:] == -1).all()
        used.append(row[:n])
    used = torch.cat(used)
    assert used.unique().numel() == used.numel(), "a block is shared by two rows"
    bt = md.block_tables.to(torch.int64)
    sm = md.slot_mapping.reshape(w.rows, w.query_len)
    for j in range(w.query_len):  # new token j sits at position c - query_len + j
        c = cl.to(torch.int64) - w.query_len + j
        expect = bt[torch.arange(w.rows), c // w.block_size] * w.block_size + c % w.block_size
        assert torch.equal(sm[:, j], expect)


def test_pool_sizes_match_the_configs():
    assert wl.metadata(wl.WORKLOADS["tiny-fp32"]).num_blocks == 32
    long = wl.WORKLOADS["bf16-long"]
    md = wl.metadata(long)
    pool_bytes = 2 * md.num_blocks * long.block_size * long.kv_heads * long.head_dim * 2
    assert md.num_blocks == 65536 and abs(pool_bytes / 1e9 - 8.6) < 0.05
    g4 = wl.WORKLOADS["bf16-gqa4"]
    md = wl.metadata(g4)
    need = sum(-(-int(c) // 16) for c in md.context_lens)
    assert md.num_blocks == math.ceil(1.25 * need)


def test_loguniform_contexts_span_the_range():
    w = wl.WORKLOADS["bf16-ragged-bs8"]
    cl = wl.context_lengths(w).double()
    assert cl.min() < 64 and cl.max() > 4096
    # log-uniform: log c is roughly uniform on [ln 16, ln 16384]
    lc = torch.log(cl)
    assert abs(float(lc.mean()) - 0.5 * (math.log(16) + math.log(16384))) < 0.6


def test_poison_and_one_oracle_step():
    w = wl.WORKLOADS["tiny-fp32"]
    inp = wl.make_inputs(w)
    kp = wl.host_array(inp.k_pool)
    vp = wl.host_array(inp.v_pool)
    assert np.isnan(kp).any()
    for r in range(w.rows):
        s = int(inp.slot_mapping[r])
        b, off = divmod(s, w.block_size)
        assert np.isnan(kp[b, off]).all()  # the new token's slot is empty before the step
    rc = oracle.kv_append(kp, vp, wl.host_array(inp.k_new), wl.host_array(inp.v_new),
                          inp.slot_mapping.numpy())
    assert rc == oracle.OK
    out, lse = oracle.paged_decode(wl.host_array(inp.q), kp, vp, inp.block_tables.numpy(),
                                   inp.context_lens.numpy(), w.softmax_scale)
    assert np.isfinite(out).all() and np.isfinite(lse).all()


def test_row_subproblem_is_the_same_read():
    w = wl.WORKLOADS["tiny-fp32"]
    inp = wl.make_inputs(w)
    kp, vp = wl.host_array(inp.k_pool), wl.host_array(inp.v_pool)
    oracle.kv_append(kp, vp, wl.host_array(inp.k_new), wl.host_array(inp.v_new),
                     inp.slot_mapping.numpy())
    full, _ = oracle.paged_decode(wl.host_array(inp.q), kp, vp, inp.block_tables.numpy(),
                                  inp.context_lens.numpy(), w.softmax_scale)
    sub = wl.row_subproblem(inp, [1])
    skp, svp = sub["k_pool"], sub["v_pool"]
    oracle.kv_append(skp, svp, sub["k_new"], sub["v_new"], sub["slot_mapping"])
    part, _ = oracle.paged_decode(sub["q"], skp, svp, sub["block_tables"],
                                  sub["context_lens"], w.softmax_scale)
    assert np.array_equal(part[0], full[1])
