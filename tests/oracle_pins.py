"""Pins for the CPU oracle: checks against facts fixed outside the oracle.

Each ``check_*`` takes an oracle library handle and raises AssertionError if
the oracle disagrees with the fact it pins.  ``test_oracle_pins.py`` runs
them on the real oracle; ``test_oracle_mutants.py`` runs them on copies of
the oracle with one planted mistake each and requires that some check fails.

What pins what:
  * library conversions: the oracle's bf16 widening equals torch's;
  * library special case: with any block table, the read equals torch SDPA
    (fp64, GQA via ``enable_gqa``) over the contiguous history the pool was
    filled from -- the pool is filled by walking each table block by block,
    not by the oracle's div/mod form;  lse equals ``torch.logsumexp`` of the
    scores;
  * invariants: permuting physical blocks (and the tables with them) changes
    nothing, bit for bit (paging changes where K/V are stored, never the attention result:
    "Day 17: paging under the sampling path", Diagram);  NaN in every slot outside the history never reaches the
    output;
  * closed forms: one token gives exactly V_0; zero scale or zero query gives
    the mean of V and lse = log(c); identical keys give the mean of V; one
    dominant score gives that token's V;
  * brute force: every ordered choice of blocks from a 4-block pool;
  * split identity: per-split partials combined by the reduce equal the
    unsplit read, each partial equals SDPA over its own token range;
  * append: equals torch's indexed assignment, bit for bit; negative slots
    skipped; out-of-pool slots refused.
"""
from __future__ import annotations

import itertools
import math

import numpy as np
import torch
import torch.nn.functional as F

import oracle

RNG_SEED = 1234


def _bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 bit pattern array."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16).copy()


def _tt(a: np.ndarray) -> torch.Tensor:
    """A torch copy of a storage array (bf16 bits as int16, for indexing)."""
    a = np.ascontiguousarray(a).copy()
    return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)


def _store(x64: np.ndarray, dtype: str):
    """Round float64 values to the storage dtype.

    Returns (storage array for the oracle, the exact float64 values stored).
    """
    t = torch.from_numpy(np.asarray(x64, dtype=np.float64))
    if dtype == "f32":
        s = t.to(torch.float32)
        return s.numpy().copy(), s.double().numpy()
    s = t.to(torch.bfloat16)
    return _bits(s), s.double().numpy()


def _case(rng: np.random.Generator, contexts, q_heads, kv_heads, head_dim,
          block_size, dtype="f32", spare_blocks=3, scale=None):
    """Random contiguous histories, scattered into a pool by random tables.

    The pool is filled by walking each row's table one block at a time and
    each block one offset at a time (logical block j of the row is physical
    block table[j]); every slot not written holds NaN.
    """
    rows = len(contexts)
    needed = [-(-c // block_size) for c in contexts]
    nb = sum(needed) + spare_blocks
    mb = max(max(needed), 1)
    perm = rng.permutation(nb)
    tables = np.full((rows, mb), -1, dtype=np.int32)
    pos = 0
    for r, n in enumerate(needed):
        tables[r, :n] = perm[pos:pos + n]
        pos += n
    q_st, q64 = _store(rng.standard_normal((rows, q_heads, head_dim)), dtype)
    hist_k, hist_v = [], []
    kp64 = np.full((nb, block_size, kv_heads, head_dim), np.nan)
    vp64 = np.full((nb, block_size, kv_heads, head_dim), np.nan)
    for r, c in enumerate(contexts):
        _, hk = _store(rng.standard_normal((c, kv_heads, head_dim)), dtype)
        _, hv = _store(rng.standard_normal((c, kv_heads, head_dim)), dtype)
        hist_k.append(hk)
        hist_v.append(hv)
        t = 0
        for j in range(needed[r]):
            b = tables[r, j]
            for off in range(block_size):
                if t == c:
                    break
                kp64[b, off] = hk[t]
                vp64[b, off] = hv[t]
                t += 1
    kp, _ = _store(kp64, dtype)
    vp, _ = _store(vp64, dtype)
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)
    return dict(q=q_st, q64=q64, k_pool=kp, v_pool=vp, block_tables=tables,
                context_lens=np.asarray(contexts, dtype=np.int32),
                hist_k=hist_k, hist_v=hist_v, scale=scale)


def _sdpa(q64_row, hk, hv, scale):
    """torch SDPA in fp64 for one row: q [Hq, D], history [c, Hk, D] -> [Hq, D]."""
    q = torch.from_numpy(q64_row)[None, :, None, :]
    k = torch.from_numpy(hk).permute(1, 0, 2)[None]
    v = torch.from_numpy(hv).permute(1, 0, 2)[None]
    out = F.scaled_dot_product_attention(q, k, v, scale=scale, enable_gqa=True)
    return out[0, :, 0, :].numpy()


def _lse(q64_row, hk, scale):
    """torch.logsumexp of the fp64 scores; query head h uses kv head h // g."""
    q = torch.from_numpy(q64_row)
    k = torch.from_numpy(hk)  # [c, Hk, D]
    g = q.shape[0] // k.shape[1]
    kk = k.repeat_interleave(g, dim=1)  # [c, Hq, D]
    s = torch.einsum("hd,thd->ht", q, kk) * scale
    return torch.logsumexp(s, dim=1).numpy()


def _run(lib, c, **kw):
    return oracle.paged_decode(c["q"], c["k_pool"], c["v_pool"], c["block_tables"],
                               c["context_lens"], c["scale"], lib=lib, **kw)


SHAPES = [
    # contexts, q_heads, kv_heads, head_dim, block_size, dtype
    ([1, 7, 13], 4, 2, 8, 4, "f32"),
    ([16, 64], 4, 2, 16, 8, "f32"),
    ([5, 33, 2], 3, 3, 8, 8, "f32"),        # MHA (group 1)
    ([9, 20], 10, 2, 8, 4, "bf16"),         # group 5
    ([40, 1, 17], 8, 1, 16, 16, "bf16"),    # group 8, one kv head
]


def check_widen(lib):
    g = torch.Generator().manual_seed(RNG_SEED)
    x = torch.randn(257, generator=g) * 100
    x[:6] = torch.tensor([0.0, -0.0, float("inf"), float("-inf"), 1e-40, 3.0e38])
    b = x.to(torch.bfloat16)
    bits = _bits(b)
    ref = b.double().numpy()
    for i in range(len(ref)):
        got = oracle.widen(bits, i, lib=lib)
        assert got == ref[i] or (math.isnan(got) and math.isnan(ref[i])), (i, got, ref[i])
    f = x.numpy().astype(np.float32)
    for i in range(len(f)):
        assert oracle.widen(f, i, lib=lib) == float(f[i])


def check_sdpa_equivalence(lib):
    rng = np.random.default_rng(RNG_SEED)
    for contexts, hq, hk, d, bs, dt in SHAPES:
        c = _case(rng, contexts, hq, hk, d, bs, dt)
        out, lse = _run(lib, c)
        for r in range(len(contexts)):
            ref = _sdpa(c["q64"][r], c["hist_k"][r], c["hist_v"][r], c["scale"])
            np.testing.assert_allclose(out[r], ref, rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse[r], _lse(c["q64"][r], c["hist_k"][r], c["scale"]),
                                       rtol=0, atol=1e-12)


def check_paging_invariance(lib):
    rng = np.random.default_rng(RNG_SEED + 1)
    for contexts, hq, hk, d, bs, dt in SHAPES:
        c = _case(rng, contexts, hq, hk, d, bs, dt)
        out, lse = _run(lib, c)
        nb = c["k_pool"].shape[0]
        pi = rng.permutation(nb)           # physical block b moves to pi[b]
        kp = np.empty_like(c["k_pool"])
        vp = np.empty_like(c["v_pool"])
        kp[pi] = c["k_pool"]
        vp[pi] = c["v_pool"]
        bt = c["block_tables"].copy()
        used = bt >= 0
        bt[used] = pi[bt[used]]
        c2 = dict(c, k_pool=kp, v_pool=vp, block_tables=bt)
        out2, lse2 = _run(lib, c2)
        assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def check_poison_never_read(lib):
    rng = np.random.default_rng(RNG_SEED + 2)
    for contexts, hq, hk, d, bs, dt in SHAPES:
        c = _case(rng, contexts, hq, hk, d, bs, dt)
        out, lse = _run(lib, c)
        assert np.isfinite(out).all() and np.isfinite(lse).all()


def check_closed_forms(lib):
    rng = np.random.default_rng(RNG_SEED + 3)
    # one token: output is V_0 exactly, lse is the single score
    c = _case(rng, [1, 1], 4, 2, 8, 4, "f32")
    out, lse = _run(lib, c)
    for r in range(2):
        v0 = c["hist_v"][r][0]                    # [Hk, D]
        assert np.array_equal(out[r], np.repeat(v0, 2, axis=0))
        s = (c["q64"][r] * np.repeat(c["hist_k"][r][0], 2, axis=0)).sum(-1) * c["scale"]
        np.testing.assert_allclose(lse[r], s, rtol=0, atol=1e-12)
    # zero scale: uniform weights -> mean of V, lse = log(c)
    contexts = [3, 10, 25]
    c = _case(rng, contexts, 6, 2, 8, 4, "f32", scale=0.0)
    out, lse = _run(lib, c)
    for r, n in enumerate(contexts):
        mean = np.repeat(c["hist_v"][r].mean(axis=0), 3, axis=0)
        np.testing.assert_allclose(out[r], mean, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[r], math.log(n), rtol=0, atol=1e-12)
    # zero query: same
    c = _case(rng, contexts, 6, 2, 8, 4, "f32")
    c["q"] = np.zeros_like(c["q"])
    out, lse = _run(lib, c)
    for r, n in enumerate(contexts):
        mean = np.repeat(c["hist_v"][r].mean(axis=0), 3, axis=0)
        np.testing.assert_allclose(out[r], mean, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[r], math.log(n), rtol=0, atol=1e-12)
    # identical keys: every score equal -> mean of V, whatever q is
    c = _case(rng, [12], 2, 1, 8, 4, "f32")
    kp = c["k_pool"]
    bt = c["block_tables"][0]
    row = rng.standard_normal(8).astype(np.float32)
    for j in range(3):
        kp[bt[j]] = row
    out, _ = _run(lib, c)
    mean = c["hist_v"][0].mean(axis=0)            # [1, D]
    np.testing.assert_allclose(out[0], np.repeat(mean, 2, axis=0), rtol=0, atol=1e-12)
    # one dominant score: key 7 parallel to q with a huge score -> its V
    c = _case(rng, [12], 1, 1, 8, 4, "f32")
    t = 7
    qv = c["q"][0, 0]
    b, off = c["block_tables"][0, t // 4], t % 4
    c["k_pool"][b, off, 0] = (qv / np.dot(qv, qv) * 4000.0).astype(np.float32)
    out, _ = _run(lib, c)
    np.testing.assert_allclose(out[0, 0], c["hist_v"][0][t, 0], rtol=0, atol=1e-12)


def check_brute_force_tables(lib):
    """All ordered choices of blocks from a 4-block pool, every context length."""
    rng = np.random.default_rng(RNG_SEED + 4)
    bs, nb, hq, hk, d = 2, 4, 2, 1, 4
    pool_k = rng.standard_normal((nb, bs, hk, d)).astype(np.float32)
    pool_v = rng.standard_normal((nb, bs, hk, d)).astype(np.float32)
    q = rng.standard_normal((1, hq, d)).astype(np.float32)
    scale = 0.7
    for n in range(1, nb + 1):
        for tab in itertools.permutations(range(nb), n):
            for c in range(2 * n - 1, 2 * n + 1):
                # the history in logical order: block tab[0], offsets 0..bs-1, ...
                hkk = np.concatenate([pool_k[b] for b in tab])[:c].astype(np.float64)
                hvv = np.concatenate([pool_v[b] for b in tab])[:c].astype(np.float64)
                s = np.einsum("hd,td->ht", q[0].astype(np.float64), hkk[:, 0]) * scale
                w = np.exp(s - s.max(axis=1, keepdims=True))
                ref = (w @ hvv[:, 0]) / w.sum(axis=1, keepdims=True)
                bt = np.array([list(tab)], dtype=np.int32)
                out, _ = oracle.paged_decode(q, pool_k, pool_v, bt, [c], scale, lib=lib)
                np.testing.assert_allclose(out[0], ref, rtol=0, atol=1e-12)


def check_splits(lib):
    rng = np.random.default_rng(RNG_SEED + 5)
    contexts = [1, 37, 64, 100]
    c = _case(rng, contexts, 4, 2, 8, 8, "f32")
    full, full_lse = _run(lib, c)
    cap = c["block_tables"].shape[1] * 8
    for split_len in (8, 16, 24, 64):
        ns = -(-cap // split_len)
        part, plse = _run(lib, c, split_len=split_len, num_splits=ns)
        for r, n in enumerate(contexts):
            for s in range(ns):
                tb, te = s * split_len, min((s + 1) * split_len, n)
                if tb >= te:
                    assert np.all(plse[r, :, s] == -np.inf)
                    assert np.all(part[r, :, s] == 0)
                    continue
                ref = _sdpa(c["q64"][r], c["hist_k"][r][tb:te], c["hist_v"][r][tb:te], c["scale"])
                np.testing.assert_allclose(part[r, :, s], ref, rtol=0, atol=1e-12)
                np.testing.assert_allclose(
                    plse[r, :, s], _lse(c["q64"][r], c["hist_k"][r][tb:te], c["scale"]),
                    rtol=0, atol=1e-12)
        merged = oracle.reduce(part, plse, lib=lib)
        np.testing.assert_allclose(merged, full, rtol=0, atol=1e-12)
        # the lse of the whole row is the logsumexp of the split lse's
        m = torch.logsumexp(torch.from_numpy(plse), dim=2).numpy()
        np.testing.assert_allclose(m, full_lse, rtol=0, atol=1e-12)


def check_reduce_cases(lib):
    # two splits, lse log 1 and log 3: weights 1/4 and 3/4
    o = np.array([[[[4.0, 0.0], [0.0, 8.0]]]])
    lse = np.array([[[0.0, math.log(3.0)]]])
    np.testing.assert_allclose(oracle.reduce(o, lse, lib=lib)[0, 0], [1.0, 6.0],
                               rtol=0, atol=1e-14)
    # an empty split (lse -inf, garbage o) is ignored
    o = np.array([[[[2.0, 2.0], [np.nan, np.nan], [4.0, -2.0]]]])
    lse = np.array([[[1.5, -np.inf, 1.5]]])
    np.testing.assert_allclose(oracle.reduce(o, lse, lib=lib)[0, 0], [3.0, 0.0],
                               rtol=0, atol=1e-14)
    # all empty: zeros
    o = np.full((1, 1, 3, 2), np.nan)
    lse = np.full((1, 1, 3), -np.inf)
    assert np.array_equal(oracle.reduce(o, lse, lib=lib), np.zeros((1, 1, 2)))
    # shift invariance: adding a constant to every lse changes nothing
    rng = np.random.default_rng(RNG_SEED + 6)
    o = rng.standard_normal((2, 3, 5, 4))
    lse = rng.standard_normal((2, 3, 5)) * 3
    a = oracle.reduce(o, lse, lib=lib)
    b = oracle.reduce(o, lse + 123.25, lib=lib)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def check_f32_twin(lib):
    """The fp32 instantiation agrees with fp64 far inside 1e-5 / 1e-4."""
    rng = np.random.default_rng(RNG_SEED + 7)
    c = _case(rng, [300, 1000, 2048], 16, 4, 64, 16, "f32", spare_blocks=5)
    a, la = _run(lib, c, precision="f64")
    b, lb = _run(lib, c, precision="f32")
    assert np.abs(a - b).max() < 1e-6
    assert np.abs(la - lb).max() < 1e-5


def check_append(lib):
    rng = np.random.default_rng(RNG_SEED + 8)
    for dt in ("f32", "bf16"):
        nb, bs, hk, d = 6, 4, 2, 8
        kp, _ = _store(rng.standard_normal((nb, bs, hk, d)), dt)
        vp, _ = _store(rng.standard_normal((nb, bs, hk, d)), dt)
        kn, _ = _store(rng.standard_normal((5, hk, d)), dt)
        vn, _ = _store(rng.standard_normal((5, hk, d)), dt)
        slots = np.array([3, -1, 23, 0, 9], dtype=np.int64)
        ref_k = _tt(kp).view(nb * bs, hk, d)
        ref_v = _tt(vp).view(nb * bs, hk, d)
        keep = torch.from_numpy(slots >= 0)
        idx = torch.from_numpy(slots)[keep]
        ref_k[idx] = _tt(kn)[keep]
        ref_v[idx] = _tt(vn)[keep]
        k2, v2 = kp.copy(), vp.copy()
        rc = oracle.kv_append(k2, v2, kn, vn, slots, lib=lib)
        assert rc == oracle.OK
        assert k2.tobytes() == ref_k.numpy().tobytes()
        assert v2.tobytes() == ref_v.numpy().tobytes()
        # a slot past the pool is refused; the others are still written
        k3, v3 = kp.copy(), vp.copy()
        bad = np.array([2, nb * bs, 5], dtype=np.int64)
        rc = oracle.kv_append(k3, v3, kn[:3], vn[:3], bad, lib=lib)
        assert rc == oracle.BAD_BLOCK
        r3 = _tt(kp).view(nb * bs, hk, d)
        r3[torch.tensor([2, 5])] = _tt(kn[[0, 2]])
        assert k3.tobytes() == r3.numpy().tobytes()


def check_refusals(lib):
    rng = np.random.default_rng(RNG_SEED + 9)
    c = _case(rng, [10, 5], 4, 2, 8, 4, "f32")
    bt = c["block_tables"].copy()
    bt[0, 1] = c["k_pool"].shape[0]             # a block past the pool
    try:
        _run(lib, dict(c, block_tables=bt))
        raise AssertionError("out-of-pool block id accepted")
    except oracle.OracleError as e:
        assert e.code == oracle.BAD_BLOCK
    try:
        _run(lib, dict(c, context_lens=np.array([10, 13], np.int32)))
        raise AssertionError("context past the table accepted")
    except oracle.OracleError as e:
        assert e.code == oracle.BAD_CONTEXT
    try:
        _run(lib, dict(c, q=np.zeros((2, 3, 8), np.float32)))
        raise AssertionError("q_heads not a multiple of kv_heads accepted")
    except oracle.OracleError as e:
        assert e.code == oracle.BAD_ARG
    # zero context: zeros and lse = -inf
    out, lse = _run(lib, dict(c, context_lens=np.array([0, 5], np.int32)))
    assert np.all(out[0] == 0) and np.all(lse[0] == -np.inf) and np.isfinite(out[1]).all()


def _mq_case(rng, contexts, query_len, q_heads, kv_heads, head_dim, block_size, dtype="f32"):
    c = _case(rng, contexts, q_heads, kv_heads, head_dim, block_size, dtype)
    rows = len(contexts)
    q_st, q64 = _store(rng.standard_normal((rows, query_len, q_heads, head_dim)), dtype)
    c["q"], c["q64"] = q_st, q64
    return c


def _sdpa_causal(q64_row, hk, hv, scale):
    """torch SDPA (fp64) of Q query tokens that are the last Q positions of a
    c-token history: query i may see positions t <= c - Q + i."""
    qn, c = q64_row.shape[0], hk.shape[0]
    q = torch.from_numpy(q64_row).permute(1, 0, 2)[None]          # [1, Hq, Q, D]
    k = torch.from_numpy(hk).permute(1, 0, 2)[None]               # [1, Hk, c, D]
    v = torch.from_numpy(hv).permute(1, 0, 2)[None]
    pos = torch.arange(c)[None, :]
    lim = (c - qn + torch.arange(qn))[:, None]
    mask = pos <= lim                                             # [Q, c]
    out = F.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=scale, enable_gqa=True)
    return out[0].permute(1, 0, 2).numpy()                         # [Q, Hq, D]


def check_multi_query_sdpa(lib):
    rng = np.random.default_rng(RNG_SEED + 10)
    for contexts, qn, hq, hk, d, bs, dt in [
        ([5, 40, 17], 3, 4, 2, 8, 4, "f32"),
        ([64, 9], 4, 8, 2, 16, 8, "bf16"),
        ([33, 100], 2, 10, 2, 8, 16, "f32"),
    ]:
        c = _mq_case(rng, contexts, qn, hq, hk, d, bs, dt)
        out, lse = _run(lib, c)
        assert out.shape == (len(contexts), qn, hq, d)
        for r in range(len(contexts)):
            ref = _sdpa_causal(c["q64"][r], c["hist_k"][r], c["hist_v"][r], c["scale"])
            np.testing.assert_allclose(out[r], ref, rtol=0, atol=1e-12)
            for i in range(qn):
                e = contexts[r] - qn + i + 1
                np.testing.assert_allclose(
                    lse[r, i], _lse(c["q64"][r][i], c["hist_k"][r][:e], c["scale"]),
                    rtol=0, atol=1e-12)


def check_multi_query_prefix(lib):
    """Query i of a Q-token read is the one-token read of the history's first
    c - Q + i + 1 positions, bit for bit (same tokens, same order)."""
    rng = np.random.default_rng(RNG_SEED + 11)
    contexts, qn = [20, 7, 33], 4
    c = _mq_case(rng, contexts, qn, 4, 2, 8, 4, "f32")
    out, lse = _run(lib, c)
    for i in range(qn):
        ctx_i = np.array([n - qn + i + 1 for n in contexts], dtype=np.int32)
        single = dict(c, q=c["q"][:, i], context_lens=ctx_i)
        o1, l1 = _run(lib, single)
        assert np.array_equal(out[:, i], o1) and np.array_equal(lse[:, i], l1)


def check_multi_query_splits_and_short_rows(lib):
    rng = np.random.default_rng(RNG_SEED + 12)
    contexts, qn = [2, 50, 90], 3
    c = _mq_case(rng, contexts, qn, 4, 2, 8, 8, "f32")
    full, full_lse = _run(lib, c)
    part, plse = _run(lib, c, split_len=16, num_splits=12)
    merged = oracle.reduce(part.reshape(3, qn * 4, 12, 8), plse.reshape(3, qn * 4, 12), lib=lib)
    np.testing.assert_allclose(merged.reshape(3, qn, 4, 8), full, rtol=0, atol=1e-12)
    # a row shorter than the query run: its first query tokens see nothing
    c2 = _mq_case(rng, [2], 4, 4, 2, 8, 8, "f32")
    out, lse = _run(lib, c2)
    assert np.all(out[0, :2] == 0) and np.all(lse[0, :2] == -np.inf)
    assert np.isfinite(out[0, 2:]).all()


ALL_CHECKS = [
    check_widen,
    check_sdpa_equivalence,
    check_paging_invariance,
    check_poison_never_read,
    check_closed_forms,
    check_brute_force_tables,
    check_splits,
    check_reduce_cases,
    check_f32_twin,
    check_append,
    check_refusals,
    check_multi_query_sdpa,
    check_multi_query_prefix,
    check_multi_query_splits_and_short_rows,
]
