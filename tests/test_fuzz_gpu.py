"""GPU parity on seeded random shapes: every supported combination of dtype,
head_dim, GQA group, kv heads, block size, query tokens, ragged contexts
(empty and one-token rows included), schedule (balanced, unsplit, split) and
append (fused or separate) is drawn at random, small enough for the oracle,
and compared element by element with it; the pools after the append must
match the oracle's bit for bit.
"""
from __future__ import annotations

import random

import pytest

import workloads as wl
from test_parity_gpu import _full_parity

pytestmark = pytest.mark.gpu

N_CASES = 60


def _draw(i: int):
    rnd = random.Random(1000 + i)
    dtype = rnd.choice(["bf16", "f32"])
    head_dim = rnd.choice([16, 32, 64, 128, 256])
    group = rnd.choice([1, 2, 3, 4, 5, 6, 7, 8, 16] if dtype == "bf16" else [1, 2, 3, 4, 5, 6, 7, 8])
    kv_heads = rnd.choice([1, 2, 3, 4, 8, 8, 12, 16])
    block_size = rnd.choice([1, 3, 8, 16, 24, 32, 64])
    rows = rnd.randint(1, 12)
    # several query tokens: (query token, head) rows g*Q <= 16 on bf16, <= 8 on fp32
    hg = max(d for d in range(1, 9) if kv_heads % d == 0)  # kv heads per CTA
    bt = 1  # bf16 TMA box tokens: the largest power of two dividing the block, <= 16
    while bt < (8 if head_dim >= 256 else 16) and block_size % (2 * bt) == 0:
        bt *= 2
    balanced_ok = (head_dim % (64 if dtype == "bf16" else 32) == 0
                   and (dtype == "f32" or (bt * hg) % 8 == 0))
    q_max = (16 if dtype == "bf16" else 8) // group
    query_len = rnd.choice([1, 1, 1, max(1, min(q_max, rnd.randint(2, 5)))])
    budget = 60_000 // (kv_heads * max(head_dim, 32))  # keeps the oracle fast
    ctx = []
    for _ in range(rows):
        kind = rnd.random()
        if kind < 0.1:
            ctx.append(0)
        elif kind < 0.2:
            ctx.append(1)
        else:
            ctx.append(rnd.randint(query_len, max(query_len, min(budget, 3000))))
    if all(c == 0 for c in ctx):
        ctx[0] = 5
    if query_len > 1:  # rows hold their query run (shorter rows are covered elsewhere)
        ctx = [max(c, query_len) if c else 0 for c in ctx]
    sched = rnd.choice([1, rnd.randint(2, 9)])
    if balanced_ok and rnd.random() < 0.7:
        sched = 0  # the default schedule where it applies
    fused = rnd.random() < 0.6
    w = wl.Workload(f"fuzz-{i}", rows=rows, q_heads=kv_heads * group, kv_heads=kv_heads,
                    head_dim=head_dim, block_size=block_size, dtype=dtype,
                    ctx=("fixed", tuple(ctx)), pool=("spare", rnd.randint(0, 5)),
                    seed=2000 + i, query_len=query_len)
    return w, sched, fused


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_shape(nplib, i):
    w, sched, fused = _draw(i)
    _full_parity(nplib, w, num_splits=sched, fused=fused)
