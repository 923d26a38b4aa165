"""The balanced read's partition arithmetic, modelled on the CPU.

The read lays the virtual rows' chunks end to end and gives CTA b the
chunks [floor(b*W/Pe), floor((b+1)*W/Pe)); its merge needs, for every row
cut between CTAs, the first and last covering CTA and the slot of the
first one's partial.  The kernel computes those in closed form (the first
CTA b0 = ceil((pre[v] + 1)*Pe/W) - 1, the last bl = min(Pe - 1,
(pre[v+1]*Pe - 1) // W), slot 0 exactly when floor(b0*W/Pe) >= pre[v]).
This test models the partition directly (each CTA's start found by a
binary search over the prefix, as the kernel does) and checks the closed
forms against it by brute force over random length mixes.
"""
import random


def _partition(chunks, P):
    V = len(chunks)
    pre = [0]
    for x in chunks:
        pre.append(pre[-1] + x)
    W = pre[V]
    Pe = min(P, max(1, (W + 3) // 4))

    def point(bb):
        u = W if bb >= Pe else bb * W // Pe
        lo, hi = 0, V
        while lo < hi:  # the last v with pre[v] <= u
            mid = (lo + hi + 1) >> 1
            if pre[mid] <= u:
                lo = mid
            else:
                hi = mid - 1
        return lo, (u - pre[lo]) if lo < V else 0

    return pre, W, Pe, [point(bb) for bb in range(P + 1)]


def test_closed_forms_match_the_partition():
    rnd = random.Random(5)
    cut_rows = 0
    for _ in range(3000):
        V = rnd.randint(1, 40)
        P = rnd.choice([1, 2, 7, 19, 64, 152, 160])
        chunks = [0 if rnd.random() < 0.15 else rnd.randint(1, rnd.choice([2, 50, 5000]))
                  for _ in range(V)]
        if sum(chunks) == 0:
            continue
        pre, W, Pe, pts = _partition(chunks, P)
        # brute force: CTA b begins row v and cuts it when its range ends
        # inside v and it did not start after v's first chunk
        owner = {}
        for b in range(P):
            (vb, tb), (ve, te) = pts[b], pts[b + 1]
            if te > 0 and ve < V and (vb < ve or tb == 0):
                assert ve not in owner
                owner[ve] = b
        for v in range(V):
            if chunks[v] == 0:
                continue
            b0 = -(-(pre[v] + 1) * Pe // W) - 1
            bl = min(Pe - 1, (pre[v + 1] * Pe - 1) // W)
            covering = [b for b in range(P) if pts[b] < (v, chunks[v]) and pts[b + 1] > (v, 0)]
            if v in owner:
                cut_rows += 1
                assert owner[v] == b0 and covering[0] == b0
                assert bl == covering[-1] and b0 < bl
                slot = 0 if b0 * W // Pe >= pre[v] else 1
                assert slot == (0 if pts[b0][0] == v else 1)
                # every later covering CTA starts inside row v
                assert all(pts[c][0] == v and pts[c][1] > 0 for c in range(b0 + 1, bl + 1))
            else:
                assert b0 == bl and covering == [b0]
    assert cut_rows > 1000


def test_chunk_shares_differ_by_at_most_one():
    rnd = random.Random(6)
    for _ in range(500):
        chunks = [rnd.randint(0, 3000) for _ in range(rnd.randint(1, 64))]
        if sum(chunks) == 0:
            continue
        P = rnd.choice([19, 152, 160])
        pre, W, Pe, pts = _partition(chunks, P)
        shares = [(b + 1) * W // Pe - b * W // Pe for b in range(Pe)]
        assert sum(shares) == W and max(shares) - min(shares) <= 1
        assert min(shares) >= 3 or Pe == 1
