"""Run one decode step on the GPU (through the C ABI) and on the oracle."""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
import workloads as wl


def gpu_step(npg, inp: wl.Inputs, num_splits: int | None = None, append: bool = True,
             err: torch.Tensor | None = None, stream=None, fused: bool = True):
    """Append + read (+ reduce) with the library; returns (out, num_splits, workspace)."""
    w = inp.w
    dev = inp.q.device
    bt = inp.block_tables.to(dev)
    cl = inp.context_lens.to(dev)
    sm = inp.slot_mapping.to(dev)
    if num_splits is None:
        num_splits = npg.np_paged_decode_plan(w.rows, w.q_heads, w.kv_heads, w.head_dim,
                                              w.block_size, bt.shape[1], w.torch_dtype)
    ws = npg.workspace(w.rows, w.q_heads, w.head_dim, num_splits, device=dev,
                       query_len=w.query_len)
    out = torch.full_like(inp.q, float("nan"))
    kw = dict(k_new=inp.k_new, v_new=inp.v_new, slot_mapping=sm) if append else {}
    npg.decode_step(out, inp.q, inp.k_pool, inp.v_pool, bt, cl, w.softmax_scale,
                    num_splits=num_splits, workspace=ws, err_word=err, stream=stream,
                    fused=fused, **kw)
    torch.cuda.synchronize()
    return out, num_splits, ws


def oracle_append(kp, vp, host: dict) -> int:
    """The step's append on the host copies (new tokens flattened to [T, Hk, D])."""
    hk, d = kp.shape[2], kp.shape[3]
    return oracle.kv_append(kp, vp, host["k_new"].reshape(-1, hk, d),
                            host["v_new"].reshape(-1, hk, d), host["slot_mapping"].reshape(-1))


def oracle_step(host: dict, scale: float, append: bool = True, **kw):
    kp, vp = host["k_pool"].copy(), host["v_pool"].copy()
    if append:
        rc = oracle_append(kp, vp, host)
        assert rc == oracle.OK
    return oracle.paged_decode(host["q"], kp, vp, host["block_tables"], host["context_lens"],
                               scale, **kw)


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().double().numpy()


def error_stats(got: np.ndarray, ref: np.ndarray, dtype: str) -> dict:
    """How close the GPU result is to the oracle: the largest and the 99.9th
    percentile absolute error, and the largest error as a fraction of the
    gate's bound (atol + rtol * |ref|) -- 1.0 is the edge of the gate."""
    atol, rtol = wl.TOLERANCE[dtype]
    err = np.abs(got - ref)
    frac = err / (atol + rtol * np.abs(ref))
    flat = err.reshape(-1)
    return {"max_abs": float(np.max(flat)) if flat.size else 0.0,
            "p999_abs": float(np.quantile(flat, 0.999)) if flat.size else 0.0,
            "max_frac_of_tol": float(np.max(frac)) if frac.size else 0.0,
            "n": int(flat.size)}


def assert_parity(got: torch.Tensor | np.ndarray, ref: np.ndarray, dtype: str, what: str = ""):
    """Element-wise gate: |gpu - oracle| <= atol + rtol * |oracle| everywhere
    (NaN fails).  Returns the error statistics (error_stats)."""
    g = to64(got) if isinstance(got, torch.Tensor) else np.asarray(got, dtype=np.float64)
    atol, rtol = wl.TOLERANCE[dtype]
    assert g.shape == ref.shape, (g.shape, ref.shape)
    err = np.abs(g - ref)
    bound = atol + rtol * np.abs(ref)
    bad = ~(err <= bound)
    if bad.any():
        i = np.unravel_index(np.argmax(np.where(bad, err - bound, -np.inf)), err.shape)
        fin = err[np.isfinite(err)]
        p999 = float(np.quantile(fin, 0.999)) if fin.size else float("nan")
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {err.size} outside atol={atol} rtol={rtol}; "
            f"worst at {i}: gpu={g[i]!r} oracle={ref[i]!r}; max abs err {np.nanmax(err):.3e} "
            f"(p99.9 {p999:.3e}; the margin is the error over atol + rtol*|oracle|)")
    return error_stats(g, ref, dtype)


# ------------------------------------------------------ full-size steps ---
def host_copy(t: torch.Tensor) -> np.ndarray:
    """A host numpy array of ``t``'s bytes (bf16 as its raw uint16 pattern),
    made with one device-to-host copy (full-size pools are GBs)."""
    c = t.detach().to("cpu")
    if c.dtype == torch.bfloat16:
        return c.view(torch.int16).numpy().view(np.uint16)
    return c.numpy()


def host_inputs(inp: wl.Inputs) -> dict:
    """Host copies of every input of a step, whole pools included.  Take
    them before any kernel touches the pools."""
    return dict(q=host_copy(inp.q), k_new=host_copy(inp.k_new), v_new=host_copy(inp.v_new),
                k_pool=host_copy(inp.k_pool), v_pool=host_copy(inp.v_pool),
                block_tables=inp.block_tables.numpy().copy(),
                context_lens=inp.context_lens.numpy().astype(np.int32),
                slot_mapping=inp.slot_mapping.numpy().copy())


def oracle_step_in_place(host: dict, scale: float, threads: int | None = None):
    """The whole step on the oracle, for full-size inputs: the append
    written into ``host``'s own pool copies (no further copy of the pools),
    then every row's read.  Rows are independent, so they are dealt over
    host threads (longest first, each to the least loaded thread); each
    thread runs the oracle on its rows against the shared pools (the C calls
    release the interpreter lock).  Returns (out, lse) for all rows."""
    from concurrent.futures import ThreadPoolExecutor

    rc = oracle_append(host["k_pool"], host["v_pool"], host)
    assert rc == oracle.OK
    cl = host["context_lens"]
    rows = cl.shape[0]
    n = max(1, min(rows, threads or len(os.sched_getaffinity(0))))
    load = [0] * n
    parts: list[list[int]] = [[] for _ in range(n)]
    for r in sorted(range(rows), key=lambda r: -int(cl[r])):
        i = min(range(n), key=lambda i: load[i])
        parts[i].append(r)
        load[i] += int(cl[r]) + 1

    def run(idx):
        idx = np.array(sorted(idx), dtype=np.int64)
        o, l = oracle.paged_decode(host["q"][idx], host["k_pool"], host["v_pool"],
                                   host["block_tables"][idx], cl[idx], scale)
        return idx, o, l

    out = lse = None
    with ThreadPoolExecutor(n) as ex:
        for idx, o, l in ex.map(run, [p for p in parts if p]):
            if out is None:
                out = np.zeros((rows,) + o.shape[1:], dtype=o.dtype)
                lse = np.zeros((rows,) + l.shape[1:], dtype=l.dtype)
            out[idx], lse[idx] = o, l
    return out, lse


def assert_pool_equal(dev_pool: torch.Tensor, host_pool: np.ndarray, what: str,
                      chunk_blocks: int = 2048) -> None:
    """The device pool equals ``host_pool`` byte for byte, compared in
    chunks of blocks (NaN payloads included)."""
    nb = dev_pool.shape[0]
    assert host_pool.shape == tuple(dev_pool.shape), what
    for s in range(0, nb, chunk_blocks):
        e = min(nb, s + chunk_blocks)
        got = host_copy(dev_pool[s:e])
        want = host_pool[s:e]
        if not np.array_equal(got.view(np.uint8), want.view(np.uint8)):
            ne = got.view(np.uint8) != want.view(np.uint8)
            diff = np.nonzero(np.any(ne.reshape(e - s, -1), axis=1))[0]
            raise AssertionError(f"{what}: blocks {(diff + s)[:8].tolist()} differ "
                                 f"({diff.size} in blocks {s}..{e - 1})")
