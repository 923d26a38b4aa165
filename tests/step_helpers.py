"""Run one decode step on the GPU (through the C ABI) and on the oracle."""
from __future__ import annotations

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


def assert_parity(got: torch.Tensor | np.ndarray, ref: np.ndarray, dtype: str, what: str = ""):
    g = to64(got) if isinstance(got, torch.Tensor) else np.asarray(got, dtype=np.float64)
    atol, rtol = wl.TOLERANCE[dtype]
    assert g.shape == ref.shape, (g.shape, ref.shape)
    err = np.abs(g - ref)
    bound = atol + rtol * np.abs(ref)
    bad = ~(err <= bound)
    if bad.any():
        i = np.unravel_index(np.argmax(np.where(bad, err - bound, -np.inf)), err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {err.size} outside atol={atol} rtol={rtol}; "
            f"worst at {i}: gpu={g[i]!r} oracle={ref[i]!r}; max abs err {err.max():.3e}")
    return float(err.max())
