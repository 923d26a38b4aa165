"""paged_kv_decode_np_gb300 -- GB300 (sm_103a) batched paged-attention decode.

A thin ctypes binding over ``libnp_paged.so`` (C ABI in
``include/np_paged.h``).  The functions keep the C names and only marshal
arguments: every step of the append, the read and the reduce runs in the
library's CUDA kernels.  torch supplies device memory and streams.  There is
no CPU fallback: if the library is missing, or a tensor is not on a CUDA
device, the call raises.

Typical decode step::

    import paged_kv_decode_np_gb300 as npg
    S = npg.np_paged_decode_plan(rows, q_heads, kv_heads, head_dim, block_size,
                                 max_blocks_per_row, torch.bfloat16)
    ws = npg.workspace(rows, q_heads, head_dim, S, device="cuda")   # zeroed
    npg.np_paged_append_decode(out if S <= 1 else None, q, k_new, v_new,
                               slot_mapping, k_pool, v_pool, block_tables,
                               context_lens, scale, num_splits=S, workspace=ws)
    if S > 1:
        npg.np_paged_decode_reduce(out, ws, num_splits=S)

S == 0 (the balanced read) writes ``out`` itself; S > 1 leaves split
partials for np_paged_decode_reduce.  A loop that runs the same step on the
same buffers again and again can check and convert the arguments once::

    step = npg.PreparedStep(out, q, k_new, v_new, slot_mapping, k_pool, v_pool,
                            block_tables, context_lens, scale, S, ws)
    step.launch()   # the same library calls, ~4 us of host time
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

__all__ = [
    "load", "NPError", "np_abi_version", "np_status_string", "np_kv_append",
    "np_paged_decode_plan", "np_paged_decode_split_len",
    "np_paged_decode_workspace_bytes", "np_paged_decode", "np_paged_decode_reduce",
    "np_paged_decode_noalloc", "NP_NOALLOC_SCRATCH_BYTES", "np_paged_append_decode",
    "np_selftest_bounded_wait",
    "workspace", "decode_step", "PreparedStep", "NP_OK", "NP_ERR_INVALID_ARG",
    "NP_ERR_UNSUPPORTED",
    "NP_ERR_WORKSPACE", "NP_ERR_OUT_OF_RANGE", "NP_ERR_CUDA", "NP_F32", "NP_BF16",
    "NP_FLAG_BLOCK_ID", "NP_FLAG_CONTEXT", "NP_FLAG_SLOT", "NP_FLAG_TIMEOUT", "NP_FLAG_CONFIG",
]

NP_OK = 0
NP_ERR_INVALID_ARG = 1
NP_ERR_UNSUPPORTED = 2
NP_ERR_WORKSPACE = 3
NP_ERR_OUT_OF_RANGE = 4
NP_ERR_CUDA = 5

NP_F32 = 0
NP_BF16 = 1

NP_FLAG_BLOCK_ID = 0x1
NP_FLAG_CONTEXT = 0x2
NP_FLAG_SLOT = 0x4
NP_FLAG_TIMEOUT = 0x8
NP_FLAG_CONFIG = 0x10

NP_NOALLOC_SCRATCH_BYTES = 32 << 20

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libnp_paged.so")

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_LIB: ctypes.CDLL | None = None


class NPError(RuntimeError):
    def __init__(self, status: int, call: str):
        self.status = status
        name = load().np_status_string(status).decode() if _LIB else str(status)
        super().__init__(f"{call} returned {name}")


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libnp_paged.so (built by ``__graft_entry__.build()``)."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is not built; run `python -c 'import __graft_entry__ as g; "
                           "g.build()'` (nvcc, sm_103a)")
    lib = ctypes.CDLL(p)
    lib.np_status_string.restype = ctypes.c_char_p
    lib.np_status_string.argtypes = [ctypes.c_int]
    lib.np_abi_version.restype = _I32
    lib.np_abi_version.argtypes = []
    lib.np_kv_append.restype = ctypes.c_int
    lib.np_kv_append.argtypes = [_P, _P, ctypes.c_int, _I64, _I32, _I32, _I32, _P, _P, _P,
                                 _I32, _P, _P]
    lib.np_paged_decode_plan.restype = ctypes.c_int
    lib.np_paged_decode_plan.argtypes = [_I32, _I32, _I32, _I32, _I32, _I32, ctypes.c_int,
                                         _I32, ctypes.POINTER(_I32)]
    lib.np_paged_decode_split_len.restype = _I64
    lib.np_paged_decode_split_len.argtypes = [_I32, _I32, _I32]
    lib.np_paged_decode_workspace_bytes.restype = ctypes.c_size_t
    lib.np_paged_decode_workspace_bytes.argtypes = [_I32, _I32, _I32, _I32]
    lib.np_paged_decode.restype = ctypes.c_int
    lib.np_paged_decode.argtypes = [_P, _P, _P, _P, ctypes.c_int, _I64, _I32, _I32, _I32, _P,
                                    _I32, _P, _I32, _I32, _I32, ctypes.c_float, _I32, _P,
                                    ctypes.c_size_t, _P, _P]
    lib.np_paged_append_decode.restype = ctypes.c_int
    lib.np_paged_append_decode.argtypes = [_P, _P, _P, _P, _P, _P, _P, ctypes.c_int, _I64, _I32,
                                           _I32, _I32, _P, _I32, _P, _I32, _I32, _I32,
                                           ctypes.c_float, _I32, _P, ctypes.c_size_t, _P, _P]
    lib.np_paged_decode_noalloc.restype = ctypes.c_int
    lib.np_paged_decode_noalloc.argtypes = [_P, _P, _P, _P, ctypes.c_int, _I64, _I32, _I32, _I32,
                                            _P, _I32, _P, _I32, _I32, _I32, ctypes.c_float, _I32,
                                            _P, _P]
    lib.np_paged_decode_reduce.restype = ctypes.c_int
    lib.np_paged_decode_reduce.argtypes = [_P, ctypes.c_int, _P, ctypes.c_size_t, _I32, _I32,
                                           _I32, _I32, _P]
    lib.np_selftest_bounded_wait.restype = ctypes.c_int
    lib.np_selftest_bounded_wait.argtypes = [_P, _I64, _P]
    if path is None:
        _LIB = lib
    return lib


def _check(status: int, call: str) -> None:
    if status != NP_OK:
        raise NPError(status, call)


def _dtype_code(dt) -> int:
    if dt in (torch.float32, "f32", NP_F32):
        return NP_F32
    if dt in (torch.bfloat16, "bf16", NP_BF16):
        return NP_BF16
    raise TypeError(f"unsupported dtype {dt}; the library stores float32 or bfloat16")


def _current_device() -> int:
    """The CUDA device the library's kernels launch on: torch's current one
    (the stream, the tensor maps and the no-allocation scratch all belong
    to it); -1 where CUDA cannot initialise, so that the tensors' own check
    reports the problem."""
    try:
        return torch.cuda.current_device()
    except (RuntimeError, AssertionError):
        return -1


def _dev(t: torch.Tensor, name: str, cur: int) -> int:
    """The device address of ``t``, after checking that it is a contiguous
    tensor on device ``cur`` (a tensor on another GPU would be dereferenced
    by kernels running on this one)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device (no CPU path exists)")
    if t.device.index != cur:
        raise ValueError(f"{name} is on {t.device} but the current device is cuda:{cur}; "
                         "call inside torch.cuda.device(...) of the tensors' GPU")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _opt(t: torch.Tensor | None, name: str, cur: int) -> int | None:
    return None if t is None else _dev(t, name, cur)


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        if stream.device.index != _current_device():
            raise ValueError(f"stream is on {stream.device} but the current device is "
                             f"cuda:{_current_device()}")
        return stream.cuda_stream
    return int(stream)


def _q_shape(q: torch.Tensor, name: str = "q"):
    """(rows, query_len, q_heads, head_dim) of a [R, Hq, D] or [R, Q, Hq, D] tensor."""
    if q.dim() == 3:
        return q.shape[0], 1, q.shape[1], q.shape[2]
    if q.dim() == 4:
        return tuple(q.shape)
    raise ValueError(f"{name} must be [rows, q_heads, head_dim] or "
                     "[rows, query_len, q_heads, head_dim]")


def np_abi_version() -> int:
    return load().np_abi_version()


def np_status_string(status: int) -> str:
    return load().np_status_string(status).decode()


def np_kv_append(k_pool, v_pool, k_new, v_new, slot_mapping, err_word=None, stream=None):
    """Scatter [T, Hk, D] new K/V rows into the pools at ``slot_mapping`` (int64 [T]).

    Leading dimensions are flattened: [R, Q, Hk, D] tokens with [R, Q] slots
    are R*Q tokens.
    """
    nb, bs, hk, d = k_pool.shape
    if k_new.dim() > 3:
        k_new, v_new = k_new.reshape(-1, hk, d), v_new.reshape(-1, hk, d)
        slot_mapping = slot_mapping.reshape(-1)
    if v_pool.shape != k_pool.shape or k_new.shape != v_new.shape or \
            k_new.shape[1:] != (hk, d) or k_new.dtype != k_pool.dtype or \
            v_new.dtype != k_pool.dtype or v_pool.dtype != k_pool.dtype:
        raise ValueError("np_kv_append: shape/dtype mismatch")
    if slot_mapping.dtype != torch.int64 or slot_mapping.shape != (k_new.shape[0],):
        raise ValueError("np_kv_append: slot_mapping must be int64 [num_tokens]")
    cur = _current_device()
    st = load().np_kv_append(
        _dev(k_pool, "k_pool", cur), _dev(v_pool, "v_pool", cur), _dtype_code(k_pool.dtype), nb,
        bs, hk, d, _dev(k_new, "k_new", cur), _dev(v_new, "v_new", cur),
        _dev(slot_mapping, "slot_mapping", cur), k_new.shape[0], _opt(err_word, "err_word", cur),
        _stream(stream))
    _check(st, "np_kv_append")


def np_paged_decode_plan(rows, q_heads, kv_heads, head_dim, block_size, max_blocks_per_row,
                         dtype, num_sms: int = 0) -> int:
    out = _I32(0)
    st = load().np_paged_decode_plan(rows, q_heads, kv_heads, head_dim, block_size,
                                     max_blocks_per_row, _dtype_code(dtype), num_sms,
                                     ctypes.byref(out))
    _check(st, "np_paged_decode_plan")
    return out.value


def np_paged_decode_split_len(block_size, max_blocks_per_row, num_splits) -> int:
    return load().np_paged_decode_split_len(block_size, max_blocks_per_row, num_splits)


def np_paged_decode_workspace_bytes(rows, q_heads, head_dim, num_splits) -> int:
    return load().np_paged_decode_workspace_bytes(rows, q_heads, head_dim, num_splits)


def workspace(rows, q_heads, head_dim, num_splits, device="cuda",
              query_len: int = 1) -> torch.Tensor | None:
    """A workspace of the size the library asks for (None if unsplit).  No
    call needs its contents initialised; zero-filled only to be reproducible."""
    n = np_paged_decode_workspace_bytes(rows * query_len, q_heads, head_dim, num_splits)
    if n == 0:
        return None
    return torch.zeros(n, dtype=torch.uint8, device=device)


def _check_read_args(call, out, q, k_pool, v_pool, block_tables, context_lens):
    rows, qn, q_heads, d = _q_shape(q)
    nb, bs, hk, d2 = k_pool.shape
    if d2 != d or v_pool.shape != k_pool.shape or q.dtype != k_pool.dtype or \
            v_pool.dtype != k_pool.dtype:
        raise ValueError(f"{call}: q/pool shape or dtype mismatch")
    if block_tables.dtype != torch.int32 or block_tables.dim() != 2 or \
            block_tables.shape[0] != rows:
        raise ValueError(f"{call}: block_tables must be int32 [rows, max_blocks]")
    if context_lens.dtype != torch.int32 or context_lens.shape != (rows,):
        raise ValueError(f"{call}: context_lens must be int32 [rows]")
    if out is not None and (out.shape != q.shape or out.dtype != q.dtype):
        raise ValueError(f"{call}: out must match q")
    return rows, qn, q_heads, d, nb, bs, hk


def np_paged_decode(out, q, k_pool, v_pool, block_tables, context_lens, scale,
                    num_splits: int = 1, workspace=None, err_word=None, stream=None):
    """The decode read (see np_paged.h).  Writes ``out`` when num_splits == 1.

    q is [rows, q_heads, head_dim] (one query token per row) or
    [rows, query_len, q_heads, head_dim] (the rows' last query_len positions).
    """
    rows, qn, q_heads, d, nb, bs, hk = _check_read_args(
        "np_paged_decode", out, q, k_pool, v_pool, block_tables, context_lens)
    cur = _current_device()
    ws_ptr = _opt(workspace, "workspace", cur)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load().np_paged_decode(
        _opt(out, "out", cur), _dev(q, "q", cur), _dev(k_pool, "k_pool", cur),
        _dev(v_pool, "v_pool", cur), _dtype_code(q.dtype), nb, bs, hk, d,
        _dev(block_tables, "block_tables", cur), block_tables.shape[1],
        _dev(context_lens, "context_lens", cur), rows, qn, q_heads, float(scale), num_splits,
        ws_ptr, ws_bytes, _opt(err_word, "err_word", cur), _stream(stream))
    _check(st, "np_paged_decode")


def np_paged_append_decode(out, q, k_new, v_new, slot_mapping, k_pool, v_pool, block_tables,
                           context_lens, scale, num_splits: int = 1, workspace=None,
                           err_word=None, stream=None):
    """Append each row's new tokens (at its newest positions) and read, in one launch.

    k_new/v_new: [rows, kv_heads, head_dim] (or [rows, query_len, kv_heads,
    head_dim]); slot_mapping: int64 [rows] (or [rows, query_len]).
    """
    st = load().np_paged_append_decode(*_append_decode_args(
        out, q, k_new, v_new, slot_mapping, k_pool, v_pool, block_tables, context_lens, scale,
        num_splits, workspace, err_word, stream))
    _check(st, "np_paged_append_decode")


def _append_decode_args(out, q, k_new, v_new, slot_mapping, k_pool, v_pool, block_tables,
                        context_lens, scale, num_splits, workspace, err_word, stream) -> list:
    """np_paged_append_decode's C arguments, after the checks."""
    rows, qn, q_heads, d, nb, bs, hk = _check_read_args(
        "np_paged_append_decode", out, q, k_pool, v_pool, block_tables, context_lens)
    want = (rows, hk, d) if q.dim() == 3 else (rows, qn, hk, d)
    if tuple(k_new.shape) != want or v_new.shape != k_new.shape or \
            k_new.dtype != k_pool.dtype or v_new.dtype != k_pool.dtype:
        raise ValueError(f"np_paged_append_decode: k_new/v_new must be {list(want)}")
    want_sm = (rows,) if q.dim() == 3 else (rows, qn)
    if slot_mapping.dtype != torch.int64 or tuple(slot_mapping.shape) != want_sm:
        raise ValueError(f"np_paged_append_decode: slot_mapping must be int64 {list(want_sm)}")
    cur = _current_device()
    ws_ptr = _opt(workspace, "workspace", cur)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return [_opt(out, "out", cur), _dev(q, "q", cur), _dev(k_new, "k_new", cur),
            _dev(v_new, "v_new", cur), _dev(slot_mapping, "slot_mapping", cur),
            _dev(k_pool, "k_pool", cur), _dev(v_pool, "v_pool", cur), _dtype_code(q.dtype), nb,
            bs, hk, d, _dev(block_tables, "block_tables", cur), block_tables.shape[1],
            _dev(context_lens, "context_lens", cur), rows, qn, q_heads, float(scale),
            num_splits, ws_ptr, ws_bytes, _opt(err_word, "err_word", cur), _stream(stream)]


def np_paged_decode_reduce(out, workspace, num_splits: int, stream=None):
    """Merge split partials in ``workspace`` into ``out`` ([rows, q_heads, head_dim]
    or [rows, query_len, q_heads, head_dim])."""
    st = load().np_paged_decode_reduce(*_reduce_args(out, workspace, num_splits, stream))
    _check(st, "np_paged_decode_reduce")


def _reduce_args(out, workspace, num_splits, stream) -> list:
    rows, qn, q_heads, d = _q_shape(out, "out")
    ws_bytes = workspace.numel() * workspace.element_size()
    cur = _current_device()
    return [_dev(out, "out", cur), _dtype_code(out.dtype), _dev(workspace, "workspace", cur),
            ws_bytes, rows * qn, q_heads, d, num_splits, _stream(stream)]


class PreparedStep:
    """One decode step -- the fused append and read (np_paged_append_decode)
    and, for a split read, np_paged_decode_reduce -- with its arguments
    checked and converted to C types once.  ``launch()`` re-issues the same
    calls at a fraction of the binding's per-call host cost, for loops that
    run a step again and again on the same buffers (their contents may
    change between launches; their addresses, shapes, the schedule and the
    stream may not).  Arguments as for np_paged_append_decode; ``out`` is
    always the step's output.
    """

    def __init__(self, out, q, k_new, v_new, slot_mapping, k_pool, v_pool, block_tables,
                 context_lens, scale, num_splits: int = 1, workspace=None, err_word=None,
                 stream=None):
        lib = load()
        calls = [("np_paged_append_decode", _append_decode_args(
            out if num_splits <= 1 else None, q, k_new, v_new, slot_mapping, k_pool, v_pool,
            block_tables, context_lens, scale, num_splits, workspace, err_word, stream))]
        if num_splits > 1:
            calls.append(("np_paged_decode_reduce",
                          _reduce_args(out, workspace, num_splits, stream)))
        self._calls = []
        for name, args in calls:
            typed = getattr(lib, name)
            # a second handle to the same symbol, without argtypes: it passes
            # the already-typed arguments through unconverted
            raw = lib._FuncPtr((name, lib))
            raw.restype = ctypes.c_int
            cargs = tuple(t(a) for t, a in zip(typed.argtypes, args))
            self._calls.append((name, raw, cargs))
        self.launches = (2 if num_splits == 0 else 1) + (1 if num_splits > 1 else 0)
        self._refs = (out, q, k_new, v_new, slot_mapping, k_pool, v_pool, block_tables,
                      context_lens, workspace, err_word)  # keep the buffers alive

    def launch(self) -> int:
        """Issue the step; returns the number of library kernels launched."""
        for name, fn, cargs in self._calls:
            st = fn(*cargs)
            if st != NP_OK:
                raise NPError(st, name)
        return self.launches


def np_paged_decode_noalloc(out, q, k_pool, v_pool, block_tables, context_lens, scale,
                            num_splits: int = 1, err_word=None, stream=None):
    """The read plus the split merge with no workspace argument: for callers
    that cannot allocate device memory, the split partials go to a fixed
    NP_NOALLOC_SCRATCH_BYTES array inside the library (see np_paged.h)."""
    if out is None:
        raise ValueError("np_paged_decode_noalloc: out is required")
    rows, qn, q_heads, d, nb, bs, hk = _check_read_args(
        "np_paged_decode_noalloc", out, q, k_pool, v_pool, block_tables, context_lens)
    cur = _current_device()
    st = load().np_paged_decode_noalloc(
        _dev(out, "out", cur), _dev(q, "q", cur), _dev(k_pool, "k_pool", cur),
        _dev(v_pool, "v_pool", cur), _dtype_code(q.dtype), nb, bs, hk, d,
        _dev(block_tables, "block_tables", cur), block_tables.shape[1],
        _dev(context_lens, "context_lens", cur), rows, qn, q_heads, float(scale), num_splits,
        _opt(err_word, "err_word", cur), _stream(stream))
    _check(st, "np_paged_decode_noalloc")


def np_selftest_bounded_wait(err_word, limit_cycles: int, stream=None):
    """Device check of the read's wait-timeout path: a wait that nothing
    completes gives up after ``limit_cycles`` and ORs NP_FLAG_TIMEOUT into
    ``err_word`` (a device int32 tensor); see np_paged.h."""
    st = load().np_selftest_bounded_wait(_dev(err_word, "err_word", _current_device()),
                                         int(limit_cycles), _stream(stream))
    _check(st, "np_selftest_bounded_wait")


def decode_step(out, q, k_pool, v_pool, block_tables, context_lens, scale, *, k_new=None,
                v_new=None, slot_mapping=None, num_splits: int = 1, workspace=None,
                err_word=None, stream=None, fused: bool = True) -> int:
    """One decode step: append (if new K/V given), read, reduce (if split).

    With ``fused`` (the default) and one new token per row, the append runs
    inside the read's launch (np_paged_append_decode); otherwise
    np_kv_append runs first.  Returns the number of library kernels launched.
    """
    launches = 0
    o = out if num_splits <= 1 else None  # 0: the balanced read writes out itself
    if k_new is not None and fused and k_new.shape[0] == q.shape[0] and \
            k_new.dim() == q.dim():
        np_paged_append_decode(o, q, k_new, v_new, slot_mapping, k_pool, v_pool, block_tables,
                               context_lens, scale, num_splits, workspace, err_word, stream)
        launches += (2 if num_splits == 0 else 1) if q.shape[0] > 0 else 0  # + the merge
    else:
        if k_new is not None:
            np_kv_append(k_pool, v_pool, k_new, v_new, slot_mapping, err_word, stream)
            launches += 1 if k_new.shape[0] > 0 else 0
        np_paged_decode(o, q, k_pool, v_pool, block_tables, context_lens, scale, num_splits,
                        workspace, err_word, stream)
        launches += (2 if num_splits == 0 else 1) if q.shape[0] > 0 else 0
    if num_splits > 1:
        np_paged_decode_reduce(out, workspace, num_splits, stream)
        launches += 1 if q.shape[0] > 0 else 0
    return launches


def default_scale(head_dim: int) -> float:
    return 1.0 / math.sqrt(head_dim)
