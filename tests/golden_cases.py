"""Loader for the hand-worked fixtures in tests/golden/."""
import json
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _num(x):
    if isinstance(x, list):
        return [_num(v) for v in x]
    if isinstance(x, str):
        return float(x)  # "nan", "-inf", "inf"
    return x


def load(name: str) -> dict:
    with open(os.path.join(GOLDEN, name)) as f:
        raw = json.load(f)
    out = {}
    for k, v in raw.items():
        if k in ("what", "citation", "derivation", "dtype"):
            out[k] = v
        elif k in ("block_tables", "context_lens"):
            out[k] = np.asarray(v, dtype=np.int32)
        elif k == "slot_mapping":
            out[k] = np.asarray(v, dtype=np.int64)
        elif isinstance(v, list):
            arr = np.asarray(_num(v), dtype=np.float64)
            out[k] = arr
        else:
            out[k] = v
    for k in ("q", "k_pool", "v_pool", "k_new", "v_new"):
        if k in out:
            out[k] = out[k].astype(np.float32)
    return out


def names():
    return sorted(f for f in os.listdir(GOLDEN) if f.endswith(".json"))
