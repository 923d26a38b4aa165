"""Each pin earns its place: an oracle with one planted mistake must fail one.

Every mutant is a copy of the oracle's C source with a single textual change
(a dropped term, a wrong sign, a wrong index, an off-by-one), compiled into a
temporary directory on the CPU.  The real oracle passes every check in
``oracle_pins``; each mutant must fail at least one of them.
"""
import os
import shutil
import subprocess
import sys

import pytest

import oracle
import oracle_pins
from oracle import build as obuild

MUTANTS = {
    # the block-table walk: logical block index and offset swapped
    "walk_block_index": ("decode_body.h", "t / block_size]", "t % block_size]"),
    "walk_offset": ("decode_body.h", "block * block_size + t % block_size",
                    "block * block_size + t / block_size"),
    # the slot's element offset ignores the kv head
    "kv_head_ignored": ("decode_body.h", "(slot * kv_heads + kh) * head_dim + d",
                        "(slot * kv_heads) * head_dim + d"),
    # GQA: query heads paired with the wrong kv head
    "gqa_wrong_group": ("decode_body.h",
                        "for (int32_t h = kh * group; h < (kh + 1) * group; ++h)",
                        "for (int32_t h = kh; h < q_heads; h += kv_heads)"),
    # the scale factor dropped
    "scale_dropped": ("decode_body.h", "sco[t] = sc * dot;", "sco[t] = dot;"),
    # exponent sign flipped
    "exp_sign": ("decode_body.h", "NPO_EXP(sco[t] - m)", "NPO_EXP(m - sco[t])"),
    # softmax not normalised
    "no_normalise": ("decode_body.h", "o[d] /= z;", "o[d] /= 1;"),
    # the last history token dropped
    "range_off_by_one": ("decode_body.h", "tb + split_len < e ? tb + split_len : e",
                         "tb + split_len < e - 1 ? tb + split_len : e - 1"),
    # one slot past the history read
    "range_one_past": ("decode_body.h", "tb + split_len < e ? tb + split_len : e",
                       "tb + split_len < e + 1 ? tb + split_len : e + 1"),
    # causal limit of a query token off by one
    "causal_limit": ("decode_body.h", "int64_t e = c - query_len + qi + 1;",
                     "int64_t e = c - query_len + qi;"),
    # query tokens read in the wrong order
    "query_order": ("decode_body.h", "int64_t rq = (int64_t)r * query_len + qi;",
                    "int64_t rq = (int64_t)r * query_len + (query_len - 1 - qi);"),
    # query element taken from the wrong head
    "q_wrong_head": ("decode_body.h", "(rq * q_heads + h) * head_dim + d);",
                     "(rq * q_heads + kh) * head_dim + d);"),
    # V gathered from the K pool
    "v_from_k": ("decode_body.h", "npo_load(v_pool, dtype, idx)", "npo_load(k_pool, dtype, idx)"),
    # lse missing the max
    "lse_no_max": ("decode_body.h", "lse[rhs] = m + NPO_LOG(z);", "lse[rhs] = NPO_LOG(z);"),
    # reduce weights with the wrong sign
    "reduce_sign": ("np_oracle.c", "double w = exp(lse[s] - big);", "double w = exp(big - lse[s]);"),
    # reduce not normalised
    "reduce_no_norm": ("np_oracle.c", "o[d] /= wsum;", "o[d] /= 1.0;"),
    # append writes the token's own index instead of its slot
    "append_dst": ("np_oracle.c", "(char*)k_pool + s * row_bytes", "(char*)k_pool + i * row_bytes"),
    # append ignores the negative-slot skip
    "append_negative": ("np_oracle.c", "if (s < 0) continue;", "if (s < -1) continue;"),
    # bf16 widening shifted wrong
    "bf16_shift": ("np_oracle.c", "(uint32_t)h << 16", "(uint32_t)h << 15"),
}


def _build_mutant(tmp_path, name, target, old, new):
    d = tmp_path / name
    d.mkdir()
    for f in ("np_oracle.c", "decode_body.h"):
        shutil.copy(os.path.join(obuild.HERE, f), d / f)
    path = d / target
    src = path.read_text()
    assert src.count(old) == 1, f"mutation site for {name} not unique/found"
    path.write_text(src.replace(old, new))
    so = str(d / "libmutant.so")
    obuild.compile_oracle([str(d / "np_oracle.c")], so)
    return so


# Runs every pin against one library in a child process (a mutant may write
# out of bounds and kill its process; that counts as caught).  Prints the
# names of the checks that failed.
_CHILD = """
import sys
sys.path[:0] = [{root!r}, {tests!r}]
import oracle, oracle_pins
lib = oracle.load({so!r})
for check in oracle_pins.ALL_CHECKS:
    try:
        check(lib)
    except Exception as e:
        print("FAILED", check.__name__, type(e).__name__, flush=True)
print("DONE", flush=True)
"""


def _run_checks(so):
    here = os.path.dirname(os.path.abspath(__file__))
    code = _CHILD.format(root=os.path.dirname(here), tests=here, so=so)
    p = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                       timeout=600)
    failed = [ln.split()[1] for ln in p.stdout.splitlines() if ln.startswith("FAILED")]
    crashed = p.returncode != 0 or "DONE" not in p.stdout
    return failed, crashed


def test_real_oracle_passes_in_child():
    failed, crashed = _run_checks(obuild.build())
    assert not failed and not crashed


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    target, old, new = MUTANTS[name]
    so = _build_mutant(tmp_path, name, target, old, new)
    failed, crashed = _run_checks(so)
    assert failed or crashed, f"no pin caught mutant {name}"
