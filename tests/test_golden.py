"""The oracle against the hand-worked fixtures (CPU only)."""
import numpy as np

import golden_cases
import oracle


def test_read_three_tokens_gqa(oracle_lib):
    g = golden_cases.load("read_three_tokens_gqa.json")
    out, lse = oracle.paged_decode(g["q"], g["k_pool"], g["v_pool"], g["block_tables"],
                                   g["context_lens"], g["scale"], lib=oracle_lib)
    np.testing.assert_allclose(out, g["expected_out"], rtol=0, atol=g["atol"])
    np.testing.assert_allclose(lse, g["expected_lse"], rtol=0, atol=g["atol"])


def test_append_then_read(oracle_lib):
    g = golden_cases.load("append_then_read.json")
    kp, vp = g["k_pool"].copy(), g["v_pool"].copy()
    assert oracle.kv_append(kp, vp, g["k_new"], g["v_new"], g["slot_mapping"],
                            lib=oracle_lib) == oracle.OK
    np.testing.assert_array_equal(kp, g["expected_k_pool"].astype(np.float32))
    np.testing.assert_array_equal(vp, g["expected_v_pool"].astype(np.float32))
    out, lse = oracle.paged_decode(g["q"], kp, vp, g["block_tables"], g["context_lens"],
                                   g["scale"], lib=oracle_lib)
    np.testing.assert_allclose(out, g["expected_out"], rtol=0, atol=g["atol"])
    np.testing.assert_allclose(lse, g["expected_lse"], rtol=0, atol=g["atol"])


def test_split_combine(oracle_lib):
    g = golden_cases.load("split_combine.json")
    out = oracle.reduce(g["o_part"], g["lse_part"], lib=oracle_lib)
    np.testing.assert_allclose(out, g["expected_out"], rtol=0, atol=g["atol"])
