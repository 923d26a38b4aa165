"""bench.py's host-side accounting on the CPU: the clock summary keeps only
the samples taken inside the timed window and reports every throttle reason
seen there; the L2 handling picks rotation or a flush by pool size."""
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_clock_summary_uses_the_timed_window():
    c = bench.ClockSampler(torch.device("cpu"))
    c.samples = [(0.0, 900.0, 2070.0, ["sw_thermal_slowdown"]),  # before the window
                 (1.0, 2070.0, 2070.0, []), (1.1, 2050.0, 2070.0, ["sw_power_cap"]),
                 (1.2, 2060.0, 2070.0, []),
                 (5.0, 800.0, 2070.0, ["hw_slowdown"])]  # after it
    c.mark(0.99, 1.25)
    s = c.summary()
    assert s["samples"] == 3 and s["in_timed_region"]
    assert s["sm_mhz"] == 2060.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]


def test_clock_summary_without_samples_in_the_window():
    c = bench.ClockSampler(torch.device("cpu"))
    c.samples = [(0.0, 2070.0, 2070.0, [])]
    c.mark(3.0, 3.001)
    s = c.summary()
    assert s["samples"] == 1 and not s["in_timed_region"]
    c.samples = []
    assert bench.ClockSampler.summary(c)["reasons"] == ["unsampled"]


def test_nvidia_smi_line_parsing():
    c = bench.ClockSampler(torch.device("cpu"))

    class P:
        stdout = ["0, 2070, 2070, 800.5, 0x4, Not Active, Not Active, Not Active, Active\n",
                  "garbage\n",
                  "0, 1500, 2070, 900.0, 0x8, Active, Not Active, Not Active, Not Active\n"]
    c.proc = P()
    c._read()
    assert [x[1:] for x in c.samples] == [(2070.0, 2070.0, ["sw_power_cap"]),
                                          (1500.0, 2070.0, ["hw_slowdown"])]


def test_nvml_reason_bits():
    # NVML's clock-event reason mask: 0x4 software power cap, 0x8 hardware
    # slowdown, 0x20 software thermal, 0x40 hardware thermal
    names = bench._Nvml.REASONS
    assert names[0x4] == "sw_power_cap" and names[0x8] == "hw_slowdown"
    assert names[0x20] == "sw_thermal_slowdown" and names[0x40] == "hw_thermal_slowdown"


def test_l2_plan():
    L2 = bench.L2_BYTES
    assert bench.l2_plan(4 * L2, 5 * L2) == 1           # K/V read per step beyond 4x L2
    n = bench.l2_plan(85_000_000, 85_000_000)          # the fp32 Llama-style step
    assert n * 85_000_000 > 3 * L2 and (n - 1) * 85_000_000 <= 3 * L2 + 85_000_000
    assert bench.l2_plan(20_000, 40_000) == 0           # tiny pool: flush instead
    assert bench.l2_plan(L2 // 16, L2 // 16) == 0       # 49 copies: too many, flush
    assert bench.l2_plan(L2 // 8, L2 // 8) == 25


def test_algorithmic_bytes_by_hand():
    """The roofline numerator on the tiny fp32 case, counted by hand: rows 2,
    q heads 4, kv heads 2, head_dim 16, block 8, contexts 16 and 64, fp32.
    K/V history (16 + 64) tokens x 2 (K, V) x 2 heads x 16 dims x 4 B = 20480;
    q and out 2 x 2 rows x 4 heads x 16 x 4 = 1024; table entries
    (2 + 8) x 4 + context lengths 2 x 4 = 48; the append: new K and V read
    and written, 2 x 2 x 2 rows x 2 heads x 16 x 4 = 1024, plus 2 slots x 8."""
    import workloads as wl
    w = wl.WORKLOADS["tiny-fp32"]
    inp = wl.make_inputs(w, device="cpu")
    assert inp.md.context_lens.tolist() == [16, 64]
    got = bench.algorithmic_bytes(w, inp.md)
    assert got == {"kv": 20480, "decode": 20480 + 1024 + 48 + 1040, "append": 1040}
