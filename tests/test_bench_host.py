"""Host-side pins of the benchmark's roofline arithmetic (CPU): the algorithmic bytes and
flops of a call, worked out by hand for small batches, and the JSON line of the oracle
(reference) arm on the smallest workload."""
import json
import os
import subprocess
import sys

import pytest

import bench
from mla_speculative_verify_gb300 import inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_algorithmic_bytes_and_flops_by_hand():
    # two requests, H = 12: ctx 1000 (q = 4) and ctx 65 (q = 1), bf16 cache
    prob = inputs.make_problem(12, [1000, 65], [4, 1], inputs.KV_BF16, seed=1)
    kv = (1000 + 65) * 576 * 2
    q = 5 * 12 * 576 * 2
    out = 5 * 12 * 512 * 2
    lse = 5 * 12 * 4
    pages = (16 + 2) * 4          # ceil(1000 / 64) + ceil(65 / 64) page ids
    assert bench.algorithmic_bytes(prob) == kv + q + out + lse + pages
    # visible keys: tokens of the first request see 997, 998, 999, 1000; the second 65
    assert bench.algorithmic_flops(prob) == (997 + 998 + 999 + 1000 + 65) * 12 * 2176.0


def test_algorithmic_bytes_fp8_cache_counts_one_byte_per_element():
    bf = inputs.make_problem(12, [640], [2], inputs.KV_BF16, seed=2)
    f8 = inputs.make_problem(12, [640], [2], inputs.KV_FP8, seed=2)
    assert bench.algorithmic_bytes(bf) - bench.algorithmic_bytes(f8) == 640 * 576


@pytest.mark.timeout(600)
def test_reference_arm_json_line():
    """`bench.py --impl reference` on the small contiguous workload prints one JSON line
    with the contract's keys; the oracle is its timed arm."""
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "contig4096", "--steps", "1",
                        "--warmup", "0"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "config",
              "cpu_baseline", "e2e"):
        assert k in line, k
    assert line["impl"] == "reference" and line["higher_is_better"] is False
    assert line["warmup"] >= 3 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0


def test_clock_summary_reads_reasons_and_flags_low_clocks(tmp_path):
    """The nvidia-smi CSV of the timed region: median SM clock, the throttle reasons seen,
    and the flag for a median below 0.7 of the maximum clock."""
    c = bench.ClockSampler(0)
    c.proc = object()  # as if sampling had run
    c.path = str(tmp_path / "clocks.csv")
    rows = ["2026/12/03 12:00:01.000, 0, 1200, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Active",
            "2026/12/03 12:00:01.020, 0, 1300, 2070, 950.0, 0x0, Not Active, Active, Not Active, Not Active",
            "2026/12/03 12:00:01.040, 0, 1250, 2070, 940.0, 0x0, Not Active, Not Active, Not Active, Not Active"]
    (tmp_path / "clocks.csv").write_text("timestamp, index, clocks.sm\n" + "\n".join(rows) + "\n")
    s = c.summary()
    assert s["sm_mhz"] == 1250 and s["sm_max_mhz"] == 2070 and s["samples"] == 3
    assert s["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    assert s["below_70pct_of_max"] is True


def test_oracle_sample_scale_by_hand():
    # one request, H = 12, ctx 1000, q = 4: the call's rows see 997..1000 keys
    prob = inputs.make_problem(12, [1000], [4], inputs.KV_BF16, seed=3)
    whole = (997 + 998 + 999 + 1000) * 12
    # first token against the whole context: it sees 997 keys
    sub, scale = bench.oracle_sample(prob, 1)
    assert list(sub.seq_lens) == [997] and list(sub.q_lens) == [1]
    assert scale == pytest.approx(whole / (997 * 12))
    # first two tokens against the first 300 keys: they see 299 and 300
    sub, scale = bench.oracle_sample(prob, 2, 300)
    assert list(sub.seq_lens) == [300] and list(sub.q_lens) == [2]
    assert scale == pytest.approx(whole / ((299 + 300) * 12))
    # a cap above the context is the whole context; a cap below the token count keeps them
    assert list(bench.oracle_sample(prob, 1, 10**9)[0].seq_lens) == [997]
    assert list(bench.oracle_sample(prob, 3, 1)[0].seq_lens) == [3]
    # the sample's rows are the call's first rows: same query values, same page table row
    assert (sub.q.float().numpy() == prob.q[:2].float().numpy()).all()
    assert (sub.page_table[0] == prob.page_table[0]).all()


def test_clock_samples_are_selected_by_time_window():
    def line(sec, mhz, power_cap="Not Active"):
        return (f"2026/12/03 12:00:{sec:06.3f}, 0, {mhz}, 2070, 900.5, 0x0000000000000000, Not Active, "
                f"Not Active, Not Active, {power_cap}")

    text = "\n".join([line(1.0, 1000), line(2.0, 2070), line(2.02, 2070), line(2.04, 2070, "Active"),
                      line(2.06, 2070), line(3.0, 800), "garbled, line"])
    rows = bench.ClockSampler.parse(text)
    assert len(rows) == 6
    t = [r[0] for r in rows]
    # the timed region holds four samples: the idle ones before and after are left out
    s = bench.ClockSampler.summarize(rows, t[0], t[1] - 0.001, t[4] + 0.001)
    assert s["window"] == "timed region" and s["samples"] == 4
    assert s["sm_mhz"] == 2070 and s["reasons"] == ["sw_power_cap"]
    # a timed region with fewer than three samples also takes the warm-up's
    s = bench.ClockSampler.summarize(rows, t[1] - 0.001, t[3] - 0.001, t[4] + 0.001)
    assert s["window"] == "warm-up + timed region" and s["samples"] == 4
    # no window: every sample, and the low median is flagged
    s = bench.ClockSampler.summarize(rows, None, None, None)
    assert s["window"] == "whole run" and s["samples"] == 6
    s = bench.ClockSampler.summarize([rows[0], rows[5]], None, None, None)
    assert s["below_70pct_of_max"] is True
