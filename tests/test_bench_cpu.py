"""bench.py's measurement arithmetic on the CPU: the algorithmic byte model behind the roofline
figures, the job rate and the clock summary that decides whether a run is kept."""
import bench


def test_kv_bytes_follow_the_closed_form():
    # per token and layer: K and V of every kv head, head_dim bf16 values each
    assert bench.kv_bytes([1], 8, 128) == 2 * 8 * 128 * 2
    # the pages' Qwen2.5-7B figure (28 layers, 4 kv heads, head_dim 128): 7.5 GB at 128K tokens
    per_token = 28 * bench.kv_bytes([1], 4, 128)
    assert per_token == 57344
    assert round(per_token * 131072 / 1e9, 1) == 7.5
    # the headline step: batch 8, every sequence at 32768 + 1 keys once its token is appended
    assert bench.kv_bytes([32769] * 8, 8) == 8 * 32769 * 4096


def test_decode_step_bytes_add_each_stream_once():
    S, Hkv, Hq, d = [100, 200], 8, 64, 128
    bare = bench.step_kernel_bytes(S, Hkv, Hq, d, probs=False, cum=False)
    assert bare == 300 * Hkv * d * 4 + 2 * Hq * d * 2 * 2            # K and V once, q in and O out
    assert bench.step_kernel_bytes(S, Hkv, Hq, d, probs=True, cum=False) - bare == 300 * Hq * 4
    assert bench.step_kernel_bytes(S, Hkv, Hq, d, probs=False, cum=True) - bare == 300 * Hkv * 8


def test_headline_algorithmic_bytes_per_launch():
    # 3072 timed steps after 128 warm-up steps cover the 128-step window 24 times: the mean
    # live length is 32768 + 64.5, and a launch moves 1.160169 GB by the model
    S0, T, warm, steps = 32768, 128, 128, 3072
    S_steps = [S0 + (i % T) + 1 for i in range(warm, warm + steps)]
    mean = sum(bench.step_kernel_bytes([S] * 8, 8, 64) for S in S_steps) / len(S_steps)
    assert abs(mean - 1.160169e9) < 1e3


def test_job_rate_and_a_lone_rank():
    assert bench.job_rate(1, 3072, 1000.0) == 3072.0
    assert bench.job_rate(4, 10, 500.0) == 80.0       # every rank's units over the slowest time
    assert bench.slowest_rank(3.5, 1) == 3.5


def _row(sm, mx, pw, *flags):
    return ["ts", str(sm), str(mx), str(pw), "0x0", *flags]


def test_clock_summary_reads_the_throttle_reasons():
    c = bench.ClockSampler("GPU-x")
    off = "Not Active"
    c.rows = [(10.00, _row(2070, 2070, 600, off, off, off, "Active")),
              (10.05, _row(1900, 2070, 650, "Active", off, off, off)),
              (20.00, _row(1000, 2070, 100, off, off, off, off))]
    s = c.summary(10.0, 10.05)
    assert s["samples"] == 2 and s["sm_mhz"] == 1985.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert s["power_w_max"] == 650.0
    # no sample inside a short timed region: the nearest one stands for it
    near = c.summary(19.0, 19.5)
    assert near["samples"] == 1 and near["sm_mhz"] == 1000.0 and near["reasons"] == []
    assert bench.ClockSampler("GPU-y").summary(0.0, 1.0)["reasons"] == ["unsampled"]
