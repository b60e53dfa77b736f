"""The roofline accounting of bench.py (no GPU): the algorithmic bytes and FLOPs per launch
that every reported fraction divides by, against sums written out tensor by tensor from the
workloads' definitions (one layer: H = 64 heads, d = 128, 64-token chunks).
"""
import bench

T, H, D, C = 4096, 64, 128, 64
BF16, F32 = 2, 4


def test_prefill_bytes_are_the_tensors_it_must_move():
    q_k_v = 3 * T * H * D * BF16
    g = T * H * D * F32
    beta = T * H * F32
    out = T * H * D * BF16
    final_state = H * D * D * F32
    assert bench._prefill_bytes(T, H, D) == q_k_v + g + beta + out + final_state == 407_896_064
    # 98,560 bytes per token at 64 heads, plus one layer's 4 MiB state
    assert bench._prefill_bytes(T, H, D, with_state_out=False) == T * 98_560


def test_prefill_flops_count_each_contraction_once_per_chunk_and_head():
    mac = (2 * C * C * D        # A = K~ K^T and P = Q~ K^T
           + C ** 3 / 3         # T = (I + A)^-1, unit lower triangular
           + 2 * C * D * D      # X = [K Gamma; Q Gamma] S
           + C * C * D          # u = T Y
           + C * C * D          # O += P' u
           + D * C * D)         # S += Kbar^T u
    per_launch = 2 * mac * (T // C) * H
    assert abs(bench._prefill_flops(T, H, D) - per_launch) < 1.0
    assert round(per_launch / 1e9, 1) == 43.7


def test_prologue_bytes():
    raw_x, qkv = T * 3 * H * D * BF16, T * 3 * H * D * BF16
    beta_logit, beta = T * H * F32, T * H * F32
    assert bench._prologue_bytes(T, H, D) == raw_x + qkv + beta_logit + beta == 404_750_336


def test_decode_bytes_stream_the_state_once_each_way():
    n, ch = 256, 3 * H * D
    state = 2 * n * H * D * D * F32                  # read + write, in place
    conv_tail = 2 * n * 3 * ch * BF16                # read + write
    inputs_ = n * ch * BF16 + n * H * D * F32 + n * H * F32
    weights = ch * 4 * BF16
    out = n * H * D * BF16
    assert bench._decode_bytes(n, H, D) == state + conv_tail + inputs_ + weights + out
    assert state == 2 * 2**30                         # 1 GiB pool, read and written


def test_clock_summary_keeps_the_timed_window_and_its_throttle_reasons(tmp_path):
    import datetime
    t = datetime.datetime(2026, 1, 2, 3, 4, 5)
    rows = [  # before, inside (3), after the window
        (0.0, 1500, "Not Active", "Not Active"),
        (1.0, 2070, "Not Active", "Not Active"),
        (1.1, 2000, "Active", "Not Active"),
        (1.2, 1900, "Not Active", "Active"),
        (3.0, 900, "Active", "Active"),
    ]
    path = tmp_path / "clocks.csv"
    with open(path, "w") as f:
        for dt, mhz, hw, cap in rows:
            ts = (t + datetime.timedelta(seconds=dt)).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
            f.write(f"{ts}, 0, {mhz}, 2070, 900.0, 0x0, {hw}, Not Active, Not Active, {cap}\n")
    cs = bench.ClockSampler(0)
    cs.path = str(path)
    cs.t0 = t + datetime.timedelta(seconds=0.5)
    cs.t1 = t + datetime.timedelta(seconds=2.0)
    s = cs.summary()
    assert s["samples"] == 3 and s["sm_mhz"] == 2000 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["hw_slowdown", "sw_power_cap"]
    cs.path = str(tmp_path / "missing.csv")
    assert cs.summary()["reasons"] == ["unsampled"]


def test_reference_arm_prints_one_contract_line(capsys):
    """bench.py --impl reference: the oracle timed on the host cores, one JSON line with the
    keys the driver reads (rank 0 only; no GPU involved)."""
    import json
    import types
    bench.run_reference(types.SimpleNamespace(gpus=1, steps=1, warmup=0))
    lines = [x for x in capsys.readouterr().out.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["value"] > 0 and line["unit"] == "tokens/s" and line["higher_is_better"]
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": "tokens/s",
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_batch_prefill_bytes_for_the_gated_and_varlen_workloads():
    """Per token q, k, v, out (bf16), g, beta (fp32) and the gate logits (bf16) when the output
    norm and gate run: 114,944 bytes per token at 64 heads; per sequence the
    initial and final state."""
    lens = [32768] * 4
    per_tok = 3 * H * D * BF16 + H * D * F32 + H * F32 + H * D * BF16 + H * D * BF16
    assert per_tok == 114_944
    states = 4 * 2 * H * D * D * F32
    assert bench._prefill_bytes_batch(lens, H, D, gate=True, state_in=True) == \
        sum(lens) * per_tok + states
    # bf16 state storage halves the state bytes; without an initial state only the final
    assert bench._prefill_bytes_batch([100, 28], H, D, gate=False, state_in=False,
                                      state_bytes=2) == 128 * 98_560 + 2 * H * D * D * 2


def test_triangle_flop_count_per_head_token():
    # 2 (3 d^2 + 2.5 C d) at d = 128, C = 64
    assert bench.TRIANGLE_FLOPS_PER_HEAD_TOKEN == 139_264
