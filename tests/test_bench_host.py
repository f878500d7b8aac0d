"""Host arithmetic of bench.py: the algorithmic bytes and FLOPs behind every roofline
figure, the grouping of timed steps into CUDA graph replays, and the rule that a
committed ncu traffic figure is reported only for the kernel source it was taken on."""

import math

import numpy as np

import bench


def test_decode_bytes_matches_its_definition():
    # K and V rows attended, Q and O rows, one int32 table entry per block touched,
    # one int32 length per sequence (bf16/fp16 elements).
    lens, Hq, Hkv, D, bs = [37, 5, 16, 0], 4, 2, 64, 16
    want = 0
    for L in lens:
        want += L * Hkv * D * 2 * 2          # K and V
        want += 2 * Hq * D * 2               # q and out rows of the sequence
        want += 4 * math.ceil(L / bs) + 4    # table entries, length
    assert bench.decode_bytes(lens, Hq, Hkv, D, bs) == want
    assert bench.decode_bytes([37, 5], 4, 2, 64, 16) == 21504 + 2048 + 16 + 8


def test_write_bytes_matches_its_definition():
    B, Hkv, D = 64, 8, 128
    rows = 2 * B * Hkv * D * 2                # new K and V rows, bf16
    assert bench.write_bytes(B, Hkv, D) == 2 * rows + 3 * 4 * B


def test_prefill_flops_counts_visible_pairs_by_brute_force():
    rng = np.random.default_rng(5)
    for _ in range(20):
        S = int(rng.integers(1, 5))
        lens = [int(x) for x in rng.integers(0, 40, S)]
        ctx = [int(x) for x in rng.integers(0, 30, S)]
        pairs = 0
        for n, c in zip(lens, ctx):
            for i in range(n):                # query i sees cached keys and keys 0..i
                for k in range(c + n):
                    pairs += k <= c + i
        assert bench.prefill_flops(lens, ctx, 32, 128) == 4 * 32 * 128 * pairs


def test_steps_per_graph_divides_the_timed_steps():
    for steps, want in [(200, 10), (3, 3), (7, 7), (13, 1), (24, 8), (1, 1), (30, 10)]:
        got = bench.steps_per_graph(steps)
        assert got == want and steps % got == 0


def test_recorded_traffic_needs_the_matching_source_digest(tmp_path, monkeypatch):
    import json
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({
        "k/w": {"kernel_source_digest": "0123456789abcdef", "dram_bytes_per_launch": 598906624}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("k/w", "0123456789abcdef") == 598906624.0
    assert bench.recorded_traffic("k/w", "fedcba9876543210") is None
    assert bench.recorded_traffic("other", "0123456789abcdef") is None


def test_all_core_oracle_baseline_runs_on_spawned_workers():
    """The CPU baseline's pool: spawned workers, memory-mapped inputs, whole passes."""
    from synth import make_config
    case = make_config("tiny_decode", seed=0)
    gbs, n, workers, t = bench.cpu_oracle_rate_all_cores(case, budget_s=0.2)
    assert gbs > 0 and workers >= 1 and n % case.q.shape[0] == 0 and t > 0


def test_int8_decode_bytes_counts_codes_scales_and_rows():
    lens, Hq, Hkv, D, bs = [37, 5, 0], 4, 2, 128, 16
    want = sum(L * Hkv * (D + 4) * 2 for L in lens) + 3 * 2 * Hq * D * 2 + \
        4 * sum(math.ceil(L / bs) for L in lens) + 4 * 3
    assert bench.int8_decode_bytes(lens, Hq, Hkv, D, bs) == want


def test_int8_write_bytes_counts_rows_codes_scales_slots():
    B, Hkv, D = 3, 2, 128
    # 16-bit rows read (K and V), int8 codes + one fp32 scale per row written, slots written
    want = 2 * B * Hkv * D * 2 + 2 * B * Hkv * D + 2 * B * Hkv * 4 + 4 * B
    assert bench.int8_write_bytes(B, Hkv, D) == want


def test_launch_percentiles_order_and_values():
    p10, p50, p90 = bench.launch_percentiles([0.1, 0.2, 0.3, 0.4, 0.5])
    assert p10 <= p50 <= p90 and abs(p50 - 0.3) < 1e-12
