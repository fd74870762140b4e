"""Host-side helpers of the benchmark and the end-to-end step (no GPU): the
clock-sample summary that decides whether a run saw throttling, and the
layer groups whose inputs the host path copies together."""
import bench


def test_clock_summary_median_max_and_reasons():
    lines = [
        "0, 2070, 2070, 900.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n",
        "0, 1980, 2070, 1300.2, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n",
        "0, 2055, 2070, 1250.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n",
    ]
    got = bench.summarise_clocks(lines)
    assert got == {"sm_mhz": 2055.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}


def test_clock_summary_reports_every_slowdown_kind():
    lines = [
        "0, 1500, 2070, 1400, 0x8, Active, Not Active, Not Active, Not Active",
        "0, 1400, 2070, 1400, 0x48, Not Active, Active, Active, Not Active",
    ]
    got = bench.summarise_clocks(lines)
    assert got["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]
    assert got["sm_mhz"] == 1450.0


def test_clock_summary_skips_unparsable_values_and_short_lines():
    lines = ["", "garbage", "0, [N/A], 2070, 10, 0x0, Not Active, Not Active, Not Active, Not Active",
             "0, 2070, [N/A], 10, 0x0, Not Active, Not Active, Not Active, Not Active"]
    got = bench.summarise_clocks(lines)
    assert got == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 2}
    assert bench.summarise_clocks([]) is None
    assert bench.summarise_clocks(["a, b"]) is None


def test_host_copy_groups_cover_every_layer_once_in_three_waits_at_most():
    from paged_kv_decode_rope_gb300.step import host_copy_groups
    assert host_copy_groups(1) == [(0, 1)]
    assert host_copy_groups(2) == [(0, 1), (1, 2)]
    assert host_copy_groups(4) == [(0, 1), (1, 4)]
    assert host_copy_groups(16) == [(0, 1), (1, 4), (4, 16)]
    assert host_copy_groups(24) == [(0, 1), (1, 4), (4, 24)]
    for nl in range(1, 40):
        g = host_copy_groups(nl)
        assert g[0] == (0, 1) and len(g) <= 3
        assert [lo for lo, _ in g[1:]] == [hi for _, hi in g[:-1]] and g[-1][1] == nl


def test_prefill_roofline_counts_algorithmic_flops_against_the_tensor_peak():
    # 4 prompts x 2048 tokens, 32 query heads, 16 layers, 4.47 ms per pass
    pairs = 4 * 2048 * 2049 / 2 * 32 * 16
    r = bench.prefill_roofline(pairs, 4.47, 1710.2, "measured")
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["traffic"] is None
    assert abs(r["achieved"] - pairs * 256 / 4.47e-3 / 1e12) < 0.01
    assert abs(r["achieved"] - 246.3) < 0.5          # the figure the docs quote for this case
    assert abs(r["frac"] - r["achieved"] / 1710.2) < 1e-4
    peak, src = bench._tensor_peak()
    assert peak > 0 and src in ("measured", "fallback")


def test_prefill_traffic_only_while_the_source_is_the_measured_one(monkeypatch):
    # (4, 2048) has a stored capture; it is reported only for the source it was taken on
    want = bench.PREFILL_TRAFFIC[(4, 2048)]
    monkeypatch.setattr(bench, "_source_hash", lambda name: want[0])
    assert bench._prefill_traffic(4, 2048) == want[1]
    assert bench._prefill_traffic(1, 8192) is None
    monkeypatch.setattr(bench, "_source_hash", lambda name: "0" * 16)
    assert bench._prefill_traffic(4, 2048) is None
    r = bench.prefill_roofline(1e9, 3.0, 1710.2, "measured", traffic=want[1])
    assert r["traffic"] == want[1] and r["bound"] == "tensor"
