"""Host logic of bench.py that needs no GPU: the visible-pair count behind the banded
workloads' TFLOP/s, the ncu launch-list summary, and the source-hash guard on the
committed DRAM-traffic figures."""
import os

import numpy as np
import pytest

import bench
import oracle
import workloads


@pytest.mark.parametrize("spec", [
    dict(seq_len_q=[5, 9], seq_len_kv=[7, 3], alignment="top_left", right_bound=None, left_bound=None),
    dict(seq_len_q=[5, 9], seq_len_kv=[7, 12], alignment="bottom_right", right_bound=0, left_bound=None),
    dict(seq_len_q=None, seq_len_kv=None, alignment="top_left", right_bound=0, left_bound=4),
    dict(seq_len_q=[9, 2], seq_len_kv=None, alignment="bottom_right", right_bound=2, left_bound=3),
])
def test_visible_pairs_counts_the_oracle_band(spec):
    """FLOPs of a banded workload are 4E / 10E per visible (query, key) pair; the count must be
    the number of finite entries of the oracle's band bias, over batches and query heads."""
    w = workloads.get("gqa_causal_e128").with_(B=2, Hq=3, Hkv=1, L=9, S=12)
    band = oracle.Band(spec["seq_len_q"], spec["seq_len_kv"], spec["alignment"], spec["right_bound"],
                       spec["left_bound"])
    want = sum(int(np.isfinite(oracle.band_bias(w.L, w.S, band, b)).sum()) for b in range(w.B)) * w.Hq
    assert bench.visible_pairs(w, spec) == want


def test_summarize_launches_aggregates_per_kernel(tmp_path):
    rows = [
        '"ID","Kernel Name","Metric Name","Metric Unit","Metric Value"',
        '"0","void sdpa_impl::fwd_tc_kernel<2, 2, 0, false>(CUtensorMap_st)","gpu__time_duration.sum","us","200.5"',
        '"1","void sdpa_impl::bwd_tc_kernel<128, false, false>(CUtensorMap_st)","gpu__time_duration.sum","ms","0.6"',
        '"2","void sdpa_impl::fwd_tc_kernel<2, 2, 0, false>(CUtensorMap_st)","gpu__time_duration.sum","ns","199,500"',
        '"3","void sdpa_impl::fwd_tc_kernel<2, 2, 0, false>(CUtensorMap_st)","dram__bytes_read.sum","byte","5"',
    ]
    path = tmp_path / "launches.csv"
    path.write_text("==PROF== noise line\n" + "\n".join(rows) + "\n")
    out = bench.summarize_launches(str(path)).splitlines()
    assert out[0].split()[:2] == ["kernel", "launches"]
    body = {ln.split()[0]: ln.split()[-3:] for ln in out[1:]}
    # bwd: 600 us in one launch, 60 % of 1000 us; fwd: two launches, 400 us, 40 %
    assert body["sdpa_impl::bwd_tc_kernel<128,"] == ["1", "0.600", "60.00%"]
    assert body["sdpa_impl::fwd_tc_kernel<2,"] == ["2", "0.400", "40.00%"]


def test_traffic_figures_are_dropped_when_the_source_differs():
    """A committed DRAM-traffic figure is reported only while the kernel's sources hash to the
    value recorded with it; any other source set (or an unknown kernel) gives None."""
    assert bench.traffic_for("fwd_tc_kernel", ["decode.cu", "ptx.cuh", "common.cuh"]) is None
    assert bench.traffic_for("no_such_kernel", ["fwd_tc_kernel.cuh"]) is None
    sha = bench.source_sha("fwd_tc_kernel.cuh", "ptx.cuh", "common.cuh")
    assert len(sha) == 16 and sha == bench.source_sha("fwd_tc_kernel.cuh", "ptx.cuh", "common.cuh")
    assert os.path.exists(os.path.join(bench.ROOT, "profiles", "traffic.json"))


@pytest.mark.parametrize("name", ["gqa_causal_e128", "mha_causal_e64", "padded_seqlen_e128", "gqa_swa_e128",
                                  "gqa_decode_s32k"])
def test_group_work_sums_to_the_workload_total(name):
    """The CPU baseline scales its sampled KV groups by work: the groups' work must add up to
    the workload's (nominal FLOPs, visible-pair FLOPs, or the decode's bytes)."""
    w = workloads.get(name)
    spec = workloads.make_band(w, seed=0)
    total = sum(bench.group_work(w, spec, b) for b in range(w.B) for _ in range(w.Hkv))
    if "bwd" not in w.phases:
        want = w.B * w.Hkv * w.S * (w.E + w.Ev) * 2 + w.B * w.Hq * w.L * ((w.E + w.Ev) * 2 + 4)
    elif spec is None:
        want = w.flops("fwd") + w.flops("bwd")
    else:
        want = 14.0 * w.E * bench.visible_pairs(w, spec)
    assert total == pytest.approx(want, rel=1e-12)


def test_computed_peak_is_sms_times_rate_times_clock():
    assert bench.computed_peak_tflops(152, 2070.0) == pytest.approx(152 * 8182 * 2.07e9 / 1e12)


def test_clock_sampler_keeps_only_the_samples_inside_its_window(tmp_path):
    """Clock figures come from the samples taken between two host-time marks (the loops under
    load), not from the idle samples around them."""
    import datetime
    t0 = datetime.datetime(2026, 1, 1, 12, 0, 0)
    path = tmp_path / "clocks.csv"
    rows = []
    for i, (mhz, cap) in enumerate([(1000, "Not Active"), (2070, "Not Active"), (2040, "Active"),
                                    (2070, "Not Active"), (900, "Not Active")]):
        ts = (t0 + datetime.timedelta(milliseconds=200 * i)).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        rows.append(f"{ts}, 0, {mhz}, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, {cap}")
    path.write_text("\n".join(rows) + "\n")
    clk = bench.ClockSampler(0)
    clk.proc, clk.path = object(), str(path)
    clk.marks = {"a": t0 + datetime.timedelta(milliseconds=100), "b": t0 + datetime.timedelta(milliseconds=700)}
    s = clk.summary("a", "b")
    assert s["samples"] == 3 and s["sm_mhz"] == 2070 and s["sm_mhz_min"] == 2040
    assert s["reasons"] == ["sw_power_cap"]
    assert clk.summary()["samples"] == 5
