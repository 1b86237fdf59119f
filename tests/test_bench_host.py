"""Host-side arithmetic of bench.py, checked without a GPU: the FLOP
convention, the algorithmic bytes of a paged decode call, the whole-job rate,
the per-rank workloads of the weak-scaling run, the peak denominators, the CPU
oracle sample, and the rule that an ncu traffic figure is reported only while
the kernel's sources are the ones it was captured on."""

import json
import os
import shutil

import pytest

import bench
from causal_head_attention_gb300.inputs import HEADLINE, TINY, PagedWorkload


def test_forward_flop_convention():
    # 4 * B * H * T^2 * Dh / 2: the unmasked half of the two T x T x Dh products.
    assert bench.fwd_flops(HEADLINE) == 4 * 4 * 16 * 2048 * 2048 * 64 / 2 == 34359738368


def test_decode_bytes_by_hand():
    w = PagedWorkload("bytes", 2, 4, 2, 16, 16, 40, "bf16", 1)
    lens = [5, 17]
    kv = (5 + 17) * 2 * 16 * 2 * 2  # positions x Hkv x Dh x (K and V) x bf16
    q_out = 2 * 2 * 4 * 16 * 2  # query and output: B x Hq x Dh each, bf16
    lse = 2 * 4 * 4  # B x Hq fp32
    table = (1 + 2) * 4  # pages in use: ceil(5/16) + ceil(17/16), int32
    seq_lens = 2 * 4
    assert bench.decode_bytes(w, lens) == kv + q_out + lse + table + seq_lens
    w32 = PagedWorkload("bytes32", 2, 4, 2, 16, 16, 40, "fp32", 1)
    assert bench.decode_bytes(w32, lens) == 2 * kv + 2 * q_out + lse + table + seq_lens


def test_materialized_bytes_by_brute_force():
    """Each figure counted element by element on small [T, T] blocks: kept
    entries j <= i, whole rows, and the tiled VJP's columns j < min(T, 128
    (i // 128 + 1)), with T past one tile and ragged."""
    for E, T in ((1, 1), (2, 5), (3, 130), (1, 300)):
        kept = sum(i + 1 for i in range(T)) * E * 4
        rows = E * T * T * 4
        tiled = E * 4 * sum(len([j for j in range(T) if j < min(T, 128 * (i // 128 + 1))]) for i in range(T))
        mb = bench.materialized_bytes(E, T)
        assert mb["tri"] == kept and mb["full"] == rows
        assert mb["fwd"] == rows + kept
        assert mb["softmax"] == kept + rows + E * T * 4
        assert mb["softmax_bwd"] == 2 * kept + rows
        assert mb["softmax_bwd_tiled128"] == 2 * kept + tiled
        assert mb["bwd_products"] == 4 * kept
    # the tiled VJP writes less than whole rows once a row has a tile past its diagonal one
    assert bench.materialized_bytes(1, 300)["softmax_bwd_tiled128"] < bench.materialized_bytes(1, 300)["softmax_bwd"]


def test_aggregate_rate_counts_every_rank_over_the_slowest():
    assert bench.aggregate_tflops(1e12, 1, 1000.0) == pytest.approx(1.0)
    assert bench.aggregate_tflops(1e12, 4, 500.0) == pytest.approx(8.0)


def test_rank_workloads_are_distinct_and_same_shape():
    ws = [bench.rank_workload(HEADLINE, r) for r in range(4)]
    assert ws[0] is HEADLINE
    assert len({w.seed for w in ws}) == 4
    assert all((w.B, w.Hq, w.Hkv, w.T, w.Dh, w.dtype) == (HEADLINE.B, HEADLINE.Hq, HEADLINE.Hkv, HEADLINE.T,
                                                       HEADLINE.Dh, HEADLINE.dtype) for w in ws)


def test_peaks_measured_or_fallback(tmp_path, monkeypatch):
    p = bench.peaks()
    if os.path.exists(os.path.join(bench.ROOT, "MEASURED_PEAKS.json")):
        assert p["source"] == "measured" and p["hbm_gbs"] > 0 and p["bf16_tflops"] > 0
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    fb = bench.peaks()
    assert fb["source"] == "fallback" and fb["hbm_gbs"] == 6800.0 and fb["bf16_tflops"] == 1900.0


def test_traffic_is_reported_only_for_the_captured_sources(tmp_path, monkeypatch):
    src = os.path.join(bench.ROOT, "causal_head_attention_gb300", "csrc")
    dst = tmp_path / "causal_head_attention_gb300" / "csrc"
    shutil.copytree(src, dst)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.src_digest("decode") == bench.src_digest("decode")
    assert bench.src_digest("decode") != bench.src_digest("fwd")
    (tmp_path / "profiles").mkdir()
    traffic = {"wl": {"decode": {"dram_bytes_per_launch": 123.0, "src_digest": bench.src_digest("decode")}}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(traffic))
    assert bench.ncu_traffic("decode", "wl") == 123.0
    assert bench.ncu_traffic("decode", "other") is None
    fwd_before = bench.src_digest("fwd")
    with open(dst / "decode.cu", "a") as f:
        f.write("\n// edited\n")
    assert bench.ncu_traffic("decode", "wl") is None  # the capture no longer describes the kernel
    assert bench.src_digest("fwd") == fwd_before  # other kernels' digests are unaffected


def test_oracle_sample_is_bounded_and_counts_whole_groups():
    flops, secs, threads, groups = bench.oracle_sample(TINY, 0.0, max_groups=2)
    per_group = 3.5 * 4.0 * TINY.group * TINY.T * TINY.T * TINY.Dh / 2.0
    assert 1 <= groups <= 2 and threads >= 1 and secs >= 0
    assert flops == groups * per_group


def test_step_spread_percentiles():
    s = bench.spread([float(x) for x in range(1, 12)])  # 1 .. 11
    assert s["mean"] == pytest.approx(6.0) and s["median"] == pytest.approx(6.0)
    assert s["p10"] == pytest.approx(2.0) and s["p90"] == pytest.approx(10.0)


def test_nominal_peak_arithmetic():
    # 152 SMs x 8192 bf16 FLOP per clock x 2070 MHz; TF32 at half the rate
    assert bench.nominal_tflops(152, 2070.0, "bf16") == pytest.approx(152 * 8192 * 2.07e9 / 1e12)
    assert bench.nominal_tflops(152, 2070.0, "fp32") == pytest.approx(bench.nominal_tflops(152, 2070.0, "bf16") / 2)


def test_both_arms_print_the_same_config(capsys):
    cfg = bench.config_for(HEADLINE, 1)
    nsets, set_bytes = bench.input_sets(HEADLINE)
    assert set_bytes == 2 * 4 * 2048 * 64 * (2 * 16 + 2 * 16)
    assert nsets * set_bytes > 2 * bench.L2_BYTES
    assert cfg["workload"] == HEADLINE.describe() and cfg["global_batch"] == 4 and str(nsets) in cfg["l2"]

    class A:
        steps, warmup = 1, 0
        metric = "m"

    assert bench.run_reference(A, TINY, 1, 0) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["config"] == bench.config_for(TINY, 1)
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_launch_count_per_step():
    assert bench.launches_per_step(HEADLINE) == 4
    assert bench.launches_per_step(TINY) == 8
