"""Host-side arithmetic of the benchmark (no GPU): the algorithmic bytes behind
the attention roofline, and the rule that DRAM traffic from a committed ncu
summary is reported only while that summary was taken on the current kernel
source."""
import hashlib
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from block_diffusion_speculative_fusion_gb300 import synth  # noqa: E402
from block_diffusion_speculative_fusion_gb300 import workloads as W  # noqa: E402


def test_attn_bytes_counts_every_row_once():
    # count the bytes row by row: each sequence's context rows and block rows,
    # for K and V, every kv head, D bf16 values; Q read once and O written once
    wl = W.LLAMA8B_B64
    ctx = synth.ctx_lengths(wl, 0).tolist()
    nbytes = 0
    for c in ctx:
        for _row in range(c + wl.k):
            for _tensor in ("K", "V"):
                nbytes += wl.Hkv * wl.D * 2
    for _tensor in ("Q", "O"):
        nbytes += wl.B * wl.k * wl.Hq * wl.D * 2
    assert bench.attn_bytes(float(sum(ctx)), wl) == nbytes
    # the throughput workload moves 1.165 GB per layer
    assert abs(nbytes / 1e9 - 1.165) < 1e-3


def _fake_tree(tmp_path, src_text, recorded_hash, traffic):
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "attn_tc_kernel_llama8b_b64.md").write_text(
        f"# summary\n\n- source_sha256_16: {recorded_hash}\n- dram_bytes_per_launch_full_size: {traffic}\n")
    csrc = tmp_path / "block_diffusion_speculative_fusion_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "attn.cu").write_text(src_text)


def test_traffic_reported_only_for_the_profiled_source(tmp_path, monkeypatch):
    src = "// kernel source\n"
    digest = hashlib.sha256(src.encode()).hexdigest()[:16]
    _fake_tree(tmp_path, src, digest, 1234)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_from_profile("attn.cu") == 1234.0
    # the kernel changed after the capture: no traffic figure
    (tmp_path / "block_diffusion_speculative_fusion_gb300" / "csrc" / "attn.cu").write_text(src + "// edit\n")
    assert bench.traffic_from_profile("attn.cu") is None


def test_committed_profile_carries_the_keys_bench_reads():
    path = os.path.join(ROOT, "profiles", "attn_tc_kernel_llama8b_b64.md")
    keys = {}
    for line in open(path):
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            keys[k.strip()] = v.strip()
    assert len(keys["source_sha256_16"]) == 16
    int(keys["source_sha256_16"], 16)
    assert float(keys["dram_bytes_per_launch_full_size"]) > 1e9


@pytest.mark.parametrize("steps,ms,world,expect", [(500, 820.0, 1, 500 / 0.82), (500, 820.0, 4, 4 * 500 / 0.82)])
def test_replica_throughput_counts_all_ranks(steps, ms, world, expect):
    assert abs(bench.replica_throughput(steps, ms, world) - expect) < 1e-9


def test_kernel_durations_count_dependents_from_their_predecessor():
    # a programmatic dependent that started while its predecessor ran is
    # charged from the predecessor's end; other kernels keep their own span
    ev = [("void dflash::mat_gather_kernel(int)", 0.0, 10.0),
          ("dflash::gemm_tc_kernel(CUtensorMap_st)", 5.0, 50.0),
          ("void dflash::mat_bias_kernel<__nv_bfloat16>(float*)", 40.0, 60.0),
          ("void dflash::greedy_kernel<__nv_bfloat16>(int)", 45.0, 70.0),
          ("void dflash::sample_draw_kernel<float>(int)", 65.0, 80.0)]
    d = bench.kernel_durations(ev)
    assert d == {"mat_gather_kernel": [10.0], "gemm_tc_kernel": [40.0], "mat_bias_kernel": [10.0],
                 "greedy_kernel": [25.0], "sample_draw_kernel": [15.0]}
