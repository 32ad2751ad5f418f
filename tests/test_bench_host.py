"""Host-side bookkeeping of bench.py that needs no GPU: the recorded DRAM traffic of a kernel is reported
only while the kernel's sources are the ones it was captured on, and the rescale ceiling follows its
definition (FP32 instructions per 32-k element-block)."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from block_quantized_int8_q8_gb300 import synth  # noqa: E402


def test_recorded_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    rec = {"w": {"kernel": "mmq_gemm_tma_kernel", "kernel_hash": bench.kernel_source_hash("mmq_gemm_tma_kernel"),
                 "dram_bytes_per_launch": 1234.0}}
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    os.symlink(os.path.join(ROOT, "block_quantized_int8_q8_gb300"), tmp_path / "block_quantized_int8_q8_gb300")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("w", "mmq_gemm_tma_kernel") == 1234.0
    assert bench.recorded_traffic("w", "mmq_w8a8_tma_kernel") is None       # another kernel's record
    assert bench.recorded_traffic("absent", "mmq_gemm_tma_kernel") is None
    rec["w"]["kernel_hash"] = "0" * 16                                         # sources changed since
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    assert bench.recorded_traffic("w", "mmq_gemm_tma_kernel") is None


def test_committed_traffic_matches_the_committed_kernels():
    # every workload has a record in profiles/traffic.json naming the kernel bench.py times for it; the
    # extra records are token-count runs ("<workload>_m<M>", bench.py --tokens M) of the few-token kernel
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    assert set(synth.WORKLOADS) <= set(rec)
    for w, ent in rec.items():
        if w in synth.WORKLOADS:
            want = "mmq_w8a8_tma_kernel" if synth.WORKLOADS[w]["wtype"] == synth.W8A8 else "mmq_gemm_tma_kernel"
        else:
            base, _, m = w.rpartition("_m")
            assert base in synth.WORKLOADS and synth.WORKLOADS[base]["wtype"] != synth.W8A8 and 1 <= int(m) <= 8
            want = "mmvq_kernel"
        assert ent["kernel"] == want
        assert ent["dram_bytes_per_launch"] > 0


def test_rescale_ceiling_definition():
    ops = 2.0 * 2048 * 4096 * 4096
    c = bench.rescale_ceiling(synth.Q4_0, ops, 30.0)
    assert c["element_blocks"] == ops / 64
    # 30 TFLOP/s of FMA = 15 T FP32 instructions/s; 2 per element-block of 64 ops
    assert abs(c["ceiling_tops"] - 15.0 / 2 * 64) < 1e-9
    assert bench.rescale_ceiling(synth.Q4_K, ops, 30.0)["fp32_instr_per_element_block"] == 3
    assert bench.rescale_ceiling(synth.W8A8, ops, 30.0) is None
    assert bench.rescale_ceiling(synth.Q4_0, ops, None) is None


def test_fewtoken_bytes_counts_only_the_routed_experts():
    # the few-token roofline's bytes: weight rows read (a MoE call reads only its tokens' experts), the
    # q8_1 codes and (d, s) pairs of the tokens, the f32 outputs (one row per (token, slot) pair)
    M, N, K, E = 2, 64, 256, 8
    pb = synth.make_problem(synth.IQ1_M, M, N, K, seed=3, experts=E, slots=2)
    ids = pb.ids.copy()
    ids[:] = [[1, 5], [5, 2]]
    pb.ids = ids
    per_expert = N * (K // 256) * 76
    assert pb.W.nbytes == E * per_expert
    assert bench.fewtoken_bytes(dict(pb=pb, M=M, N=N, K=K)) == 3 * per_expert + M * K + M * (K // 32) * 8 + 4 * N * 4
    dense = synth.make_problem(synth.Q4_0, M, N, K, seed=4)
    assert bench.fewtoken_bytes(dict(pb=dense, M=M, N=N, K=K)) == N * (K // 32) * 18 + M * K + M * (K // 32) * 8 + M * N * 4


def test_workload_ops_count_every_routed_row_and_config_names_the_routing():
    ops, tokens = bench.workload_ops("iq1_m_moe")
    w = synth.WORKLOADS["iq1_m_moe"]
    assert tokens == w["M"] and ops == 2.0 * w["M"] * w["slots"] * w["N"] * w["K"]
    cfg = bench.workload_config("iq1_m_moe")
    assert cfg["experts"] == w["experts"] and cfg["slots"] == w["slots"] and cfg["wtype"] == "IQ1_M"
    assert "experts" not in bench.workload_config("q4_0_7b")
    # weak scaling: every rank does a step's units; the job rate is over the slowest rank's time
    assert bench.job_throughput(10.0, 4, 3, 2.0) == 60.0


class _FakeProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def test_clock_record_keeps_the_timed_window_and_reports_throttle_reasons(tmp_path):
    # nvidia-smi lines: timestamp, sm, max sm, power, active mask, hw_slowdown, hw_thermal, sw_thermal,
    # sw_power_cap; the first and last samples fall outside the timed window and are dropped
    lines = [
        "2026/01/02 10:00:00.000, 900 MHz, 2070 MHz, 120.0 W, 0x0, Not Active, Not Active, Not Active, Not Active",
        "2026/01/02 10:00:01.000, 2070 MHz, 2070 MHz, 900.5 W, 0x4, Not Active, Not Active, Not Active, Active",
        "2026/01/02 10:00:01.020, 2040 MHz, 2070 MHz, 910.0 W, 0x0, Not Active, Not Active, Not Active, Not Active",
        "2026/01/02 10:00:01.040, 2055 MHz, 2070 MHz, 905.0 W, 0x0, Not Active, Not Active, Not Active, Not Active",
        "2026/01/02 10:00:05.000, 600 MHz, 2070 MHz, 100.0 W, 0x8, Active, Not Active, Not Active, Not Active",
        "garbage line",
    ]
    import datetime
    ts = lambda s: datetime.datetime.strptime(s, "%Y/%m/%d %H:%M:%S.%f").timestamp()   # noqa: E731
    cs = bench.ClockSampler("0")
    cs.path = str(tmp_path / "clocks.csv")
    with open(cs.path, "w") as f:
        f.write("\n".join(lines) + "\n")
    cs.out = open(cs.path, "a")
    cs.proc = _FakeProc()
    cs.mark(ts("2026/01/02 10:00:01.000"), ts("2026/01/02 10:00:01.040"))
    rec = cs.stop()
    assert rec["samples"] == 3
    assert rec["sm_mhz"] == 2055.0 and rec["sm_max_mhz"] == 2070.0 and rec["power_w_max"] == 910.0
    assert rec["reasons"] == ["sw_power_cap"]          # the hw_slowdown sample lies outside the window


def test_clock_record_without_nvidia_smi_says_so():
    rec = bench.ClockSampler("0").stop()
    assert rec["samples"] == 0 and rec["sm_mhz"] is None and rec["reasons"] == ["nvidia-smi unavailable"]


def test_cpu_baseline_is_the_oracle_on_a_bounded_sample():
    pb = synth.workload("q8_0_tiny")
    rec = bench.cpu_baseline(pb, "q8_0_tiny", target_s=0.3)
    assert rec["kind"] == "oracle" and rec["unit"] == "TOPS" and rec["cores"] >= 1 and rec["value"] > 0
    n = int(rec["sample"].split(" of ")[0])
    assert 1 <= n <= pb.M and f"of {pb.M} token rows of q8_0_tiny" in rec["sample"]
    assert rec["tok_per_s"] > 0


def test_reference_arm_runs_on_rank_zero_only():
    # the reference arm times the oracle on the host; under torchrun the other ranks exit 0 without work
    import subprocess
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "q8_0_tiny",
           "--steps", "2", "--warmup", "3"]
    r1 = subprocess.run(cmd, env=dict(os.environ, RANK="1", WORLD_SIZE="2"), capture_output=True, text=True,
                        timeout=300)
    assert r1.returncode == 0 and r1.stdout.strip() == ""
    r0 = subprocess.run(cmd, env=dict(os.environ, RANK="0"), capture_output=True, text=True, timeout=300)
    assert r0.returncode == 0
    line = json.loads(r0.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["steps"] == 2 and line["warmup"] == 3 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["config"]["workload"] == "q8_0_tiny" and line["higher_is_better"] is True
