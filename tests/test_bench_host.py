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
