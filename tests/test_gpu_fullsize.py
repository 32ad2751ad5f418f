"""Full-size parity: every workload at its full shape, through the same calls and launch configuration
the benchmark times, checked against the CPU oracle on sampled outputs.

The oracle cannot recompute a 2048 x 11008 x 4096 product in test time, so each case compares a sample
of whole output rows (tokens), chosen to include the first and last token and tokens in the ragged
last tile, against the oracle's blockwise product for exactly those tokens (oracle.gemm_rows /
oracle.w8a8 / oracle.gemm_id on the sampled rows).  The quantizer is checked bit for bit on the whole
activation matrix.  Bars as in test_gpu_parity: f32 within 1e-3 of the sample's output scale, W8A8
bf16 bit-exact, q8_1 codes / scales / sums bit-exact.
"""
import numpy as np
import pytest
import torch

import oracle
from block_quantized_int8_q8_gb300 import api, synth

pytestmark = pytest.mark.gpu
TOL = 1e-3
DEV = "cuda"
N_SAMPLE = 12


@pytest.fixture(scope="module", autouse=True)
def _lib():
    api.load()
    yield
    assert api.read_device_errors() == 0


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _sample_rows(M, seed):
    g = np.random.default_rng(seed)
    last_tile = (M - 1) // 128 * 128
    rows = {0, M - 1, last_tile, min(M - 1, last_tile + 1)}
    rows.update(int(r) for r in g.choice(M, size=min(M, N_SAMPLE), replace=False))
    return np.array(sorted(rows), dtype=np.int64)


def _rel_err(got, ref):
    scale = np.abs(ref).max()
    return float(np.abs(got.astype(np.float64) - ref).max() / (scale if scale > 0 else 1.0))


@pytest.mark.parametrize("name", ["q8_0_tiny", "q4_0_7b", "q4_k_ffn_up", "iq1_m_dense", "q6_k_ffn_down"])
def test_dense_block_workload_full_size(name):
    pb = synth.workload(name)
    M, N, K = pb.M, pb.N, pb.K
    xq = api.quantize_q8_1(_dev(pb.x))
    out = api.gemm(pb.wtype, _dev(pb.W.reshape(-1)), xq, M, N, K)
    torch.cuda.synchronize()
    # the whole q8_1 matrix bit for bit
    q, d, s = oracle.quantize_q8_1(pb.x)
    qg, dsg = api.q8_1_views(xq, M, K)
    assert np.array_equal(qg.cpu().numpy(), q)
    assert np.array_equal(dsg[..., 0].cpu().numpy().view(np.uint32), d.view(np.uint32))
    assert np.array_equal(dsg[..., 1].cpu().numpy().view(np.uint32), s.view(np.uint32))
    # sampled token rows of the product
    rows = _sample_rows(M, seed=M + N)
    ref = oracle.gemm_rows(pb.wtype, pb.W, q, d, s, N, rows)
    got = out[torch.from_numpy(rows).to(DEV)].cpu().numpy()
    assert np.all(np.isfinite(got))
    assert _rel_err(got, ref) <= TOL


@pytest.mark.parametrize("name", ["w8a8_m3072", "w8a8_m4096"])
def test_w8a8_workload_full_size_bit_exact(name):
    pb = synth.workload(name)
    M, N, K = pb.M, pb.N, pb.K
    out = api.gemm(synth.W8A8, _dev(pb.W), _dev(synth.pack_w8a8_acts(pb.X, pb.xs)), M, N, K)
    rows = _sample_rows(M, seed=M + N)
    got = out[torch.from_numpy(rows).to(DEV)].view(torch.int16).cpu().numpy().view(np.uint16)
    ref = oracle.w8a8(pb.fields.W, pb.fields.ws, pb.X[rows], pb.xs[rows])
    assert np.array_equal(got, ref)


def test_iq1_m_moe_workload_full_size():
    pb = synth.workload("iq1_m_moe")
    M, N, K, E = pb.M, pb.N, pb.K, pb.experts
    xq = api.quantize_q8_1(_dev(pb.x))
    out = api.gemm_id(pb.wtype, _dev(pb.W.reshape(-1)), E, xq, _dev(pb.ids), M, N, K)
    q, d, s = oracle.quantize_q8_1(pb.x)
    rows = _sample_rows(M, seed=7)
    ref = oracle.gemm_id(pb.wtype, pb.W, E, q[rows], d[rows], s[rows], pb.ids[rows], N)
    got = out[torch.from_numpy(rows).to(DEV)].cpu().numpy()
    for i in range(len(rows)):
        for j in range(pb.ids.shape[1]):
            assert _rel_err(got[i, j], ref[i, j]) <= TOL, (int(rows[i]), j)
