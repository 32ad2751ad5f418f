"""mmq_gemm_id_noalloc: the MoE product for callers that cannot allocate device memory.

Such callers (an engine with a fixed device-memory budget, a framework allocator that owns the
device, a plugin handed only its buffers) cannot pass mmq_gemm_id a workspace; this entry point keeps
the routing lists in the library's static scratch array.  The test calls it through the C ABI twice in
a row and checks both results against mmq_gemm_id (same tolerance as the other parity tests), and
that a problem too large for the array is rejected.  It lives in its own file, collected last.
"""
import numpy as np
import pytest
import torch

from block_quantized_int8_q8_gb300 import _build, api, synth

pytestmark = pytest.mark.gpu
TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    _build.build()
    api.load()
    yield


def _rel(a, b):
    return float((a.double() - b.double()).abs().max() / b.double().abs().max().clamp_min(1e-30))


@pytest.mark.parametrize("wtype,M,E,slots,N,K", [(synth.IQ1_M, 512, 64, 8, 1536, 4096),
                                                  (synth.Q4_K, 70, 9, 3, 200, 512)])
def test_noalloc_matches_workspace_entry_point_twice(wtype, M, E, slots, N, K):
    pb = synth.make_problem(wtype, M, N, K, seed=91 + M, experts=E, slots=slots)
    dev = "cuda"
    W = torch.from_numpy(pb.W.reshape(-1)).to(dev)
    xq = api.quantize_q8_1(torch.from_numpy(pb.x).to(dev))
    ids = torch.from_numpy(pb.ids).to(dev)
    ref = api.gemm_id(wtype, W, E, xq, ids, M, N, K)
    first = api.gemm_id_noalloc(wtype, W, E, xq, ids, M, N, K)
    second = api.gemm_id_noalloc(wtype, W, E, xq, ids, M, N, K)
    torch.cuda.synchronize()
    assert api.read_device_errors() == 0
    assert _rel(first, ref) <= TOL
    assert _rel(second, ref) <= TOL


@pytest.mark.parametrize("wtype", [synth.Q8_0, synth.Q4_0, synth.Q4_K, synth.IQ1_M])
def test_noalloc_larger_call_then_smaller_call(wtype):
    # the shared array keeps the previous call's lists: a larger problem (more experts, more rows) run
    # first must not leak into a smaller one with a different expert count run right after
    N, K = 136, 1024
    big = synth.make_problem(wtype, 90, N, K, seed=201, experts=24, slots=4)
    small = synth.make_problem(wtype, 17, N, K, seed=202, experts=5, slots=2)
    dev = "cuda"
    for pb in (big, small):
        pb.Wd = torch.from_numpy(pb.W.reshape(-1)).to(dev)
        pb.xq = api.quantize_q8_1(torch.from_numpy(pb.x).to(dev))
        pb.idsd = torch.from_numpy(pb.ids).to(dev)
    ref_small = api.gemm_id(wtype, small.Wd, small.experts, small.xq, small.idsd, small.M, N, K)
    api.gemm_id_noalloc(wtype, big.Wd, big.experts, big.xq, big.idsd, big.M, N, K)
    got_small = api.gemm_id_noalloc(wtype, small.Wd, small.experts, small.xq, small.idsd, small.M, N, K)
    torch.cuda.synchronize()
    assert api.read_device_errors() == 0
    assert _rel(got_small, ref_small) <= TOL


def test_noalloc_rejects_problems_beyond_the_scratch_array():
    M, E, slots, N, K = 300000, 4, 1, 128, 256
    assert M * slots * 4 > api.NOALLOC_SCRATCH_BYTES       # the rowlist alone exceeds the array
    fake = 1 << 20
    rc = api.load().mmq_gemm_id_noalloc(synth.Q4_0, fake, E, fake, fake, slots, fake, M, N, K, None)
    assert rc == 6                      # MMQ_ERR_WORKSPACE
