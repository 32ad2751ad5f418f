"""Host-side checks of the C ABI (no GPU needed): the library loads, exports every symbol the header
declares, computes the documented buffer sizes, and rejects bad arguments synchronously (status codes
are returned before any CUDA call is made, so fake pointers are safe here)."""
import ctypes
import os
import re

import pytest

from block_quantized_int8_q8_gb300 import _build, api

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return api.load()


def test_header_declares_exactly_the_exported_api(lib):
    header = open(os.path.join(ROOT, "include", "mmq.h")).read()
    declared = set(re.findall(r"\b(mmq_[a-z0-9_]+)\s*\(", header))
    assert declared == set(api.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name


def test_sizes(lib):
    o = api.q8_1_offsets(3, 64)
    assert o["ds"] == 3 * 64 and o["h"] % 256 == 0 and o["h"] >= 3 * 64 + 3 * 2 * 8
    assert o["dT"] >= o["h"] + 3 * 64 * 2 and o["dT"] % 256 == 0 and o["sT"] == o["dT"] + 4 * 2 * 4
    assert api.q8_1_bytes(3, 64) == (o["sT"] + 4 * 2 * 4 + 255) // 256 * 256
    assert api.q8_1_bytes(3, 64) == int(api.load().mmq_q8_1_bytes(3, 64))
    assert api.q8_1_bytes(3, 32) == 0                     # K % 64 required
    assert api.weight_bytes(api.Q8_0, 5, 256) == 5 * 8 * 34
    assert api.weight_bytes(api.Q4_0, 5, 256) == 5 * 8 * 18
    assert api.weight_bytes(api.Q4_K, 5, 512) == 5 * 2 * 144
    assert api.weight_bytes(api.IQ1_M, 5, 512) == 5 * 2 * 76
    assert api.weight_bytes(api.Q6_K, 5, 512) == 5 * 2 * 224
    assert api.weight_bytes(api.Q6_K, 5, 100) == 0
    assert api.weight_bytes(api.W8A8, 5, 64) == 5 * 64 + 20
    assert api.weight_bytes(api.Q4_K, 5, 100) == 0
    assert api.w8a8_act_bytes(7, 64) == 7 * 64 + 28
    assert api.gemm_id_workspace_bytes(512, 4096, 8, 64) > 512 * 8 * (4 + 2 * 4096)


FAKE = 1 << 20          # 16-byte aligned, never dereferenced: every case fails validation first


@pytest.mark.parametrize("K", [32, 64, 96, 128, 256, 288, 512, 1024, 0, -256])
def test_size_helpers_agree_with_the_entry_points(lib, K):
    """A size helper returns 0 exactly where its entry point rejects the shape: with a null pointer the
    entry point answers MMQ_ERR_SHAPE (2) for a bad K and MMQ_ERR_INVALID_ARG (1) once the shape passes,
    so no kernel is ever launched here."""
    for t in (api.Q8_0, api.Q4_0, api.Q4_K, api.IQ1_M, api.W8A8, api.Q6_K):
        st = lib.mmq_gemm(t, None, FAKE, FAKE, 4, 4, K, None)
        assert st in (1, 2), (t, K, st)
        assert (api.weight_bytes(t, 4, K) == 0) == (st == 2), (t, K)
        if t != api.W8A8:
            sid = lib.mmq_gemm_id(t, None, 2, FAKE, FAKE, 2, FAKE, 4, 4, K, FAKE, 1 << 30, None)
            assert sid == st, (t, K, sid)
    sq = lib.mmq_quantize_q8_1(None, 4, K, FAKE, None)
    assert sq in (1, 2)
    assert (api.q8_1_bytes(4, K) == 0) == (sq == 2), K
    assert (api.w8a8_act_bytes(4, K) == 0) == (lib.mmq_gemm(api.W8A8, None, FAKE, FAKE, 4, 4, K, None) == 2), K


@pytest.mark.parametrize("args,status", [
    ((api.Q4_0, FAKE, FAKE, FAKE, 4, 4, 100), 2),        # K not a multiple of 256
    ((api.Q4_0, FAKE, FAKE, FAKE, -1, 4, 256), 2),       # negative M
    ((api.W8A8, FAKE, FAKE, FAKE, 4, 4, 96), 2),         # W8A8 K % 64
    ((7, FAKE, FAKE, FAKE, 4, 4, 256), 1),               # unknown type
    ((api.Q4_0, None, FAKE, FAKE, 4, 4, 256), 1),        # null weights
    ((api.Q4_0, FAKE + 4, FAKE, FAKE, 4, 4, 256), 3),    # misaligned
    ((api.Q4_0, FAKE, FAKE, FAKE, 1 << 20, 1 << 12, 1 << 12), 2),   # M*K beyond int32
])
def test_gemm_argument_validation(lib, args, status):
    assert lib.mmq_gemm(*args, None) == status


def test_quantize_and_gemm_id_validation(lib):
    assert lib.mmq_quantize_q8_1(FAKE, 4, 33, FAKE, None) == 2
    assert lib.mmq_quantize_q8_1(None, 4, 64, FAKE, None) == 1
    assert lib.mmq_quantize_q8_1(FAKE, 4, 64, FAKE + 8, None) == 3
    assert lib.mmq_q8_1_prepare(FAKE, 4, 96, None) == 2
    assert lib.mmq_q8_1_prepare(None, 4, 64, None) == 1
    ok = (api.IQ1_M, FAKE, 4, FAKE, FAKE, 2, FAKE, 16, 128, 256)
    need = api.gemm_id_workspace_bytes(16, 256, 2, 4)
    assert lib.mmq_gemm_id(*ok, FAKE, need - 1, None) == 6          # workspace too small
    assert lib.mmq_gemm_id(*ok, None, need, None) == 6
    assert lib.mmq_gemm_id(api.W8A8, *ok[1:], FAKE, need, None) == 4
    assert lib.mmq_gemm_id(api.IQ1_M, FAKE, 0, *ok[3:], FAKE, need, None) == 1
    # four tokens take the matrix-vector kernel, which uses no workspace; the contract still checks it
    few = (api.Q4_0, FAKE, 4, FAKE, FAKE, 2, FAKE, 4, 128, 256)
    need4 = api.gemm_id_workspace_bytes(4, 256, 2, 4)
    assert lib.mmq_gemm_id(*few, FAKE, need4 - 1, None) == 6
    assert lib.mmq_gemm_id(*few, None, need4, None) == 6
    assert lib.mmq_gemm_id(*few, FAKE + 8, need4, None) == 3
    assert lib.mmq_gemm_id(api.Q4_0, FAKE, 4, FAKE, FAKE, 2, FAKE, 4, 128, 96, FAKE, need4, None) == 2
    assert lib.mmq_gemm_debug_partials(api.Q4_K, FAKE, FAKE, FAKE, 4, 4, 128, None) == 2
    assert lib.mmq_gemm_debug_partials(api.Q6_K, FAKE, FAKE, FAKE, 4, 4, 256, None) == 4   # TMA kernel only
    assert lib.mmq_gemm(6, FAKE, FAKE, FAKE, 4, 4, 256, None) == 1                         # unknown type
    # the no-allocation MoE entry point: types it does not implement, and its shape rules
    for t in (api.W8A8, api.Q6_K):
        assert lib.mmq_gemm_id_noalloc(t, FAKE, 4, FAKE, FAKE, 2, FAKE, 16, 128, 256, None) == 4
    assert lib.mmq_gemm_id_noalloc(api.Q4_0, FAKE, 4, FAKE, FAKE, 2, FAKE, 16, 128, 96, None) == 2
    assert lib.mmq_gemm_id_noalloc(api.Q4_0, None, 4, FAKE, FAKE, 2, FAKE, 16, 128, 256, None) == 1
    for s in range(7):
        assert lib.mmq_status_string(s)
    assert lib.mmq_read_device_errors(None, None) == 1
