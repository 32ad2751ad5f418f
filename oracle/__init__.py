"""CPU oracle for block-quantized int8 MMQ (test infrastructure).

This package is TEST INFRASTRUCTURE.  Only `tests/`, `__graft_entry__.smoke()` and the CPU-baseline /
reference legs of `bench.py` may import it.  The CUDA library and its Python binding never import,
link or call anything here, and nothing here is shared with them: the oracle is plain C
(`mmq_oracle.c`, scalar loops, f32 in written order, `-ffp-contract=off`) wrapped by ctypes.

Functions and the passages they follow (page title, section):
  quantize_q8_1   "08 · R1 — int8 MMQ prefill GEMM", §2.2 q8_1 activation pipeline and §3.2 reference
  decode          "08 · R1", §2.1/§2.2 (Q8_0, Q4_0, Q4_K unsigned nibbles + min term);
                  "CUDA: add IQ1_M to MMQ", Design (IQ1_M fold 8g±1, per-16 scale d(2s+1)/8);
                  "08 · R1", §2.2 (q6_K: 6-bit grid minus 32, int8 scales per 16 elements)
  partials        "08 · R1", §2.1 (exact in-block int32 dot)
  block_sums      the same 32-k block dot on the weights with their integer sub-scales folded in
                  ("08 · R1" §2.2 per-sub-block scales, q6_K's two scaled dots; "CUDA: add IQ1_M to
                  MMQ", Design: d(2s+1) per 16 values)
  gemm/gemm_rows  "When the Product Won't Collapse: A Negative Result on int8 Tensor-Core MMQ", §2
                  (blockwise contraction) with the §3.2 per-block correction of "08 · R1"
  w8a8            "INT8 W8A8 GEMM — Prefill", §1-§2 (full-K int32, scale epilogue, bf16)
  gemm_id         "CUDA: add IQ1_M to MMQ", PR description (MUL_MAT_ID: token x routed experts)

Parity pins: every function is pinned by tests in `tests/test_oracle_pins.py` against closed forms,
invariants, brute force and an f64 dequantise-then-matmul bound; see that file's header.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mmq_oracle.c")
_LIB = os.path.join(_HERE, "libmmq_oracle.so")
_lib = None
# The pin suite's mutation self-test points this at a deliberately broken build of the oracle.
_LIB_OVERRIDE = os.environ.get("MMQ_ORACLE_LIB")

Q8_0, Q4_0, Q4_K, IQ1_M, W8A8, Q6_K = 0, 1, 2, 3, 4, 5


def build(force: bool = False, out: str | None = None, defines=()) -> str:
    """Compile the oracle with gcc (plain C, OpenMP over output rows, no fp contraction)."""
    target = out or _LIB
    if force or out or not os.path.exists(target) or os.path.getmtime(target) < os.path.getmtime(_SRC):
        tmp = target + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-std=gnu11",
                               *[f"-D{d}" for d in defines], "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, target)
    return target


def _load():
    global _lib
    if _lib is None:
        if _LIB_OVERRIDE:
            lib = ctypes.CDLL(_LIB_OVERRIDE)
        else:
            build()
            lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        lib.oracle_quantize_q8_1.argtypes = [P, I64, I64, P, P, P]
        lib.oracle_decode.argtypes = [ctypes.c_int, P, I64, I64, P, P, P]
        lib.oracle_partials.argtypes = [ctypes.c_int, P, P, I64, I64, I64, P]
        lib.oracle_block_sums.argtypes = [ctypes.c_int, P, P, I64, I64, I64, P]
        lib.oracle_gemm.argtypes = [ctypes.c_int, P, P, P, P, I64, I64, I64, P]
        lib.oracle_gemm_rows.argtypes = [ctypes.c_int, P, P, P, P, I64, I64, I64, P, I64, P]
        lib.oracle_w8a8.argtypes = [P, P, P, P, I64, I64, I64, P]
        lib.oracle_gemm_id.argtypes = [ctypes.c_int, P, I64, P, P, P, P, I64, I64, I64, I64, P]
        lib.oracle_half_to_float.argtypes = [ctypes.c_uint16]
        lib.oracle_half_to_float.restype = ctypes.c_float
        lib.oracle_float_to_bf16.argtypes = [ctypes.c_float]
        lib.oracle_float_to_bf16.restype = ctypes.c_uint16
        lib.oracle_max_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int):
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (rc={rc})")


def max_threads() -> int:
    return _load().oracle_max_threads()


def quantize_q8_1(x: np.ndarray):
    """x f32 [M, K] -> (q int8 [M, K], d f32 [M, K/32], s f32 [M, K/32])."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    M, K = x.shape
    q = np.empty((M, K), np.int8)
    d = np.empty((M, K // 32), np.float32)
    s = np.empty((M, K // 32), np.float32)
    _check(_load().oracle_quantize_q8_1(_p(x), M, K, _p(q), _p(d), _p(s)))
    return q, d, s


def group_size(wtype: int) -> int:
    return 16 if wtype in (IQ1_M, Q6_K) else 32


def decode(wtype: int, W: np.ndarray, N: int, K: int):
    """Raw weight bytes -> (wq int8 [N, K], wsc f32 [N, K/G], wmin f32 [N, K/32])."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    wq = np.empty((N, K), np.int8)
    wsc = np.empty((N, K // group_size(wtype)), np.float32)
    wmin = np.zeros((N, K // 32), np.float32)
    _check(_load().oracle_decode(wtype, _p(W), N, K, _p(wq), _p(wsc), _p(wmin)))
    return wq, wsc, wmin


def partials(wtype: int, xq: np.ndarray, wq: np.ndarray) -> np.ndarray:
    """Exact per-group int32 dots I[m, n, g] (groups of 32, or 16 for IQ1_M and Q6_K)."""
    xq = np.ascontiguousarray(xq, dtype=np.int8)
    wq = np.ascontiguousarray(wq, dtype=np.int8)
    M, K = xq.shape
    N = wq.shape[0]
    P = np.empty((M, N, K // group_size(wtype)), np.int32)
    _check(_load().oracle_partials(wtype, _p(xq), _p(wq), M, N, K, _p(P)))
    return P


def block_sums(wtype: int, W: np.ndarray, xq: np.ndarray, N: int) -> np.ndarray:
    """Exact 32-k block sums with the weights' integer sub-scale factors folded in: int32 [M, N, K/32]
    (Q4_K: sc_b; IQ1_M: (2s+1) per 16; q6_K: sc per 16; Q8_0 / Q4_0: none)."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.int8)
    M, K = xq.shape
    A = np.empty((M, N, K // 32), np.int32)
    _check(_load().oracle_block_sums(wtype, _p(W), _p(xq), M, N, K, _p(A)))
    return A


def gemm(wtype: int, W: np.ndarray, q: np.ndarray, d: np.ndarray, s: np.ndarray, N: int) -> np.ndarray:
    """Blockwise MMQ product: f32 [M, N]."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    q = np.ascontiguousarray(q, dtype=np.int8)
    d = np.ascontiguousarray(d, dtype=np.float32)
    s = np.ascontiguousarray(s, dtype=np.float32)
    M, K = q.shape
    out = np.empty((M, N), np.float32)
    _check(_load().oracle_gemm(wtype, _p(W), _p(q), _p(d), _p(s), M, N, K, _p(out)))
    return out


def gemm_rows(wtype: int, W: np.ndarray, q: np.ndarray, d: np.ndarray, s: np.ndarray, N: int,
              rows) -> np.ndarray:
    """Blockwise MMQ product for the selected activation rows only: f32 [len(rows), N]."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    q = np.ascontiguousarray(q, dtype=np.int8)
    d = np.ascontiguousarray(d, dtype=np.float32)
    s = np.ascontiguousarray(s, dtype=np.float32)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    M, K = q.shape
    out = np.empty((len(rows), N), np.float32)
    _check(_load().oracle_gemm_rows(wtype, _p(W), _p(q), _p(d), _p(s), M, N, K, _p(rows), len(rows), _p(out)))
    return out


def w8a8(W: np.ndarray, ws: np.ndarray, X: np.ndarray, xs: np.ndarray) -> np.ndarray:
    """Per-channel W8A8: bf16 bit patterns (uint16) [M, N]."""
    W = np.ascontiguousarray(W, dtype=np.int8)
    X = np.ascontiguousarray(X, dtype=np.int8)
    ws = np.ascontiguousarray(ws, dtype=np.float32)
    xs = np.ascontiguousarray(xs, dtype=np.float32)
    N, K = W.shape
    M = X.shape[0]
    out = np.empty((M, N), np.uint16)
    _check(_load().oracle_w8a8(_p(W), _p(ws), _p(X), _p(xs), M, N, K, _p(out)))
    return out


def gemm_id(wtype: int, W: np.ndarray, n_experts: int, q: np.ndarray, d: np.ndarray, s: np.ndarray,
            ids: np.ndarray, N: int) -> np.ndarray:
    """MUL_MAT_ID: f32 [M, slots, N], expert weights stacked [n_experts * N] rows."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    q = np.ascontiguousarray(q, dtype=np.int8)
    d = np.ascontiguousarray(d, dtype=np.float32)
    s = np.ascontiguousarray(s, dtype=np.float32)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    M, K = q.shape
    slots = ids.shape[1]
    out = np.zeros((M, slots, N), np.float32)
    _check(_load().oracle_gemm_id(wtype, _p(W), n_experts, _p(q), _p(d), _p(s), _p(ids), slots, M, N, K,
                                  _p(out)))
    return out


def half_to_float(h: int) -> float:
    return _load().oracle_half_to_float(h)


def float_to_bf16(f: float) -> int:
    return _load().oracle_float_to_bf16(f)
