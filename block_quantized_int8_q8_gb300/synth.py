"""Seeded synthetic inputs for block-quantized int8 MMQ.

This module only draws random fields and packs them into the library's documented byte layouts.  It
holds none of the method's arithmetic (no quantization, no dequantization, no dot product), so both
the CUDA path and the CPU oracle may consume what it produces.

Value distributions follow the workloads the MMQ pages measure on (7B-shaped Q4_0 / Q4_K prefill
GEMMs from "08 · R1 — int8 MMQ prefill GEMM", the gfx928 W8A8 shapes of "INT8 W8A8 GEMM — Prefill",
and the IQ1_M dense / MUL_MAT_ID shapes of "CUDA: add IQ1_M to MMQ"); real model weights are replaced
by uniform codes and uniform scales:

* activations x ~ N(0, 1) f32;
* f16 block scales d (and Q4_K dmin) ~ U(1e-3, 1e-2), drawn in f32 and rounded to f16 (the stored f16
  value is the scale);
* Q8_0 codes uniform in [-127, 127]; Q4_0 / Q4_K codes uniform in 0..15; Q4_K 6-bit sc, m uniform 0..63;
* IQ1_M: g uniform in {-1, 0, 1} per value, sign uniform per 8 values, 3-bit s uniform 0..7 per 16;
* Q6_K: 6-bit codes uniform 0..63, int8 sub-block scales uniform in [-128, 127] per 16 values, f16 d per
  256 values;
* W8A8: int8 weights and activations uniform in [-127, 127], f32 per-row scales ~ U(1e-3, 1e-2);
* MoE routing: each token picks `n_slots` distinct experts uniformly.

Byte layouts (per weight row, blocks back to back; rows back to back):
  Q8_0  34 B / 32 : f16 d | int8 q[32]
  Q4_0  18 B / 32 : f16 d | 16 B, byte i = code i (low nibble) | code i+16 (high nibble)
  Q4_K 144 B / 256: f16 d | f16 dmin | 12 B little-endian bit stream of 16 six-bit fields
                    (sc[0..7] then m[0..7]) | 128 B, byte 32j+i = code 64j+i (low) | code 64j+32+i (high)
  IQ1_M 76 B / 256: 64 B 2-bit codes (value i at bits 2(i%4) of byte i/4, code = g+1) | 4 B sign bits
                    (bit j: values 8j..8j+7, 1 = minus) | 6 B little-endian bit stream of 16 three-bit s
                    | f16 d
  Q6_K 224 B / 256: int8 sc[16] | f16 d | 14 B zero | four 48 B stage records j: 32 B, byte i = low
                    nibble of code 64j+i | low nibble of code 64j+32+i << 4; 16 B, byte i = high 2 bits of
                    codes 64j+i, 64j+16+i, 64j+32+i, 64j+48+i at bits 0-1, 2-3, 4-5, 6-7
  W8A8            : int8 W [N][K] then f32 ws [N]   (activations: int8 X [M][K] then f32 xs [M])
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

Q8_0, Q4_0, Q4_K, IQ1_M, W8A8, Q6_K = 0, 1, 2, 3, 4, 5
TYPE_NAMES = {Q8_0: "q8_0", Q4_0: "q4_0", Q4_K: "q4_k", IQ1_M: "iq1_m", W8A8: "w8a8", Q6_K: "q6_k"}
TYPE_IDS = {v: k for k, v in TYPE_NAMES.items()}

#: bytes per block and values per block, per weight type
BLOCK_BYTES = {Q8_0: 34, Q4_0: 18, Q4_K: 144, IQ1_M: 76, Q6_K: 224}
BLOCK_VALUES = {Q8_0: 32, Q4_0: 32, Q4_K: 256, IQ1_M: 256, Q6_K: 256}


def weight_row_bytes(wtype: int, K: int) -> int:
    if wtype == W8A8:
        return K
    return K // BLOCK_VALUES[wtype] * BLOCK_BYTES[wtype]


def rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


def activations(g: np.random.Generator, M: int, K: int) -> np.ndarray:
    return g.standard_normal((M, K), dtype=np.float32)


def f16_scales(g: np.random.Generator, shape, lo: float = 1e-3, hi: float = 1e-2) -> np.ndarray:
    return g.uniform(lo, hi, size=shape).astype(np.float32).astype(np.float16)


def _bits_le(fields: np.ndarray, width: int) -> np.ndarray:
    """Pack the low `width` bits of each uint8 field of the last axis into a little-endian bit stream."""
    f = np.ascontiguousarray(fields, dtype=np.uint8)
    bits = np.unpackbits(f[..., None], axis=-1, bitorder="little")[..., :width]
    bits = bits.reshape(*f.shape[:-1], f.shape[-1] * width)
    return np.packbits(bits, axis=-1, bitorder="little")


def _f16_bytes(h: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(h.astype(np.float16)).view(np.uint8).reshape(*h.shape, 2)


# ------------------------------------------------------------------------------------------- fields
@dataclass
class Q8_0Fields:
    d: np.ndarray      # f16 [N, K/32]
    q: np.ndarray      # int8 [N, K]


@dataclass
class Q4_0Fields:
    d: np.ndarray      # f16 [N, K/32]
    code: np.ndarray   # uint8 [N, K] in 0..15


@dataclass
class Q4_KFields:
    d: np.ndarray      # f16 [N, K/256]
    dmin: np.ndarray   # f16 [N, K/256]
    sc: np.ndarray     # uint8 [N, K/32] in 0..63
    m: np.ndarray      # uint8 [N, K/32] in 0..63
    code: np.ndarray   # uint8 [N, K] in 0..15


@dataclass
class IQ1_MFields:
    d: np.ndarray      # f16 [N, K/256]
    s: np.ndarray      # uint8 [N, K/16] in 0..7
    neg: np.ndarray    # uint8 [N, K/8] in {0, 1}; 1 = delta -1/8
    g: np.ndarray      # int8 [N, K] in {-1, 0, 1}


@dataclass
class Q6_KFields:
    d: np.ndarray      # f16 [N, K/256]
    sc: np.ndarray     # int8 [N, K/16]
    code: np.ndarray   # uint8 [N, K] in 0..63


@dataclass
class W8A8Fields:
    W: np.ndarray      # int8 [N, K]
    ws: np.ndarray     # f32 [N]


def draw_fields(g: np.random.Generator, wtype: int, N: int, K: int):
    if wtype == Q8_0:
        return Q8_0Fields(d=f16_scales(g, (N, K // 32)),
                          q=g.integers(-127, 128, size=(N, K), dtype=np.int16).astype(np.int8))
    if wtype == Q4_0:
        return Q4_0Fields(d=f16_scales(g, (N, K // 32)), code=g.integers(0, 16, size=(N, K), dtype=np.uint8))
    if wtype == Q4_K:
        return Q4_KFields(d=f16_scales(g, (N, K // 256)), dmin=f16_scales(g, (N, K // 256)),
                          sc=g.integers(0, 64, size=(N, K // 32), dtype=np.uint8),
                          m=g.integers(0, 64, size=(N, K // 32), dtype=np.uint8),
                          code=g.integers(0, 16, size=(N, K), dtype=np.uint8))
    if wtype == IQ1_M:
        return IQ1_MFields(d=f16_scales(g, (N, K // 256)), s=g.integers(0, 8, size=(N, K // 16), dtype=np.uint8),
                           neg=g.integers(0, 2, size=(N, K // 8), dtype=np.uint8),
                           g=(g.integers(0, 3, size=(N, K), dtype=np.int8) - 1).astype(np.int8))
    if wtype == Q6_K:
        return Q6_KFields(d=f16_scales(g, (N, K // 256)),
                          sc=g.integers(-128, 128, size=(N, K // 16), dtype=np.int16).astype(np.int8),
                          code=g.integers(0, 64, size=(N, K), dtype=np.uint8))
    if wtype == W8A8:
        return W8A8Fields(W=g.integers(-127, 128, size=(N, K), dtype=np.int16).astype(np.int8),
                          ws=g.uniform(1e-3, 1e-2, size=N).astype(np.float32))
    raise ValueError(f"unknown weight type {wtype}")


# ------------------------------------------------------------------------------------------- packing
def pack(wtype: int, f) -> np.ndarray:
    """Pack drawn fields into the raw weight bytes: uint8 [N, row_bytes] (W8A8: flat buffer)."""
    if wtype == Q8_0:
        N, K = f.q.shape
        blk = np.empty((N, K // 32, 34), np.uint8)
        blk[..., 0:2] = _f16_bytes(f.d)
        blk[..., 2:34] = f.q.reshape(N, K // 32, 32).view(np.uint8)
        return blk.reshape(N, -1)
    if wtype == Q4_0:
        N, K = f.code.shape
        c = f.code.reshape(N, K // 32, 32)
        blk = np.empty((N, K // 32, 18), np.uint8)
        blk[..., 0:2] = _f16_bytes(f.d)
        blk[..., 2:18] = c[..., :16] | (c[..., 16:] << 4)
        return blk.reshape(N, -1)
    if wtype == Q4_K:
        N, K = f.code.shape
        nsb = K // 256
        blk = np.empty((N, nsb, 144), np.uint8)
        blk[..., 0:2] = _f16_bytes(f.d)
        blk[..., 2:4] = _f16_bytes(f.dmin)
        fields = np.concatenate([f.sc.reshape(N, nsb, 8), f.m.reshape(N, nsb, 8)], axis=-1)
        blk[..., 4:16] = _bits_le(fields, 6)
        c = f.code.reshape(N, nsb, 4, 64)
        blk[..., 16:144] = (c[..., :32] | (c[..., 32:] << 4)).reshape(N, nsb, 128)
        return blk.reshape(N, -1)
    if wtype == IQ1_M:
        N, K = f.g.shape
        nsb = K // 256
        blk = np.empty((N, nsb, 76), np.uint8)
        code = (f.g.astype(np.int16) + 1).astype(np.uint8).reshape(N, nsb, 64, 4)
        blk[..., 0:64] = code[..., 0] | (code[..., 1] << 2) | (code[..., 2] << 4) | (code[..., 3] << 6)
        blk[..., 64:68] = np.packbits(f.neg.reshape(N, nsb, 32), axis=-1, bitorder="little")
        blk[..., 68:74] = _bits_le(f.s.reshape(N, nsb, 16), 3)
        blk[..., 74:76] = _f16_bytes(f.d)
        return blk.reshape(N, -1)
    if wtype == Q6_K:
        N, K = f.code.shape
        nsb = K // 256
        blk = np.zeros((N, nsb, 224), np.uint8)
        blk[..., 0:16] = f.sc.reshape(N, nsb, 16).view(np.uint8)
        blk[..., 16:18] = _f16_bytes(f.d)
        c = f.code.reshape(N, nsb, 4, 64)
        lo, hi = c & 15, c >> 4
        rec = np.empty((N, nsb, 4, 48), np.uint8)
        rec[..., 0:32] = lo[..., :32] | (lo[..., 32:] << 4)
        rec[..., 32:48] = hi[..., 0:16] | (hi[..., 16:32] << 2) | (hi[..., 32:48] << 4) | (hi[..., 48:64] << 6)
        blk[..., 32:224] = rec.reshape(N, nsb, 192)
        return blk.reshape(N, -1)
    if wtype == W8A8:
        return np.concatenate([f.W.reshape(-1).view(np.uint8), f.ws.view(np.uint8)])
    raise ValueError(f"unknown weight type {wtype}")


def pack_w8a8_acts(X: np.ndarray, xs: np.ndarray) -> np.ndarray:
    """int8 X [M][K] followed by f32 xs [M], as one byte buffer."""
    return np.concatenate([np.ascontiguousarray(X).reshape(-1).view(np.uint8),
                           np.ascontiguousarray(xs, dtype=np.float32).view(np.uint8)])


def w8a8_acts(g: np.random.Generator, M: int, K: int):
    X = g.integers(-127, 128, size=(M, K), dtype=np.int16).astype(np.int8)
    xs = g.uniform(1e-3, 1e-2, size=M).astype(np.float32)
    return X, xs


def route(g: np.random.Generator, M: int, n_experts: int, n_slots: int) -> np.ndarray:
    """int32 [M, n_slots]: for each token, n_slots distinct experts drawn uniformly."""
    ids = np.empty((M, n_slots), np.int32)
    for t in range(M):
        ids[t] = g.choice(n_experts, n_slots, replace=False)
    return ids


# ------------------------------------------------------------------------------------------- workloads
#: The measured workloads: (name, weight type, M tokens, N weight rows, K, seed, experts, slots)
WORKLOADS = {
    "q8_0_tiny":      dict(wtype=Q8_0, M=64, N=256, K=1024, seed=1001),
    "q4_0_7b":        dict(wtype=Q4_0, M=2048, N=4096, K=4096, seed=1002),
    "q4_k_ffn_up":    dict(wtype=Q4_K, M=2048, N=11008, K=4096, seed=1003),
    "w8a8_m3072":     dict(wtype=W8A8, M=3072, N=1536, K=4096, seed=1004),
    "w8a8_m4096":     dict(wtype=W8A8, M=4096, N=1536, K=4096, seed=1014),
    "iq1_m_moe":      dict(wtype=IQ1_M, M=512, N=1536, K=4096, seed=1005, experts=64, slots=8),
    "iq1_m_dense":    dict(wtype=IQ1_M, M=512, N=4096, K=4096, seed=1006),
    "q6_k_ffn_down":  dict(wtype=Q6_K, M=2048, N=4096, K=11008, seed=1007),
}


@dataclass
class Problem:
    wtype: int
    M: int
    N: int
    K: int
    x: np.ndarray | None          # f32 [M, K] (block types)
    fields: object                # weight fields (one expert: fields of the stacked [E*N, K] matrix)
    W: np.ndarray                 # packed weight bytes
    X: np.ndarray | None = None   # W8A8 int8 activations
    xs: np.ndarray | None = None  # W8A8 per-token scales
    ids: np.ndarray | None = None # MoE routing [M, slots]
    experts: int = 0


def make_problem(wtype: int, M: int, N: int, K: int, seed: int, experts: int = 0, slots: int = 0) -> Problem:
    g = rng(seed)
    rows = N * experts if experts else N
    fields = draw_fields(g, wtype, rows, K)
    W = pack(wtype, fields)
    if wtype == W8A8:
        X, xs = w8a8_acts(g, M, K)
        return Problem(wtype, M, N, K, None, fields, W, X=X, xs=xs)
    x = activations(g, M, K)
    ids = route(g, M, experts, slots) if experts else None
    return Problem(wtype, M, N, K, x, fields, W, ids=ids, experts=experts)


def workload(name: str) -> Problem:
    w = dict(WORKLOADS[name])
    return make_problem(w.pop("wtype"), w.pop("M"), w.pop("N"), w.pop("K"), w.pop("seed"),
                        w.pop("experts", 0), w.pop("slots", 0))
