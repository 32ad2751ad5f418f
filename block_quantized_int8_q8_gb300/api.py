"""Thin Python binding of libmmq_gb300.so (argument marshalling only).

Every function forwards device pointers, sizes and the current CUDA stream to the C ABI declared in
include/mmq.h; all arithmetic runs in the library's sm_103a kernels.  PyTorch is used only for device
memory and streams.  If the library is missing or fails to load, every call raises: there is no CPU
fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

Q8_0, Q4_0, Q4_K, IQ1_M, W8A8, Q6_K = 0, 1, 2, 3, 4, 5
DEVERR_TIMEOUT, DEVERR_EXPERT_ID, DEVERR_DUP_EXPERT = 1, 2, 4

#: every symbol include/mmq.h declares
EXPORTS = ("mmq_status_string", "mmq_last_cuda_error", "mmq_q8_1_bytes", "mmq_weight_bytes", "mmq_w8a8_act_bytes", "mmq_quantize_q8_1",
           "mmq_gemm", "mmq_gemm_id_workspace_bytes", "mmq_gemm_id", "mmq_gemm_debug_partials",
           "mmq_gemm_debug_block_sums", "mmq_selftest_bounded_wait",
           "mmq_read_device_errors", "mmq_gemm_id_noalloc", "mmq_q8_1_prepare")
NOALLOC_SCRATCH_BYTES = 1 << 20

_lib = None


class MMQError(RuntimeError):
    pass


def library_path() -> str:
    return _build.LIB


def load():
    """Load the CUDA library (it must have been built by __graft_entry__.build() or _build.build())."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise MMQError(f"CUDA library not built: {path} is missing (run __graft_entry__.build())")
    lib = ctypes.CDLL(path)
    P, I64, I, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    lib.mmq_status_string.argtypes = [I]
    lib.mmq_status_string.restype = ctypes.c_char_p
    lib.mmq_last_cuda_error.argtypes = []
    lib.mmq_last_cuda_error.restype = ctypes.c_char_p
    lib.mmq_q8_1_bytes.argtypes = [I64, I64]
    lib.mmq_q8_1_bytes.restype = SZ
    lib.mmq_weight_bytes.argtypes = [I, I64, I64]
    lib.mmq_weight_bytes.restype = SZ
    lib.mmq_w8a8_act_bytes.argtypes = [I64, I64]
    lib.mmq_w8a8_act_bytes.restype = SZ
    lib.mmq_quantize_q8_1.argtypes = [P, I64, I64, P, P]
    lib.mmq_q8_1_prepare.argtypes = [P, I64, I64, P]
    lib.mmq_q8_1_prepare.restype = I
    lib.mmq_quantize_q8_1.restype = I
    lib.mmq_gemm.argtypes = [I, P, P, P, I64, I64, I64, P]
    lib.mmq_gemm.restype = I
    lib.mmq_gemm_id_workspace_bytes.argtypes = [I64, I64, I, I]
    lib.mmq_gemm_id_workspace_bytes.restype = SZ
    lib.mmq_gemm_id.argtypes = [I, P, I, P, P, I, P, I64, I64, I64, P, SZ, P]
    lib.mmq_gemm_id.restype = I
    lib.mmq_gemm_debug_partials.argtypes = [I, P, P, P, I64, I64, I64, P]
    lib.mmq_gemm_debug_partials.restype = I
    lib.mmq_gemm_debug_block_sums.argtypes = [I, P, P, P, I64, I64, I64, P]
    lib.mmq_gemm_debug_block_sums.restype = I
    lib.mmq_selftest_bounded_wait.argtypes = [P, P]
    lib.mmq_selftest_bounded_wait.restype = I
    lib.mmq_gemm_id_noalloc.argtypes = [I, P, I, P, P, I, P, I64, I64, I64, P]
    lib.mmq_gemm_id_noalloc.restype = I
    lib.mmq_read_device_errors.argtypes = [ctypes.POINTER(ctypes.c_uint), P]
    lib.mmq_read_device_errors.restype = I
    _lib = lib
    return lib


def _check(rc: int, what: str):
    if rc != 0:
        msg = load().mmq_status_string(rc).decode()
        if rc == 5:
            msg += "; " + load().mmq_last_cuda_error().decode()
        raise MMQError(f"{what}: status {rc} ({msg})")


def _stream(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ptr(t: torch.Tensor | None) -> int | None:
    if t is None:
        return None
    if not t.is_cuda or not t.is_contiguous():
        raise MMQError("expected a contiguous CUDA tensor")
    return t.data_ptr()


# ------------------------------------------------------------------------------------------ sizes / layouts
def q8_1_bytes(M: int, K: int) -> int:
    return int(load().mmq_q8_1_bytes(M, K))


def weight_bytes(wtype: int, N: int, K: int) -> int:
    return int(load().mmq_weight_bytes(wtype, N, K))


def w8a8_act_bytes(M: int, K: int) -> int:
    return int(load().mmq_w8a8_act_bytes(M, K))


def gemm_id_workspace_bytes(M: int, K: int, slots: int, experts: int) -> int:
    return int(load().mmq_gemm_id_workspace_bytes(M, K, slots, experts))


def q8_1_offsets(M: int, K: int) -> dict:
    """Byte offsets of the sections of a q8_1 buffer (layout in include/mmq.h)."""
    kb = K // 32
    Mp = (M + 3) // 4 * 4
    ds = M * K
    h = (M * K + M * kb * 8 + 255) // 256 * 256
    dT = (h + 2 * M * K + 255) // 256 * 256
    return {"q": 0, "ds": ds, "h": h, "dT": dT, "sT": dT + Mp * kb * 4, "Mp": Mp}


def q8_1_views(buf: torch.Tensor, M: int, K: int):
    """(q int8 [M, K], ds f32 [M, K/32, 2]) views of a q8_1 buffer's block sections."""
    o = q8_1_offsets(M, K)
    q = buf[: M * K].view(torch.int8).view(M, K)
    ds = buf[o["ds"]: o["ds"] + M * (K // 32) * 8].view(torch.float32).view(M, K // 32, 2)
    return q, ds


def q8_1_shadow_views(buf: torch.Tensor, M: int, K: int):
    """(h fp16 [M, K], dT f32 [K/32, M], sT f32 [K/32, M]) views of a q8_1 buffer's derived sections."""
    o = q8_1_offsets(M, K)
    kb, Mp = K // 32, o["Mp"]
    h = buf[o["h"]: o["h"] + 2 * M * K].view(torch.float16).view(M, K)
    dT = buf[o["dT"]: o["dT"] + Mp * kb * 4].view(torch.float32).view(kb, Mp)[:, :M]
    sT = buf[o["sT"]: o["sT"] + Mp * kb * 4].view(torch.float32).view(kb, Mp)[:, :M]
    return h, dT, sT


def q8_1_prepare(buf: torch.Tensor, M: int, K: int, stream=None) -> torch.Tensor:
    """Fill the derived sections of a q8_1 buffer from its q and ds sections (mmq_q8_1_prepare)."""
    _check(load().mmq_q8_1_prepare(_ptr(buf), M, K, _stream(stream)), "mmq_q8_1_prepare")
    return buf


def pack_q8_1(q: torch.Tensor, d: torch.Tensor, s: torch.Tensor, device="cuda") -> torch.Tensor:
    """A complete q8_1 buffer on `device` from codes [M, K], scales d and block sums s [M, K/32]."""
    M, K = q.shape
    buf = torch.zeros(q8_1_bytes(M, K), dtype=torch.uint8, device=device)
    qv, dsv = q8_1_views(buf, M, K)
    qv.copy_(q.to(device))
    dsv.copy_(torch.stack([d.float(), s.float()], dim=-1).to(device))
    return q8_1_prepare(buf, M, K)


# ------------------------------------------------------------------------------------------ entry points
def quantize_q8_1(x: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """x f32 [M, K] on the GPU -> q8_1 byte buffer (mmq_quantize_q8_1)."""
    M, K = x.shape
    if out is None:
        out = torch.empty(q8_1_bytes(M, K), dtype=torch.uint8, device=x.device)
    _check(load().mmq_quantize_q8_1(_ptr(x), M, K, _ptr(out), _stream(stream)), "mmq_quantize_q8_1")
    return out


def gemm(wtype: int, W: torch.Tensor, Xq: torch.Tensor, M: int, N: int, K: int, out: torch.Tensor | None = None,
         stream=None) -> torch.Tensor:
    """Dense MMQ product (mmq_gemm): f32 [M, N] (bf16 for W8A8)."""
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16 if wtype == W8A8 else torch.float32, device=W.device)
    _check(load().mmq_gemm(wtype, _ptr(W), _ptr(Xq), _ptr(out), M, N, K, _stream(stream)), "mmq_gemm")
    return out


def gemm_debug_partials(wtype: int, W: torch.Tensor, Xq: torch.Tensor, M: int, N: int, K: int,
                        stream=None) -> torch.Tensor:
    """Exact per-group int32 dots (mmq_gemm_debug_partials): [M, N, K/G]."""
    G = 16 if wtype == IQ1_M else 32
    out = torch.empty((M, N, K // G), dtype=torch.int32, device=W.device)
    _check(load().mmq_gemm_debug_partials(wtype, _ptr(W), _ptr(Xq), _ptr(out), M, N, K, _stream(stream)),
           "mmq_gemm_debug_partials")
    return out


def gemm_debug_block_sums(wtype: int, W: torch.Tensor, Xq: torch.Tensor, M: int, N: int, K: int,
                          stream=None) -> torch.Tensor:
    """The TMA-fed kernel's exact 32-k block accumulators (mmq_gemm_debug_block_sums): int32 [M, N, K/32]."""
    out = torch.empty((M, N, K // 32), dtype=torch.int32, device=W.device)
    _check(load().mmq_gemm_debug_block_sums(wtype, _ptr(W), _ptr(Xq), _ptr(out), M, N, K, _stream(stream)),
           "mmq_gemm_debug_block_sums")
    return out


def gemm_id(wtype: int, W: torch.Tensor, n_experts: int, Xq: torch.Tensor, ids: torch.Tensor, M: int, N: int,
            K: int, out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
            stream=None) -> torch.Tensor:
    """MoE MUL_MAT_ID (mmq_gemm_id): f32 [M, slots, N]."""
    slots = ids.shape[1]
    if out is None:
        out = torch.empty((M, slots, N), dtype=torch.float32, device=W.device)
    need = gemm_id_workspace_bytes(M, K, slots, n_experts)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=W.device)
    _check(load().mmq_gemm_id(wtype, _ptr(W), n_experts, _ptr(Xq), _ptr(ids), slots, _ptr(out), M, N, K,
                              _ptr(workspace), workspace.numel(), _stream(stream)), "mmq_gemm_id")
    return out


def gemm_id_noalloc(wtype: int, W: torch.Tensor, n_experts: int, Xq: torch.Tensor, ids: torch.Tensor, M: int,
                    N: int, K: int, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """MoE MUL_MAT_ID without a workspace (mmq_gemm_id_noalloc): the routing lists live in the
    library's static device scratch array, for callers that cannot allocate device memory."""
    slots = ids.shape[1]
    if out is None:
        out = torch.empty((M, slots, N), dtype=torch.float32, device=W.device)
    _check(load().mmq_gemm_id_noalloc(wtype, _ptr(W), n_experts, _ptr(Xq), _ptr(ids), slots, _ptr(out), M, N, K,
                                      _stream(stream)), "mmq_gemm_id_noalloc")
    return out


def read_device_errors(stream=None) -> int:
    """Synchronise and return (and clear) the device error bits (DEVERR_*)."""
    bits = ctypes.c_uint(0)
    _check(load().mmq_read_device_errors(ctypes.byref(bits), _stream(stream)), "mmq_read_device_errors")
    return bits.value


def selftest_bounded_wait(device="cuda", stream=None) -> list[int]:
    """mmq_selftest_bounded_wait: [completed, abort_flag] of the polling and of the sleeping wait."""
    res = torch.full((4,), -1, dtype=torch.int32, device=device)
    _check(load().mmq_selftest_bounded_wait(_ptr(res), _stream(stream)), "mmq_selftest_bounded_wait")
    return res.cpu().tolist()
