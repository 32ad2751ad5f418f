"""The boundary as a C program sees it (no GPU needed): include/mmq.h compiles as strict C11 and as C++,
and a C program linked against the built library gets the documented sizes and synchronous status codes
(every call here returns before any CUDA call)."""
import os
import shutil
import subprocess

import pytest

from block_quantized_int8_q8_gb300 import _build, api

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")

C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "mmq.h"

int main(void) {
    static unsigned char buf[4096] __attribute__((aligned(16)));
    void* p = buf;
    printf("q8_1_bytes %zu\n", mmq_q8_1_bytes(4, 64));
    printf("q8_1_bytes_bad %zu\n", mmq_q8_1_bytes(4, 96));
    printf("weight_bytes_q4_0 %zu\n", mmq_weight_bytes(MMQ_Q4_0, 8, 256));
    printf("weight_bytes_w8a8 %zu\n", mmq_weight_bytes(MMQ_W8A8, 8, 64));
    printf("w8a8_act_bytes %zu\n", mmq_w8a8_act_bytes(3, 64));
    printf("gemm_null %d\n", (int)mmq_gemm(MMQ_Q4_0, NULL, NULL, NULL, 4, 8, 256, NULL));
    printf("gemm_shape %d\n", (int)mmq_gemm(MMQ_Q4_0, p, p, p, 4, 8, 96, NULL));
    printf("gemm_align %d\n", (int)mmq_gemm(MMQ_Q4_0, buf + 8, p, p, 4, 8, 256, NULL));
    printf("gemm_empty %d\n", (int)mmq_gemm(MMQ_Q4_0, NULL, NULL, NULL, 0, 8, 256, NULL));
    printf("gemm_id_ws %d\n", (int)mmq_gemm_id(MMQ_IQ1_M, p, 4, p, (const int32_t*)p, 2, (float*)p, 16, 128,
                                               256, NULL, 0, NULL));
    printf("noalloc_q6k %d\n", (int)mmq_gemm_id_noalloc(MMQ_Q6_K, p, 4, p, (const int32_t*)p, 2, (float*)p,
                                                        16, 128, 256, NULL));
    printf("quantize_shape %d\n", (int)mmq_quantize_q8_1((const float*)p, 4, 33, p, NULL));
    printf("status_ok %s\n", mmq_status_string(MMQ_OK));
    printf("last_cuda_error_len %zu\n", strlen(mmq_last_cuda_error()));
    return 0;
}
"""


@pytest.fixture(scope="module")
def lib_dir():
    _build.build()
    return os.path.dirname(_build.LIB)


def test_header_is_strict_c11_and_cplusplus(tmp_path):
    for cc, std, ext in (("gcc", "-std=c11", "c"), ("g++", "-std=c++17", "cpp")):
        if shutil.which(cc) is None:
            pytest.skip(f"{cc} not available")
        src = tmp_path / f"h.{ext}"
        src.write_text('#include "mmq.h"\nint f(void) { return (int)MMQ_OK + (int)MMQ_Q6_K; }\n')
        subprocess.run([cc, std, "-Wall", "-Wextra", "-Werror", "-pedantic", "-fsyntax-only", f"-I{INCLUDE}",
                        str(src)], check=True)


def test_c_program_gets_documented_sizes_and_statuses(tmp_path, lib_dir):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = tmp_path / "boundary.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "boundary"
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", f"-I{INCLUDE}", str(src), "-o", str(exe),
                    f"-L{lib_dir}", "-lmmq_gb300", f"-Wl,-rpath,{lib_dir}"], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    got = dict(line.split(" ", 1) for line in out.strip().splitlines())
    assert int(got["q8_1_bytes"]) == api.q8_1_bytes(4, 64) > 0
    assert int(got["q8_1_bytes_bad"]) == 0
    assert int(got["weight_bytes_q4_0"]) == 8 * (256 // 32) * 18
    assert int(got["weight_bytes_w8a8"]) == 8 * 64 + 4 * 8
    assert int(got["w8a8_act_bytes"]) == 3 * 64 + 4 * 3
    assert int(got["gemm_null"]) == 1          # MMQ_ERR_INVALID_ARG
    assert int(got["gemm_shape"]) == 2         # MMQ_ERR_SHAPE
    assert int(got["gemm_align"]) == 3         # MMQ_ERR_ALIGN
    assert int(got["gemm_empty"]) == 0         # M == 0: a no-op
    assert int(got["gemm_id_ws"]) == 6         # MMQ_ERR_WORKSPACE
    assert int(got["noalloc_q6k"]) == 4        # MMQ_ERR_UNSUPPORTED
    assert int(got["quantize_shape"]) == 2
    assert got["status_ok"] and int(got["last_cuda_error_len"]) == 0
