"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the same seeded inputs.

Bars (BASELINE the benchmark spec): q8_1 codes, scales and block sums bit-exact; per-group integer partials
bit-exact; W8A8 bf16 outputs bit-exact; f32 outputs within max|diff| <= 1e-3 * max|oracle output|.
Shapes span several 128x128 tiles with ragged M and N tails, plus the degenerate sizes.
"""
import numpy as np
import pytest
import torch

import oracle
from block_quantized_int8_q8_gb300 import api, synth

pytestmark = pytest.mark.gpu
TOL = 1e-3
BLOCK_TYPES = [synth.Q8_0, synth.Q4_0, synth.Q4_K, synth.IQ1_M, synth.Q6_K]
PARTIAL_TYPES = [synth.Q8_0, synth.Q4_0, synth.Q4_K, synth.IQ1_M, synth.W8A8]   # the general kernel's types
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    api.load()
    yield
    assert api.read_device_errors() == 0


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _rel_err(got, ref):
    scale = np.abs(ref).max()
    return float(np.abs(got.astype(np.float64) - ref).max() / (scale if scale > 0 else 1.0))


def _oracle_acts(pb):
    q, d, s = oracle.quantize_q8_1(pb.x)
    return q, d, s, api.pack_q8_1(torch.from_numpy(q), torch.from_numpy(d), torch.from_numpy(s)).to(DEV)


# ---------------------------------------------------------------------------------------- quantizer
@pytest.mark.parametrize("M,K", [(1, 64), (3, 64), (37, 4096), (257, 1024), (2048, 4096)])
def test_quantizer_bit_exact(M, K):
    g = np.random.default_rng(M * 7 + K)
    x = g.standard_normal((M, K), dtype=np.float32)
    x[0, :32] = 0.0                                      # an all-zero block
    if K >= 64:
        x[0, 32:64] = 0.0
        x[0, 32] = 127.0
        x[0, 33:41] = [2.5, 3.5, -2.5, -0.5, 0.5, 1.5, 126.5, -127.0]   # exact ties at d = 1
    q, d, s = oracle.quantize_q8_1(x)
    buf = api.quantize_q8_1(_dev(x))
    torch.cuda.synchronize()
    qg, dsg = api.q8_1_views(buf, M, K)
    assert np.array_equal(qg.cpu().numpy(), q)
    assert np.array_equal(dsg[..., 0].cpu().numpy().view(np.uint32), d.view(np.uint32))
    assert np.array_equal(dsg[..., 1].cpu().numpy().view(np.uint32), s.view(np.uint32))
    _check_shadow(buf, q, d, s, M, K)


def _check_shadow(buf, q, d, s, M, K):
    # derived sections: fp16 codes equal the int8 codes; the block-major copies are d and s transposed,
    # bit for bit
    h, dT, sT = api.q8_1_shadow_views(buf, M, K)
    assert np.array_equal(h.float().cpu().numpy(), q.astype(np.float32))
    assert np.array_equal(dT.cpu().numpy().view(np.uint32), np.ascontiguousarray(d.T).view(np.uint32))
    assert np.array_equal(sT.cpu().numpy().view(np.uint32), np.ascontiguousarray(s.T).view(np.uint32))


def test_prepare_rebuilds_the_quantizer_shadow():
    M, K = 130, 1024
    x = np.random.default_rng(5).standard_normal((M, K), dtype=np.float32)
    buf = api.quantize_q8_1(_dev(x))
    q, d, s = oracle.quantize_q8_1(x)
    packed = api.pack_q8_1(torch.from_numpy(q), torch.from_numpy(d), torch.from_numpy(s))
    torch.cuda.synchronize()
    o = api.q8_1_offsets(M, K)
    assert torch.equal(buf[o["h"]:], packed[o["h"]:])
    _check_shadow(packed, q, d, s, M, K)


def test_quantizer_codes_next_to_rounding_boundaries_bit_exact():
    # every value an f32 neighbour (0..3 ulps either way) of (k + 1/2) * d for its block's own d, so the
    # quotient x/d sits on or right next to a half-integer: the rounded code must still be that of the
    # correctly rounded quotient, ties to even; the fp16 shadow must hold the codes' exact bits (+0 for 0)
    g = np.random.default_rng(29)
    M, K = 64, 1024
    amax = (g.uniform(0.5, 2.0, size=(M, K // 32)) * 10.0 ** g.integers(-20, 20, size=(M, 1))).astype(np.float32)
    d = (amax / np.float32(127)).astype(np.float32)
    k = g.integers(-127, 127, size=(M, K // 32, 32)).astype(np.float32)
    x = ((k + np.float32(0.5)) * d[..., None]).astype(np.float32)
    steps = g.integers(-3, 4, size=x.shape)
    for _ in range(3):
        x = np.where(steps > 0, np.nextafter(x, np.float32(np.inf)), np.where(steps < 0, np.nextafter(x, np.float32(-np.inf)), x))
        steps = steps - np.sign(steps)
    x[..., 0] = amax                                   # the block's amax, so its d is the one above
    x = x.reshape(M, K).astype(np.float32)
    q, dq, s = oracle.quantize_q8_1(x)
    assert np.array_equal(dq.view(np.uint32), d.view(np.uint32))
    buf = api.quantize_q8_1(_dev(x))
    qg, dsg = api.q8_1_views(buf, M, K)
    assert np.array_equal(qg.cpu().numpy(), q)
    assert np.array_equal(dsg[..., 1].cpu().numpy().view(np.uint32), s.view(np.uint32))
    h, _, _ = api.q8_1_shadow_views(buf, M, K)
    assert np.array_equal(h.cpu().numpy().view(np.uint16), q.astype(np.float16).view(np.uint16))


def test_quantizer_subnormal_scales_bit_exact():
    # blocks whose amax is so small that d = amax/127 is subnormal (or zero): the codes then come from the
    # exact quotient and the clamp to [-127, 127] can act; codes, d and s must still equal the oracle's
    g = np.random.default_rng(17)
    M, K = 16, 512
    mags = np.float32(10.0) ** g.integers(-44, -34, size=(M, K // 32, 1)).astype(np.float32)
    x = (g.uniform(-1.0, 1.0, size=(M, K // 32, 32)).astype(np.float32) * mags).astype(np.float32)
    x[0, 0] = np.float32(1e-45)                       # the smallest subnormal, repeated
    x[0, 1] = 0.0
    x = x.reshape(M, K)
    q, d, s = oracle.quantize_q8_1(x)
    assert (d[d > 0] < np.float32(1.17549435e-38)).any()
    qg, dsg = api.q8_1_views(api.quantize_q8_1(_dev(x)), M, K)
    assert np.array_equal(qg.cpu().numpy(), q)
    assert np.array_equal(dsg[..., 0].cpu().numpy().view(np.uint32), d.view(np.uint32))
    assert np.array_equal(dsg[..., 1].cpu().numpy().view(np.uint32), s.view(np.uint32))


def test_quantizer_extreme_scales_bit_exact():
    g = np.random.default_rng(3)
    x = (g.standard_normal((64, 512)) * 10.0 ** g.integers(-30, 30, size=(64, 1))).astype(np.float32)
    q, d, s = oracle.quantize_q8_1(x)
    qg, dsg = api.q8_1_views(api.quantize_q8_1(_dev(x)), 64, 512)
    assert np.array_equal(qg.cpu().numpy(), q)
    assert np.array_equal(dsg[..., 0].cpu().numpy().view(np.uint32), d.view(np.uint32))
    assert np.array_equal(dsg[..., 1].cpu().numpy().view(np.uint32), s.view(np.uint32))


# ---------------------------------------------------------------------------------------- block GEMM
SHAPES = [(1, 1, 256), (5, 130, 256), (130, 257, 512), (200, 300, 1024), (256, 384, 2048), (64, 128, 5376),
          (20, 1, 1024), (9, 3, 256),           # tile path (M > 8) with one and three weight rows
          (64, 300, 1024), (65, 300, 1024)]     # either side of the four-converter kernel for <= 64 tokens


@pytest.mark.parametrize("wtype", BLOCK_TYPES)
@pytest.mark.parametrize("shape", SHAPES)
def test_block_gemm_matches_oracle(wtype, shape):
    M, N, K = shape
    pb = synth.make_problem(wtype, M, N, K, seed=11 + M + N + K + wtype)
    q, d, s, xq = _oracle_acts(pb)
    out = api.gemm(wtype, _dev(pb.W.reshape(-1)), xq, M, N, K).cpu().numpy()
    ref = oracle.gemm(wtype, pb.W, q, d, s, N)
    assert _rel_err(out, ref) <= TOL


@pytest.mark.parametrize("wtype", BLOCK_TYPES)
@pytest.mark.parametrize("shape", [(1, 1, 256), (3, 130, 1280), (8, 257, 4096), (5, 64, 768), (4, 200, 11008),
                                   (2, 40001, 256), (7, 3, 512)])
def test_few_token_path_bit_exact(wtype, shape):
    # M <= 8 runs on the matrix-vector kernel, which forms every block term and sum in the
    # blockwise definition's order: the f32 output equals the oracle's bit for bit (K = 1280, 768 and
    # 11008 leave a partial chunk of 32-value blocks; 40001 rows outnumber one pass of the grid)
    M, N, K = shape
    pb = synth.make_problem(wtype, M, N, K, seed=13 + M + N + wtype)
    q, d, s, xq = _oracle_acts(pb)
    out = api.gemm(wtype, _dev(pb.W.reshape(-1)), xq, M, N, K).cpu().numpy()
    ref = oracle.gemm(wtype, pb.W, q, d, s, N)
    assert np.array_equal(out.view(np.uint32), ref.view(np.uint32)), np.abs(out - ref).max()


def _extreme_fields(wtype, N, K, g):
    """Weight fields at the ends of their ranges, alternating sign by row and by value."""
    f = synth.draw_fields(g, wtype, N, K)
    alt = (np.arange(N)[:, None] + np.arange(K)[None, :]) % 2 == 0
    if wtype == synth.Q8_0:
        f.q[...] = np.where(alt, 127, -127).astype(np.int8)
    elif wtype == synth.Q4_0:
        f.code[...] = np.where(alt, 0, 15).astype(np.uint8)         # -8 and +7
    elif wtype == synth.Q4_K:
        f.code[...] = 15
        f.sc[...] = 63
        f.m[...] = 63
    elif wtype == synth.IQ1_M:
        f.g[...] = np.where(alt, 1, -1).astype(np.int8)
        f.s[...] = 7
    elif wtype == synth.Q6_K:
        f.code[...] = np.where(alt, 0, 63).astype(np.uint8)         # -32 and +31
        f.sc[...] = np.where(np.arange(K // 16)[None, :] % 2 == 0, -128, 127).astype(np.int8)
    return f


@pytest.mark.parametrize("wtype", [synth.Q4_0, synth.Q6_K])
def test_few_token_chain_reads_what_the_kernels_before_it_wrote(wtype):
    # the quantizer and the matrix-vector kernel start early as programmatic dependents; each must still
    # see the previous kernel's writes: layer after layer on one stream, overwrite the weights and the
    # activations in place with a device copy right before each quantize -> GEMV pair, no host sync
    # between layers, and every layer's output must equal the oracle's for that layer's inputs
    M, N, K = 3, 520, 2048
    layers = [synth.make_problem(wtype, M, N, K, seed=300 + i + wtype) for i in range(4)]
    src_w = [_dev(pb.W.reshape(-1)) for pb in layers]
    src_x = [_dev(pb.x) for pb in layers]
    W = torch.empty_like(src_w[0])
    x = torch.empty_like(src_x[0])
    xq = torch.empty(api.q8_1_bytes(M, K), dtype=torch.uint8, device=DEV)
    outs = [torch.empty((M, N), dtype=torch.float32, device=DEV) for _ in layers]
    for i in range(len(layers)):
        W.copy_(src_w[i])
        x.copy_(src_x[i])
        api.quantize_q8_1(x, out=xq)
        api.gemm(wtype, W, xq, M, N, K, out=outs[i])
    torch.cuda.synchronize()
    for pb, o in zip(layers, outs):
        q, d, s = oracle.quantize_q8_1(pb.x)
        ref = oracle.gemm(wtype, pb.W, q, d, s, N)
        assert np.array_equal(o.cpu().numpy().view(np.uint32), ref.view(np.uint32))


def test_few_token_layers_captured_in_one_cuda_graph():
    # decode as a CUDA graph: three layers of quantize -> GEMV captured once (programmatic-dependent
    # launches become graph edges), the input rewritten between replays; each replay must reproduce the
    # oracle for that input, layer after layer (layer i+1's activations are layer i's output columns)
    wtype, M, N, K = synth.Q4_0, 2, 1024, 1024
    layers = [synth.make_problem(wtype, M, N, K, seed=500 + i) for i in range(3)]
    Ws = [_dev(pb.W.reshape(-1)) for pb in layers]
    x0 = torch.empty((M, K), dtype=torch.float32, device=DEV)
    xq = torch.empty(api.q8_1_bytes(M, K), dtype=torch.uint8, device=DEV)
    outs = [torch.empty((M, N), dtype=torch.float32, device=DEV) for _ in layers]

    def decode():
        src = x0
        for W, o in zip(Ws, outs):
            api.quantize_q8_1(src, out=xq)
            api.gemm(wtype, W, xq, M, N, K, out=o)
            src = o                                   # N == K: the next layer reads this output
    x0.copy_(_dev(layers[0].x))
    decode()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        decode()
    for seed in (7, 8):
        x = np.random.default_rng(seed).standard_normal((M, K), dtype=np.float32)
        x0.copy_(_dev(x))
        g.replay()
        torch.cuda.synchronize()
        src = x
        for pb, o in zip(layers, outs):
            q, d, s = oracle.quantize_q8_1(src)
            ref = oracle.gemm(wtype, pb.W, q, d, s, N)
            assert np.array_equal(o.cpu().numpy().view(np.uint32), ref.view(np.uint32))
            src = ref


@pytest.mark.parametrize("wtype", BLOCK_TYPES)
@pytest.mark.parametrize("M", [1, 4, 8])
def test_few_token_path_bit_exact_at_the_bounds(wtype, M):
    # weight and activation codes at the ends of their ranges (every in-block dot at or near its largest
    # magnitude), random scales: the matrix-vector kernel stays bit-identical to the oracle
    N, K = 67, 2048
    g = np.random.default_rng(41 + wtype + M)
    W = synth.pack(wtype, _extreme_fields(wtype, N, K, g))
    q = np.where(g.integers(0, 2, size=(M, K)) == 0, -127, 127).astype(np.int8)
    q[0] = 127
    d = g.uniform(1e-3, 1e-2, size=(M, K // 32)).astype(np.float32)
    s = (d * q.reshape(M, K // 32, 32).sum(-1, dtype=np.int32).astype(np.float32)).astype(np.float32)
    xq = api.pack_q8_1(torch.from_numpy(q), torch.from_numpy(d), torch.from_numpy(s)).to(DEV)
    out = api.gemm(wtype, _dev(W.reshape(-1)), xq, M, N, K).cpu().numpy()
    ref = oracle.gemm(wtype, W, q, d, s, N)
    assert np.array_equal(out.view(np.uint32), ref.view(np.uint32)), np.abs(out - ref).max()


@pytest.mark.parametrize("wtype", [synth.Q6_K, synth.Q4_K])
def test_small_grid_k_parts_at_super_stage_boundaries(wtype):
    # 2 tiles on a 152-SM part: every tile runs in 16 K parts; K = 11008 has 43 super-stages, so the
    # parts hold 2 or 3 of them
    M, N, K = 40, 200, 11008
    pb = synth.make_problem(wtype, M, N, K, seed=73 + wtype)
    q, d, s, xq = _oracle_acts(pb)
    out = api.gemm(wtype, _dev(pb.W.reshape(-1)), xq, M, N, K).cpu().numpy()
    assert api.read_device_errors() == 0
    assert _rel_err(out, oracle.gemm(wtype, pb.W, q, d, s, N)) <= TOL


@pytest.mark.parametrize("wtype", PARTIAL_TYPES)
@pytest.mark.parametrize("shape", [(3, 5, 256), (131, 200, 512)])
def test_debug_partials_bit_exact(wtype, shape):
    M, N, K = shape
    pb = synth.make_problem(wtype, M, N, K, seed=21 + M + wtype)
    if wtype == synth.W8A8:
        xq = _dev(synth.pack_w8a8_acts(pb.X, pb.xs))
        P = api.gemm_debug_partials(wtype, _dev(pb.W), xq, M, N, K).cpu().numpy()
        ref = oracle.partials(synth.W8A8, pb.X, pb.fields.W)
    else:
        q, d, s, xq = _oracle_acts(pb)
        P = api.gemm_debug_partials(wtype, _dev(pb.W.reshape(-1)), xq, M, N, K).cpu().numpy()
        wq, _, _ = oracle.decode(wtype, pb.W, N, K)
        ref = oracle.partials(wtype, q, wq)
    assert np.array_equal(P, ref)


@pytest.mark.parametrize("wtype", BLOCK_TYPES)
@pytest.mark.parametrize("shape", [(3, 5, 1024), (131, 200, 2048), (257, 130, 1024)])
def test_tma_block_sums_bit_exact(wtype, shape):
    # the production kernel's integer accumulators, sub-scales folded in, bit for bit
    M, N, K = shape
    pb = synth.make_problem(wtype, M, N, K, seed=23 + M + wtype)
    q, d, s, xq = _oracle_acts(pb)
    A = api.gemm_debug_block_sums(wtype, _dev(pb.W.reshape(-1)), xq, M, N, K).cpu().numpy()
    assert api.read_device_errors() == 0
    assert np.array_equal(A, oracle.block_sums(wtype, pb.W, q, N))


def test_tma_block_sums_exact_at_the_bounds():
    # q6_K with |q - 32| = 32 and sc = -128 everywhere against activation codes of +-127: every block sum
    # is 32 * 4096 * 127 in magnitude, the largest the folded operands can produce (< 2^24)
    M, N, K = 4, 130, 1024
    pb = synth.make_problem(synth.Q6_K, M, N, K, seed=29)
    pb.fields.code[...] = 0
    pb.fields.sc[...] = -128
    W = synth.pack(synth.Q6_K, pb.fields)
    q = np.where(np.arange(M * K).reshape(M, K) % 3 == 0, -127, 127).astype(np.int8)
    q[0] = 127                         # rows 0 and 1: every block sum at +-32 * 4096 * 127
    q[1] = -127
    d = np.full((M, K // 32), 0.01, np.float32)
    s = (d * q.reshape(M, K // 32, 32).sum(-1)).astype(np.float32)
    xq = api.pack_q8_1(torch.from_numpy(q), torch.from_numpy(d), torch.from_numpy(s)).to(DEV)
    A = api.gemm_debug_block_sums(synth.Q6_K, _dev(W.reshape(-1)), xq, M, N, K).cpu().numpy()
    ref = oracle.block_sums(synth.Q6_K, W, q, N)
    assert np.abs(ref).max() == 32 * 4096 * 127
    assert np.array_equal(A, ref)


def test_partials_exact_at_the_block_bound():
    # every product at its maximum magnitude: block dots of +-32*127*127 must come out exact
    M, N, K = 130, 130, 512
    f = synth.draw_fields(np.random.default_rng(1), synth.Q8_0, N, K)
    f.q[...] = np.where(np.arange(N)[:, None] % 2 == 0, 127, -127).astype(np.int8)
    W = synth.pack(synth.Q8_0, f)
    q = np.where(np.arange(M)[:, None] % 3 == 0, -127, 127).astype(np.int8) * np.ones((M, K), np.int8)
    d = np.ones((M, K // 32), np.float32)
    xq = api.pack_q8_1(torch.from_numpy(q), torch.from_numpy(d), torch.from_numpy(d)).to(DEV)
    P = api.gemm_debug_partials(synth.Q8_0, _dev(W.reshape(-1)), xq, M, N, K).cpu().numpy()
    ref = oracle.partials(synth.Q8_0, q, f.q)
    assert np.abs(ref).max() == 32 * 127 * 127
    assert np.array_equal(P, ref)


# ---------------------------------------------------------------------------------------- W8A8
@pytest.mark.parametrize("shape", [(1, 1, 64), (70, 200, 576), (300, 260, 4096)])
def test_w8a8_bit_exact(shape):
    M, N, K = shape
    pb = synth.make_problem(synth.W8A8, M, N, K, seed=31 + M)
    out = api.gemm(synth.W8A8, _dev(pb.W), _dev(synth.pack_w8a8_acts(pb.X, pb.xs)), M, N, K)
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    ref = oracle.w8a8(pb.fields.W, pb.fields.ws, pb.X, pb.xs)
    assert np.array_equal(got, ref)


def test_w8a8_exact_at_the_int32_range():
    # all products +-127*127 over K = 4096: |I| = 66 064 384 > 2^24, exact only with chunked accumulation
    M, N, K = 130, 129, 4096
    X = np.where(np.arange(M)[:, None] % 2 == 0, 127, -127).astype(np.int8) * np.ones((M, K), np.int8)
    W = np.full((N, K), 127, np.int8)
    W[1::3] = -127
    W[2::3, ::2] = 0
    xs = np.ones(M, np.float32)
    ws = np.ones(N, np.float32)
    out = api.gemm(synth.W8A8, _dev(synth.pack(synth.W8A8, synth.W8A8Fields(W=W, ws=ws))),
                   _dev(synth.pack_w8a8_acts(X, xs)), M, N, K)
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, oracle.w8a8(W, ws, X, xs))


# ---------------------------------------------------------------------------------------- end to end
@pytest.mark.parametrize("wtype", BLOCK_TYPES)
def test_quantize_then_gemm_end_to_end(wtype):
    M, N, K = 150, 260, 1024
    pb = synth.make_problem(wtype, M, N, K, seed=41 + wtype)
    xq = api.quantize_q8_1(_dev(pb.x))
    out = api.gemm(wtype, _dev(pb.W.reshape(-1)), xq, M, N, K).cpu().numpy()
    q, d, s = oracle.quantize_q8_1(pb.x)
    assert _rel_err(out, oracle.gemm(wtype, pb.W, q, d, s, N)) <= TOL


# ---------------------------------------------------------------------------------------- MoE
@pytest.mark.parametrize("wtype", [synth.IQ1_M, synth.Q4_K, synth.Q8_0, synth.Q6_K])
@pytest.mark.parametrize("M,E,slots,N,K", [(24, 6, 3, 130, 256), (300, 16, 4, 256, 512)])
def test_gemm_id_matches_oracle(wtype, M, E, slots, N, K):
    pb = synth.make_problem(wtype, M, N, K, seed=51 + M + wtype, experts=E, slots=slots)
    q, d, s, xq = _oracle_acts(pb)
    out = api.gemm_id(wtype, _dev(pb.W.reshape(-1)), E, xq, _dev(pb.ids), M, N, K).cpu().numpy()
    ref = oracle.gemm_id(wtype, pb.W, E, q, d, s, pb.ids, N)
    for t in range(M):
        for j in range(slots):
            assert _rel_err(out[t, j], ref[t, j]) <= TOL, (t, j)


@pytest.mark.parametrize("wtype", BLOCK_TYPES)
def test_gemm_id_tma_path_matches_oracle(wtype):
    # K % 1024 == 0: every block type takes the TMA-fed kernel on the gathered operand; N = 260 leaves a
    # ragged weight-row tile, uneven expert counts leave work items of every size
    M, E, slots, N, K = 200, 5, 3, 260, 1024
    pb = synth.make_problem(wtype, M, N, K, seed=57 + wtype, experts=E, slots=slots)
    q, d, s, xq = _oracle_acts(pb)
    out = api.gemm_id(wtype, _dev(pb.W.reshape(-1)), E, xq, _dev(pb.ids), M, N, K).cpu().numpy()
    ref = oracle.gemm_id(wtype, pb.W, E, q, d, s, pb.ids, N)
    assert api.read_device_errors() == 0
    for t in range(M):
        for j in range(slots):
            assert _rel_err(out[t, j], ref[t, j]) <= TOL, (t, j)


@pytest.mark.parametrize("E", [38, 40])
def test_gemm_id_tma_tail_split(E):
    # more (work item, row tile) pairs than one wave of CTAs on a 152-SM part: 38 items x 5 row tiles
    # leave 38 tiles in the last wave (split in 4 K parts), 40 x 5 leave 48 (split in 2); each part adds
    # into an output zeroed by the gather pass
    M, slots, N, K = 1000, 2, 640, 1024
    pb = synth.make_problem(synth.Q4_0, M, N, K, seed=67 + E, experts=E, slots=slots)
    q, d, s, xq = _oracle_acts(pb)
    out = api.gemm_id(synth.Q4_0, _dev(pb.W.reshape(-1)), E, xq, _dev(pb.ids), M, N, K).cpu().numpy()
    ref = oracle.gemm_id(synth.Q4_0, pb.W, E, q, d, s, pb.ids, N)
    assert api.read_device_errors() == 0
    for t in range(0, M, 7):
        for j in range(slots):
            assert _rel_err(out[t, j], ref[t, j]) <= TOL, (t, j)


def test_gemm_id_tma_path_with_three_kernel_routing():
    # 8200 tokens x 8 slots = 65 600 routed rows: past the single-block routing kernel's limit, so the
    # three-kernel route feeds the gather and the TMA-fed grouped GEMM
    M, E, slots, N, K = 8200, 96, 8, 130, 256
    pb = synth.make_problem(synth.Q4_0, M, N, K, seed=69, experts=E, slots=slots)
    q, d, s, xq = _oracle_acts(pb)
    out = api.gemm_id(synth.Q4_0, _dev(pb.W.reshape(-1)), E, xq, _dev(pb.ids), M, N, K).cpu().numpy()
    assert api.read_device_errors() == 0
    rows = np.arange(0, M, 97)
    ref = oracle.gemm_id(synth.Q4_0, pb.W, E, q[rows], d[rows], s[rows], pb.ids[rows], N)
    for i, t in enumerate(rows):
        for j in range(slots):
            assert _rel_err(out[t, j], ref[i, j]) <= TOL, (t, j)


def test_gemm_id_tma_path_skewed_routing():
    # expert 0 receives every token's slot 0 (300 rows: work items of 128, 128 and 44 rows), the other
    # experts share slot 1
    M, E, slots, N, K = 300, 8, 2, 130, 1024
    pb = synth.make_problem(synth.IQ1_M, M, N, K, seed=63, experts=E, slots=slots)
    pb.ids[:, 0] = 0
    pb.ids[:, 1] = 1 + np.arange(M) % (E - 1)
    q, d, s, xq = _oracle_acts(pb)
    out = api.gemm_id(synth.IQ1_M, _dev(pb.W.reshape(-1)), E, xq, _dev(pb.ids), M, N, K).cpu().numpy()
    ref = oracle.gemm_id(synth.IQ1_M, pb.W, E, q, d, s, pb.ids, N)
    assert api.read_device_errors() == 0
    assert _rel_err(out, ref) <= TOL


def test_gemm_id_skewed_routing():
    # every token routes slot 0 to expert 0: one expert receives M rows (several token tiles)
    M, E, slots, N, K = 300, 8, 2, 130, 256
    pb = synth.make_problem(synth.IQ1_M, M, N, K, seed=61, experts=E, slots=slots)
    pb.ids[:, 0] = 0
    pb.ids[:, 1] = 1 + np.arange(M) % (E - 1)
    q, d, s, xq = _oracle_acts(pb)
    out = api.gemm_id(synth.IQ1_M, _dev(pb.W.reshape(-1)), E, xq, _dev(pb.ids), M, N, K).cpu().numpy()
    ref = oracle.gemm_id(synth.IQ1_M, pb.W, E, q, d, s, pb.ids, N)
    assert _rel_err(out, ref) <= TOL


@pytest.mark.parametrize("wtype", BLOCK_TYPES)
@pytest.mark.parametrize("M,E,slots,N,K", [(1, 32, 8, 130, 1280), (3, 8, 4, 257, 2048), (8, 16, 2, 64, 768),
                                           (8, 8, 8, 96, 512), (8, 16, 9, 96, 512)])
def test_few_token_gemm_id_bit_exact(wtype, M, E, slots, N, K):
    # M <= 8 tokens: each (token, slot) pair runs as a one-token product with its expert on the
    # matrix-vector kernel, which reads the ids itself (no routing lists); every row equals the oracle's
    # bit for bit, through both MoE entry points (K = 1280 and 768 end in a partial chunk of blocks; every
    # token routed to all 8 experts; 9 slots per token)
    pb = synth.make_problem(wtype, M, N, K, seed=91 + M + wtype, experts=E, slots=slots)
    q, d, s, xq = _oracle_acts(pb)
    W, ids = _dev(pb.W.reshape(-1)), _dev(pb.ids)
    ref = oracle.gemm_id(wtype, pb.W, E, q, d, s, pb.ids, N)
    api.read_device_errors()
    out = api.gemm_id(wtype, W, E, xq, ids, M, N, K).cpu().numpy()
    assert np.array_equal(out.view(np.uint32), ref.view(np.uint32)), np.abs(out - ref).max()
    if wtype != synth.Q6_K:
        out2 = api.gemm_id_noalloc(wtype, W, E, xq, ids, M, N, K).cpu().numpy()
        assert np.array_equal(out2.view(np.uint32), ref.view(np.uint32))
    assert api.read_device_errors() == 0


def test_few_token_gemm_id_duplicate_ids_flagged_and_computed():
    # the few-token MoE path checks the routing contract too: a token that lists an expert twice raises
    # MMQ_DEVERR_DUP_EXPERT and both rows still hold that expert's product
    wtype, M, E, slots, N, K = synth.IQ1_M, 4, 6, 3, 96, 1024
    pb = synth.make_problem(wtype, M, N, K, seed=97, experts=E, slots=slots)
    ids = pb.ids.copy()
    ids[2, 2] = ids[2, 0]
    q, d, s, xq = _oracle_acts(pb)
    api.read_device_errors()
    out = api.gemm_id(wtype, _dev(pb.W.reshape(-1)), E, xq, _dev(ids), M, N, K).cpu().numpy()
    bits = api.read_device_errors()
    assert bits & api.DEVERR_DUP_EXPERT
    assert not bits & api.DEVERR_EXPERT_ID
    ref = oracle.gemm_id(wtype, pb.W, E, q, d, s, ids, N)
    assert np.array_equal(out.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("bad", ["past_end", "negative"])
@pytest.mark.parametrize("M", [8, 40])          # the matrix-vector kernel, then the routed tile path
def test_gemm_id_out_of_range_ids_flagged_and_skipped(bad, M):
    E, slots, N, K = 4, 2, 128, 256
    pb = synth.make_problem(synth.Q4_0, M, N, K, seed=71, experts=E, slots=slots)
    ids = pb.ids.copy()
    ids[3, 1] = E + 5 if bad == "past_end" else -1
    q, d, s, xq = _oracle_acts(pb)
    out = torch.full((M, slots, N), 7.0, device=DEV)
    api.gemm_id(synth.Q4_0, _dev(pb.W.reshape(-1)), E, xq, _dev(ids), M, N, K, out=out)
    bits = api.read_device_errors()
    assert bits & api.DEVERR_EXPERT_ID
    assert torch.all(out[3, 1] == 7.0)
    ids_ok = ids.copy()
    ids_ok[3, 1] = ids[3, 0]
    ref = oracle.gemm_id(synth.Q4_0, pb.W, E, q, d, s, np.where((ids >= 0) & (ids < E), ids, 0).astype(np.int32), N)
    o = out.cpu().numpy()
    for t in range(M):
        for j in range(slots):
            if (t, j) != (3, 1):
                assert _rel_err(o[t, j], ref[t, j]) <= TOL


@pytest.mark.parametrize("wtype,M,E,slots,N,K", [(synth.Q4_0, 24, 6, 3, 130, 512),      # TMA path, fused routing
                                                  (synth.IQ1_M, 40, 9, 4, 128, 1024),
                                                  (synth.Q4_K, 24, 6, 3, 130, 512)])
def test_gemm_id_duplicate_expert_ids_flagged_and_computed(wtype, M, E, slots, N, K):
    # a token that lists the same expert twice breaks the routing contract (ids distinct per token):
    # the device raises MMQ_DEVERR_DUP_EXPERT, and every (token, slot) row -- the repeated ones
    # included -- still holds W_{ids[t][j]} applied to token t, as the definition gives
    pb = synth.make_problem(wtype, M, N, K, seed=73 + M, experts=E, slots=slots)
    ids = pb.ids.copy()
    ids[5, 2] = ids[5, 0]
    ids[M - 1, 1] = ids[M - 1, 2]
    q, d, s, xq = _oracle_acts(pb)
    out = api.gemm_id(wtype, _dev(pb.W.reshape(-1)), E, xq, _dev(ids), M, N, K)
    bits = api.read_device_errors()
    assert bits & api.DEVERR_DUP_EXPERT
    assert not bits & api.DEVERR_EXPERT_ID
    ref = oracle.gemm_id(wtype, pb.W, E, q, d, s, ids, N)
    o = out.cpu().numpy()
    for t in range(M):
        for j in range(slots):
            assert _rel_err(o[t, j], ref[t, j]) <= TOL, (t, j)


# ---------------------------------------------------------------------------------------- failure handling
def test_bounded_wait_gives_up_reports_and_leaves_the_context_usable():
    # a barrier that nothing arrives at: both wait flavours give up, flag the CTA and record the timeout
    res = api.selftest_bounded_wait(DEV)
    assert res == [0, 1, 0, 1], res
    assert api.read_device_errors() & api.DEVERR_TIMEOUT
    assert api.read_device_errors() == 0                   # read and cleared
    # the context still runs the product
    M, N, K = 64, 130, 512
    pb = synth.make_problem(synth.Q4_0, M, N, K, seed=81)
    q, d, s, xq = _oracle_acts(pb)
    out = api.gemm(synth.Q4_0, _dev(pb.W.reshape(-1)), xq, M, N, K).cpu().numpy()
    assert _rel_err(out, oracle.gemm(synth.Q4_0, pb.W, q, d, s, N)) <= TOL


# ---------------------------------------------------------------------------------------- degenerate sizes
def test_empty_inputs_are_noops():
    W = torch.zeros(1024, dtype=torch.uint8, device=DEV)
    xq = torch.zeros(1024, dtype=torch.uint8, device=DEV)
    out = torch.zeros(16, device=DEV)
    assert api.load().mmq_gemm(synth.Q4_0, W.data_ptr(), xq.data_ptr(), out.data_ptr(), 0, 5, 256, None) == 0
    assert api.load().mmq_gemm(synth.Q4_0, W.data_ptr(), xq.data_ptr(), out.data_ptr(), 5, 0, 256, None) == 0
    assert api.load().mmq_quantize_q8_1(out.data_ptr(), 0, 64, xq.data_ptr(), None) == 0
    torch.cuda.synchronize()
    assert torch.all(out == 0)
