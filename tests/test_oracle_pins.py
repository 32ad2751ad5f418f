"""Pins of the CPU oracle against what the pages and the mathematics fix (no GPU needed).

Each test checks the oracle against something other than itself:
  * library routines for pure conversions (numpy's IEEE half decode, torch's bf16 rounding);
  * closed forms (blocks whose scale is a power of two, so the codes are known integers; ties);
  * invariants of the q8_1 quantizer ("08 · R1 — int8 MMQ prefill GEMM", §2.2 / §3.2);
  * the generator's independent byte packer (round trip) and hand-written single-bit blocks;
  * the IQ1_M fold identity and value set printed in "CUDA: add IQ1_M to MMQ" (Design), exhaustively;
  * brute-force int64 dots for the per-group integer partials ("08 · R1", §2.1), and the bounds;
  * an f64 dequantise-then-matmul of the generator's fields with the f32 summation error bound
    ("A Negative Result on int8 Tensor-Core MMQ", §2: the blockwise sum equals the dequantised product);
  * special cases of W8A8 and MoE routing that reduce to integer matmuls or to the dense product.
A dropped min term, a wrong sign polarity, swapped nibbles, a transposed operand, round-half-away or
an off-by-one group size each fail at least one test here (see test_oracle_mutants.py).
"""
import os

import numpy as np
import pytest

import oracle
from block_quantized_int8_q8_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_ints(name):
    vals = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                vals.append(line)
    return vals


# ---------------------------------------------------------------------------------- scalar helpers
def test_half_to_float_matches_ieee_library_for_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = np.array([oracle.half_to_float(int(b)) for b in bits], np.float32)
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite].view(np.uint32), ref[finite].view(np.uint32))
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isinf(got), np.isinf(ref))


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    g = np.random.default_rng(7)
    vals = np.concatenate([
        g.standard_normal(20000).astype(np.float32) * np.float32(1e3),
        # exact ties between two bf16 values (lower 16 bits = 0x8000), both parities
        (np.arange(1000, dtype=np.uint32) * 0x10000 + 0x3F808000).view(np.float32),
        np.array([0.0, -0.0, 1.0, -1.0, 3.4e38, -3.4e38, 1e-40], np.float32),
    ])
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.float_to_bf16(float(v)) for v in vals], np.uint16)
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------------------------- q8_1 quantizer
def test_quantizer_closed_form_power_of_two_scale():
    # x = c*k with c a power of two and max|k| = 127: d = 127c/127 = c exactly, so q = k, s = c*sum(k).
    g = np.random.default_rng(1)
    for e in (-10, -4, 0, 3):
        c = np.float32(2.0 ** e)
        k = g.integers(-127, 128, size=(5, 64)).astype(np.int32)
        k[:, 0] = 127
        k[:, 33] = -127
        q, d, s = oracle.quantize_q8_1(k.astype(np.float32) * c)
        assert np.array_equal(q.astype(np.int32), k)
        assert np.all(d == c)
        sums = k.reshape(5, 2, 32).sum(-1)
        assert np.array_equal(s, (sums * float(c)).astype(np.float32))


def test_quantizer_rounds_half_to_even():
    # amax = 127 gives d = 1 exactly; x/d is then x itself, so halves are exact ties.
    x = np.zeros((1, 32), np.float32)
    x[0, :9] = [127.0, 2.5, 3.5, -2.5, -3.5, 0.5, -0.5, 1.5, 126.5]
    q, d, s = oracle.quantize_q8_1(x)
    assert d[0, 0] == 1.0
    assert list(q[0, :9]) == [127, 2, 4, -2, -4, 0, 0, 2, 126]
    assert s[0, 0] == float(sum([127, 2, 4, -2, -4, 0, 0, 2, 126]))


def test_quantizer_zero_and_single_value_blocks():
    x = np.zeros((2, 64), np.float32)
    x[1, 40] = -0.37
    q, d, s = oracle.quantize_q8_1(x)
    assert np.all(q[0] == 0) and np.all(d[0] == 0) and np.all(s[0] == 0)
    assert d[1, 0] == 0 and np.all(q[1, :32] == 0)
    assert q[1, 40] == -127 and np.count_nonzero(q[1, 32:]) == 1
    assert d[1, 1] == np.float32(np.float32(0.37) / np.float32(127.0))


@pytest.mark.parametrize("dist", ["normal", "heavy", "tiny", "mixed_scale"])
def test_quantizer_invariants(dist):
    g = np.random.default_rng(11)
    M, K = 33, 512
    if dist == "normal":
        x = g.standard_normal((M, K)).astype(np.float32)
    elif dist == "heavy":
        x = (g.standard_cauchy((M, K)) * 3).astype(np.float32)
    elif dist == "tiny":
        x = (g.standard_normal((M, K)) * 1e-30).astype(np.float32)
    else:
        x = (g.standard_normal((M, K)) * 10.0 ** g.integers(-8, 8, size=(M, 1))).astype(np.float32)
    q, d, s = oracle.quantize_q8_1(x)
    xb = x.reshape(M, K // 32, 32).astype(np.float64)
    qb = q.reshape(M, K // 32, 32).astype(np.int64)
    amax = np.abs(xb).max(-1)
    assert np.all(np.abs(qb) <= 127)
    nz = amax > 0
    assert np.all(np.abs(qb).max(-1)[nz] == 127)
    # d is the f32-rounded amax/127
    assert np.all(np.abs(d.astype(np.float64) - amax / 127.0) <= amax / 127.0 * 2.0 ** -24)
    # reconstruction error: |x - d q| <= d (1/2 + 127 * 2^-24)
    err = np.abs(xb - d[..., None].astype(np.float64) * qb)
    assert np.all(err <= d[..., None].astype(np.float64) * (0.5 + 127 * 2.0 ** -23))
    # s is d * sum(q) rounded once to f32
    exact = d.astype(np.float64) * qb.sum(-1)
    assert np.all(np.abs(s.astype(np.float64) - exact) <= np.abs(exact) * 2.0 ** -24)


# ---------------------------------------------------------------------------------- decoders
@pytest.mark.parametrize("wtype", [synth.Q8_0, synth.Q4_0, synth.Q4_K, synth.IQ1_M, synth.Q6_K])
def test_decoder_round_trip_with_generator_packer(wtype):
    N, K = 7, 1024
    f = synth.draw_fields(np.random.default_rng(3 + wtype), wtype, N, K)
    W = synth.pack(wtype, f)
    wq, wsc, wmin = oracle.decode(wtype, W, N, K)
    if wtype == synth.Q8_0:
        assert np.array_equal(wq, f.q)
        assert np.array_equal(wsc, f.d.astype(np.float32))
    elif wtype == synth.Q4_0:
        assert np.array_equal(wq.astype(np.int32), f.code.astype(np.int32) - 8)
        assert np.array_equal(wsc, f.d.astype(np.float32))
    elif wtype == synth.Q4_K:
        assert np.array_equal(wq.astype(np.int32), f.code.astype(np.int32))
        d = np.repeat(f.d.astype(np.float64), 8, axis=1)
        dm = np.repeat(f.dmin.astype(np.float64), 8, axis=1)
        assert np.array_equal(wsc.astype(np.float64), d * f.sc)      # exact: 11-bit x 6-bit
        assert np.array_equal(wmin.astype(np.float64), dm * f.m)
    elif wtype == synth.Q6_K:
        # "08 · R1" §2.2: the 6-bit grid moves to the signed domain by subtracting 32
        assert np.array_equal(wq.astype(np.int32), f.code.astype(np.int32) - 32)
        d = np.repeat(f.d.astype(np.float64), 16, axis=1)
        assert np.array_equal(wsc.astype(np.float64), d * f.sc)      # exact: 11-bit x 8-bit
    else:
        neg = np.repeat(f.neg, 8, axis=1).astype(np.int32)
        assert np.array_equal(wq.astype(np.int32), 8 * f.g.astype(np.int32) + np.where(neg == 1, -1, 1))
        d = np.repeat(f.d.astype(np.float64), 16, axis=1)
        assert np.array_equal(wsc.astype(np.float64), d * (2 * f.s.astype(np.float64) + 1) / 8)


def test_q4_k_hand_built_single_field_blocks():
    # d = 1, dmin = 2; only sc[3] = 1 and m[5] = 63 set; code of value 70 = 9 (byte 32*1+6 low nibble),
    # code of value 100 = 4 (byte 32*1+4 high nibble: value 64+32+4).
    blk = np.zeros(144, np.uint8)
    blk[0:2] = np.array([1.0], np.float16).view(np.uint8)
    blk[2:4] = np.array([2.0], np.float16).view(np.uint8)
    # six-bit field j occupies bits 6j..6j+5 of the 96-bit little-endian stream at byte 4
    stream = 0
    stream |= 1 << (6 * 3)            # sc[3] = 1
    stream |= 63 << (6 * (8 + 5))     # m[5] = 63
    blk[4:16] = np.frombuffer(stream.to_bytes(12, "little"), np.uint8)
    blk[16 + 32 + 6] = 9
    blk[16 + 32 + 4] = 4 << 4
    wq, wsc, wmin = oracle.decode(synth.Q4_K, blk[None], 1, 256)
    assert list(wsc[0]) == [0, 0, 0, 1, 0, 0, 0, 0]
    assert list(wmin[0]) == [0, 0, 0, 0, 0, 126, 0, 0]
    nz = np.flatnonzero(wq[0])
    assert list(nz) == [70, 100] and wq[0, 70] == 9 and wq[0, 100] == 4


def test_q6_k_hand_built_single_field_blocks():
    # d = 0.25; sc[2] = -3, sc[13] = 127; every code 32 (value 0) except: value 33 (stage 0, low nibble in
    # byte 1 high half, high pair in byte 1 bits 4-5) = 63 -> +31; value 64+18 (stage 1, low nibble in
    # byte 18 low half, high pair in byte 2 bits 2-3) = 0 -> -32; value 192+50 (stage 3, byte 18 high
    # half, high pair in byte 2 bits 6-7) = 47 -> +15.
    blk = np.zeros(224, np.uint8)
    blk[2] = np.uint8(np.int8(-3).view(np.uint8))
    blk[13] = 127
    blk[16:18] = np.array([0.25], np.float16).view(np.uint8)
    for j in range(4):                 # all codes 32: low nibble 0, high pair 2 -> 0b10 in every field
        blk[32 + 48 * j: 64 + 48 * j] = 0x00
        blk[64 + 48 * j: 80 + 48 * j] = 0xAA
    r0, r1, r3 = 32, 32 + 48, 32 + 3 * 48
    blk[r0 + 1] = 0xF0                                  # value 33 low nibble 15
    blk[r0 + 32 + 1] = (0xAA & ~(3 << 4)) | (3 << 4)    # value 33 high pair 3 -> code 63
    blk[r1 + 18] = 0x00                                 # value 82 low nibble 0
    blk[r1 + 32 + 2] = 0xAA & ~(3 << 2)                 # value 64+18 high pair 0 -> code 0
    blk[r3 + 18] = 0xF0                                 # value 192+50 low nibble 15
    blk[r3 + 32 + 2] = 0xAA & ~(3 << 6)                 # high pair of value 192+50 = 0... code 15
    blk[r3 + 32 + 2] |= (2 << 6)                        # ... pair 2: code 32 + 15 = 47
    wq, wsc, _ = oracle.decode(synth.Q6_K, blk[None], 1, 256)
    assert wsc[0, 2] == -0.75 and wsc[0, 13] == 31.75 and wsc[0, 0] == 0.0
    nz = np.flatnonzero(wq[0])
    assert list(nz) == [33, 82, 242], list(nz)
    assert (wq[0, 33], wq[0, 82], wq[0, 242]) == (31, -32, 15)


def test_q4_0_hand_built_nibble_order():
    blk = np.zeros(18, np.uint8)
    blk[0:2] = np.array([0.5], np.float16).view(np.uint8)
    blk[2:] = 0x88                     # all codes 8 -> value 0
    blk[2 + 3] = 0x8F                  # value 3 = 15-8 = 7
    blk[2 + 5] = 0x18                  # value 21 = 1-8 = -7
    wq, wsc, _ = oracle.decode(synth.Q4_0, np.tile(blk, 8)[None], 1, 256)
    assert wsc[0, 0] == 0.5
    assert wq[0, 3] == 7 and wq[0, 21] == -7
    assert np.count_nonzero(wq[0, :32]) == 2


def test_iq1_m_fold_exhaustive_and_value_set():
    golden = sorted(int(v) for v in _golden_ints("iq1_m_fold_values.txt"))
    ds = np.array([1e-3, 3.3e-3, 7.77e-3, 1e-2, 0.5, 65504.0, 6.1e-5], np.float16)
    for dv in ds:
        for s in range(8):
            # one super-block: values 0..15 share s; g cycles over {-1,0,1}, signs alternate per 8
            N, K = 1, 256
            f = synth.IQ1_MFields(d=np.full((1, 1), dv, np.float16),
                                  s=np.full((1, 16), s, np.uint8),
                                  neg=(np.arange(32) % 2).astype(np.uint8)[None],
                                  g=((np.arange(256) % 3) - 1).astype(np.int8)[None])
            wq, wsc, _ = oracle.decode(synth.IQ1_M, synth.pack(synth.IQ1_M, f), N, K)
            assert sorted(set(wq[0].tolist())) == golden
            gv = f.g[0].astype(np.float64)
            delta = np.where(np.repeat(f.neg[0], 8) == 1, -1.0 / 8, 1.0 / 8)
            exact = float(dv) * (2 * s + 1) * (gv + delta)                        # d(2s+1)(g+delta)
            folded64 = np.repeat(wsc[0].astype(np.float64), 16) * wq[0].astype(np.float64)
            assert np.array_equal(folded64, exact)
            folded32 = np.repeat(wsc[0], 16) * wq[0].astype(np.float32)          # f32 product exact too
            assert np.array_equal(folded32.astype(np.float64), exact)


# ---------------------------------------------------------------------------------- integer partials
@pytest.mark.parametrize("wtype", [synth.Q8_0, synth.Q4_0, synth.Q4_K, synth.IQ1_M, synth.W8A8, synth.Q6_K])
def test_partials_brute_force(wtype):
    g = np.random.default_rng(20 + wtype)
    M, N, K = 5, 6, 512
    xq = g.integers(-127, 128, size=(M, K)).astype(np.int8)
    wq = g.integers(-127 if wtype != synth.IQ1_M else -9, 128 if wtype != synth.IQ1_M else 10,
                    size=(N, K)).astype(np.int8)
    P = oracle.partials(wtype, xq, wq)
    G = 16 if wtype in (synth.IQ1_M, synth.Q6_K) else 32
    for m in range(M):
        for n in range(N):
            for gi in range(K // G):
                ref = sum(int(xq[m, k]) * int(wq[n, k]) for k in range(gi * G, gi * G + G))
                assert P[m, n, gi] == ref


@pytest.mark.parametrize("wtype", [synth.Q8_0, synth.Q4_0, synth.Q4_K, synth.IQ1_M, synth.Q6_K])
def test_block_sums_brute_force_from_generator_fields(wtype):
    # the folded 32-k block sums computed in int64 straight from the drawn fields (no oracle decoder)
    g = np.random.default_rng(60 + wtype)
    M, N, K = 3, 5, 512
    f = synth.draw_fields(g, wtype, N, K)
    W = synth.pack(wtype, f)
    xq = g.integers(-127, 128, size=(M, K)).astype(np.int8)
    if wtype == synth.Q8_0:
        wint = f.q.astype(np.int64)
    elif wtype == synth.Q4_0:
        wint = f.code.astype(np.int64) - 8
    elif wtype == synth.Q4_K:
        wint = np.repeat(f.sc.astype(np.int64), 32, 1) * f.code
    elif wtype == synth.IQ1_M:
        fold = 8 * f.g.astype(np.int64) + np.where(np.repeat(f.neg, 8, 1) == 1, -1, 1)
        wint = np.repeat(2 * f.s.astype(np.int64) + 1, 16, 1) * fold
    else:
        wint = np.repeat(f.sc.astype(np.int64), 16, 1) * (f.code.astype(np.int64) - 32)
    ref = np.einsum("mbk,nbk->mnb", xq.astype(np.int64).reshape(M, K // 32, 32), wint.reshape(N, K // 32, 32))
    A = oracle.block_sums(wtype, W, xq, N)
    assert np.array_equal(A.astype(np.int64), ref)


def test_partial_bounds_from_pages():
    bounds = dict(line.split() for line in _golden_ints("bounds.txt"))
    # IQ1_M per-16 extreme: q = 127 against the largest fold value 9 everywhere
    xq = np.full((1, 256), 127, np.int8)
    wq = np.full((1, 256), 9, np.int8)
    assert oracle.partials(synth.IQ1_M, xq, wq).max() == int(bounds["iq1_m_per16_dot_bound"])
    xq = np.full((1, 256), -128, np.int8)
    wq = np.full((1, 256), 127, np.int8)
    assert -oracle.partials(synth.Q8_0, xq, wq).min() == int(bounds["q8_block_dot_bound"])


# ---------------------------------------------------------------------------------- blockwise product
def _dequant_f64(wtype, f):
    """Dequantised weights in f64 straight from the generator's fields (no oracle code)."""
    if wtype == synth.Q8_0:
        return np.repeat(f.d.astype(np.float64), 32, 1) * f.q
    if wtype == synth.Q4_0:
        return np.repeat(f.d.astype(np.float64), 32, 1) * (f.code.astype(np.float64) - 8)
    if wtype == synth.Q4_K:
        d = np.repeat(f.d.astype(np.float64), 256, 1)
        dm = np.repeat(f.dmin.astype(np.float64), 256, 1)
        return d * np.repeat(f.sc, 32, 1) * f.code - dm * np.repeat(f.m, 32, 1)
    if wtype == synth.IQ1_M:
        d = np.repeat(f.d.astype(np.float64), 256, 1)
        s = np.repeat(f.s.astype(np.float64), 16, 1)
        delta = np.where(np.repeat(f.neg, 8, 1) == 1, -0.125, 0.125)
        return d * (2 * s + 1) * (f.g + delta)
    if wtype == synth.Q6_K:
        d = np.repeat(f.d.astype(np.float64), 256, 1)
        return d * np.repeat(f.sc.astype(np.float64), 16, 1) * (f.code.astype(np.float64) - 32)
    raise ValueError


def _term_magnitudes(wtype, f, q, d):
    """Dequantised f64 weights and activations, and sum over groups of the magnitudes of every f32
    product the blockwise sum forms (the scale of the f32 summation error bound)."""
    W = _dequant_f64(wtype, f)
    xh = np.repeat(d.astype(np.float64), 32, 1) * q
    M, K = q.shape
    G = 16 if wtype in (synth.IQ1_M, synth.Q6_K) else 32
    mags = np.zeros((M, W.shape[0]))
    if wtype == synth.Q4_K:
        pos = np.repeat(f.d.astype(np.float64), 256, 1) * np.repeat(f.sc, 32, 1) * f.code
        neg = np.repeat(f.dmin.astype(np.float64), 256, 1) * np.repeat(f.m, 32, 1)
        for g0 in range(0, K, 32):
            mags += np.abs(xh[:, g0:g0 + 32] @ pos[:, g0:g0 + 32].T)
            mags += np.abs(xh[:, g0:g0 + 32] @ neg[:, g0:g0 + 32].T)
    else:
        for g0 in range(0, K, G):
            mags += np.abs(xh[:, g0:g0 + G] @ W[:, g0:g0 + G].T)
    return W, xh, mags


@pytest.mark.parametrize("wtype", [synth.Q8_0, synth.Q4_0, synth.Q4_K, synth.IQ1_M, synth.Q6_K])
@pytest.mark.parametrize("shape", [(3, 5, 256), (17, 9, 1024)])
def test_blockwise_matches_f64_dequant_matmul(wtype, shape):
    M, N, K = shape
    g = np.random.default_rng(100 + wtype)
    f = synth.draw_fields(g, wtype, N, K)
    W = synth.pack(wtype, f)
    x = synth.activations(g, M, K)
    q, d, s = oracle.quantize_q8_1(x)
    out = oracle.gemm(wtype, W, q, d, s, N)
    Wd, xh, mags = _term_magnitudes(wtype, f, q, d)
    ref = xh @ Wd.T
    G = 16 if wtype in (synth.IQ1_M, synth.Q6_K) else 32
    # per group: scale product, product with I, (Q4_K: min product, stored s, difference), then the
    # running sum -- at most K/G + 4 roundings of 2^-24 against the sum of product magnitudes
    bound = (K // G + 4) * 2.0 ** -24 * mags
    err = np.abs(out.astype(np.float64) - ref)
    assert np.all(err <= bound + 1e-30), (err / (bound + 1e-30)).max()
    # and the result is not trivially small: the bound is far below the output scale
    assert bound.max() < 1e-4 * np.abs(ref).max()


@pytest.mark.parametrize("wtype", [synth.Q8_0, synth.Q4_0, synth.IQ1_M, synth.Q6_K])
def test_blockwise_with_unit_scales_is_integer_matmul(wtype):
    # d = 1 for weights and activations: every block term is its integer dot, so the product is the
    # plain integer matmul of the codes (exact in f32 here: |out| < 2^24).
    M, N, K = 4, 6, 512
    g = np.random.default_rng(40 + wtype)
    f = synth.draw_fields(g, wtype, N, K)
    f.d[...] = np.float16(1.0)
    if wtype == synth.IQ1_M:
        f.s[...] = 0          # (2s+1)/8 = 1/8 per 16: scale 1/8, integer values 8g+-1 -> out = dot/8
    if wtype == synth.Q6_K:
        f.sc[...] = 1         # d * sc = 1 per 16: integer values code - 32
    W = synth.pack(wtype, f)
    q = g.integers(-127, 128, size=(M, K)).astype(np.int8)
    d = np.ones((M, K // 32), np.float32)
    s = np.zeros((M, K // 32), np.float32)
    out = oracle.gemm(wtype, W, q, d, s, N)
    if wtype == synth.Q8_0:
        wint = f.q.astype(np.int64)
    elif wtype == synth.Q4_0:
        wint = f.code.astype(np.int64) - 8
    elif wtype == synth.Q6_K:
        wint = f.code.astype(np.int64) - 32
    else:
        wint = 8 * f.g.astype(np.int64) + np.where(np.repeat(f.neg, 8, 1) == 1, -1, 1)
    ref = q.astype(np.int64) @ wint.T
    if wtype == synth.IQ1_M:
        assert np.array_equal(out.astype(np.float64) * 8, ref.astype(np.float64))
    else:
        assert np.array_equal(out.astype(np.float64), ref.astype(np.float64))


def test_gemm_rows_is_a_row_subset_of_gemm():
    M, N, K = 9, 7, 512
    g = np.random.default_rng(5)
    f = synth.draw_fields(g, synth.Q4_K, N, K)
    W = synth.pack(synth.Q4_K, f)
    q, d, s = oracle.quantize_q8_1(synth.activations(g, M, K))
    full = oracle.gemm(synth.Q4_K, W, q, d, s, N)
    rows = [8, 0, 3]
    assert np.array_equal(oracle.gemm_rows(synth.Q4_K, W, q, d, s, N, rows), full[rows])


# ---------------------------------------------------------------------------------- W8A8
def test_w8a8_unit_scales_small_values_are_exact_integers():
    g = np.random.default_rng(8)
    M, N, K = 6, 5, 64
    X = g.integers(-2, 3, size=(M, K)).astype(np.int8)
    W = g.integers(-1, 2, size=(N, K)).astype(np.int8)
    out = oracle.w8a8(W, np.ones(N, np.float32), X, np.ones(M, np.float32))
    ref = X.astype(np.int64) @ W.T.astype(np.int64)           # |ref| <= 128: exact in bf16
    got = (out.astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(got.astype(np.int64), ref)


def test_w8a8_within_bf16_rounding_of_exact_product():
    g = np.random.default_rng(9)
    M, N, K = 7, 9, 4096
    X = g.integers(-127, 128, size=(M, K)).astype(np.int8)
    W = g.integers(-127, 128, size=(N, K)).astype(np.int8)
    xs = g.uniform(1e-3, 1e-2, M).astype(np.float32)
    ws = g.uniform(1e-3, 1e-2, N).astype(np.float32)
    out = oracle.w8a8(W, ws, X, xs)
    got = (out.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    exact = (X.astype(np.int64) @ W.T.astype(np.int64)) * xs[:, None].astype(np.float64) * ws[None].astype(np.float64)
    assert np.all(np.abs(got - exact) <= np.abs(exact) * (2.0 ** -8 + 2.0 ** -21))
    # worst-case |I| stays inside int32 for K = 4096 (page: int32 accumulation over the full K)
    assert 4096 * 127 * 127 < 2 ** 31


# ---------------------------------------------------------------------------------- MoE routing
def test_gemm_id_reduces_to_dense_product_per_expert():
    g = np.random.default_rng(12)
    E, M, N, K, slots = 5, 11, 7, 512, 3
    f = synth.draw_fields(g, synth.IQ1_M, E * N, K)
    W = synth.pack(synth.IQ1_M, f)
    q, d, s = oracle.quantize_q8_1(synth.activations(g, M, K))
    ids = synth.route(g, M, E, slots)
    out = oracle.gemm_id(synth.IQ1_M, W, E, q, d, s, ids, N)
    per_expert = [oracle.gemm(synth.IQ1_M, W.reshape(E, N, -1)[e], q, d, s, N) for e in range(E)]
    for t in range(M):
        for j in range(slots):
            assert np.array_equal(out[t, j], per_expert[ids[t, j]][t])


def test_gemm_id_invariant_under_expert_relabeling():
    g = np.random.default_rng(13)
    E, M, N, K, slots = 4, 6, 5, 256, 2
    f = synth.draw_fields(g, synth.Q4_0, E * N, K)
    W = synth.pack(synth.Q4_0, f).reshape(E, N, -1)
    q, d, s = oracle.quantize_q8_1(synth.activations(g, M, K))
    ids = synth.route(g, M, E, slots)
    perm = np.array([2, 0, 3, 1])
    W2 = np.empty_like(W)
    W2[perm] = W                      # expert e now stored at slot perm[e]
    out1 = oracle.gemm_id(synth.Q4_0, W.reshape(E * N, -1), E, q, d, s, ids, N)
    out2 = oracle.gemm_id(synth.Q4_0, W2.reshape(E * N, -1), E, q, d, s, perm[ids].astype(np.int32), N)
    assert np.array_equal(out1, out2)


def test_gemm_id_rejects_out_of_range_ids():
    q = np.zeros((2, 256), np.int8)
    d = np.zeros((2, 8), np.float32)
    W = np.zeros((2 * 3, 8 * 18), np.uint8)
    with pytest.raises(ValueError):
        oracle.gemm_id(synth.Q4_0, W, 2, q, d, d, np.array([[0], [2]], np.int32), 3)
