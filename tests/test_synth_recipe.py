"""The seeded input generator follows the stated recipe (no GPU needed): workload shapes and seeds, the
value range and spread of every drawn field, N(0,1) activations, distinct uniformly drawn expert ids per
token, and determinism by seed.  Both the oracle and the CUDA path read these inputs; the generator holds
none of the method's arithmetic."""
import numpy as np

from block_quantized_int8_q8_gb300 import synth

F16_LO, F16_HI = np.float16(1e-3), np.float16(1e-2)   # the scale range after rounding to f16


def test_workload_shapes_and_seeds():
    want = {"q8_0_tiny": (synth.Q8_0, 64, 256, 1024), "q4_0_7b": (synth.Q4_0, 2048, 4096, 4096),
            "q4_k_ffn_up": (synth.Q4_K, 2048, 11008, 4096), "w8a8_m3072": (synth.W8A8, 3072, 1536, 4096),
            "w8a8_m4096": (synth.W8A8, 4096, 1536, 4096), "iq1_m_moe": (synth.IQ1_M, 512, 1536, 4096),
            "iq1_m_dense": (synth.IQ1_M, 512, 4096, 4096), "q6_k_ffn_down": (synth.Q6_K, 2048, 4096, 11008)}
    assert set(synth.WORKLOADS) == set(want)
    for name, (wt, M, N, K) in want.items():
        w = synth.WORKLOADS[name]
        assert (w["wtype"], w["M"], w["N"], w["K"]) == (wt, M, N, K), name
    assert synth.WORKLOADS["iq1_m_moe"]["experts"] == 64 and synth.WORKLOADS["iq1_m_moe"]["slots"] == 8
    seeds = [w["seed"] for w in synth.WORKLOADS.values()]
    assert len(set(seeds)) == len(seeds) and all(1000 < s < 1100 for s in seeds)


def _spans(a, lo, hi):
    return a.min() == lo and a.max() == hi and len(np.unique(a)) == hi - lo + 1


def _scales_ok(d):
    d = np.asarray(d, dtype=np.float16)
    return d.min() >= F16_LO and d.max() <= F16_HI and d.max() > d.min()


def test_field_ranges_per_type():
    g = synth.rng(5)
    N, K = 64, 1024
    f = synth.draw_fields(g, synth.Q8_0, N, K)
    assert _spans(f.q.astype(int), -127, 127) and _scales_ok(f.d)
    f = synth.draw_fields(g, synth.Q4_0, N, K)
    assert _spans(f.code.astype(int), 0, 15) and _scales_ok(f.d)
    f = synth.draw_fields(g, synth.Q4_K, N, K)
    assert _spans(f.code.astype(int), 0, 15) and _spans(f.sc.astype(int), 0, 63) and _spans(f.m.astype(int), 0, 63)
    assert _scales_ok(f.d) and _scales_ok(f.dmin)
    f = synth.draw_fields(g, synth.IQ1_M, N, K)
    assert _spans(f.g.astype(int), -1, 1) and _spans(f.s.astype(int), 0, 7) and _spans(f.neg.astype(int), 0, 1)
    assert f.neg.shape == (N, K // 8) and f.s.shape == (N, K // 16) and _scales_ok(f.d)
    counts = np.bincount(f.g.reshape(-1) + 1, minlength=3) / f.g.size
    assert np.all(np.abs(counts - 1 / 3) < 0.01)            # g uniform over {-1, 0, 1}
    f = synth.draw_fields(g, synth.Q6_K, N, K)
    assert _spans(f.code.astype(int), 0, 63) and _spans(f.sc.astype(int), -128, 127) and _scales_ok(f.d)
    f = synth.draw_fields(g, synth.W8A8, N, K)
    assert _spans(f.W.astype(int), -127, 127)
    assert f.ws.dtype == np.float32 and f.ws.min() >= 1e-3 and f.ws.max() <= 1e-2
    X, xs = synth.w8a8_acts(g, 32, K)
    assert _spans(X.astype(int), -127, 127) and xs.min() >= 1e-3 and xs.max() <= 1e-2


def test_activations_are_standard_normal_f32():
    x = synth.activations(synth.rng(6), 256, 4096)
    assert x.dtype == np.float32 and x.shape == (256, 4096)
    assert abs(float(x.mean())) < 0.01 and abs(float(x.std()) - 1.0) < 0.01


def test_routing_distinct_in_range_uniform_and_seeded():
    M, E, slots = 4096, 64, 8
    ids = synth.route(synth.rng(7), M, E, slots)
    assert ids.dtype == np.int32 and ids.shape == (M, slots)
    assert ids.min() >= 0 and ids.max() < E
    assert all(len(set(r)) == slots for r in ids)            # distinct experts per token
    use = np.bincount(ids.reshape(-1), minlength=E)
    expect = M * slots / E
    assert np.all(np.abs(use - expect) < 6 * np.sqrt(expect))  # uniform usage (loose bound)
    assert np.array_equal(ids, synth.route(synth.rng(7), M, E, slots))


def test_problems_are_deterministic_by_seed():
    a = synth.make_problem(synth.Q4_K, 8, 32, 512, seed=11)
    b = synth.make_problem(synth.Q4_K, 8, 32, 512, seed=11)
    c = synth.make_problem(synth.Q4_K, 8, 32, 512, seed=12)
    assert np.array_equal(a.W, b.W) and np.array_equal(a.x, b.x)
    assert not np.array_equal(a.W, c.W)
    m = synth.make_problem(synth.IQ1_M, 6, 16, 256, seed=13, experts=5, slots=3)
    assert m.W.shape[0] == 5 * 16 and m.ids.shape == (6, 3) and m.experts == 5
