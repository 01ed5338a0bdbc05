"""The seeded input generator: definition, determinism and distribution (CPU only)."""
import numpy as np

import synth


def test_splitmix64_reference_vector():
    # SplitMix64 started at state 1234567: the first outputs of the published
    # reference generator (Vigna's splitmix64.c test vector).
    expect = [6457827717110365317, 3203168211198807973, 9817491932198370423,
              4593380528125082431, 16408922859458223821]
    got = [synth.splitmix64_at(1234567, n) for n in range(1, 6)]
    assert got == expect


def test_c_matches_numpy_restatement():
    for (seed, stream, first, count, sigma) in [(1000, 0, 0, 4097, 1.0), (7, 2, 12345, 999, 4.0)]:
        c = synth.normal_bf16(seed, stream, (count,), sigma=sigma, first=first)
        n = synth.normal_bf16_numpy(seed, stream, count, sigma=sigma, first=first)
        # libm and numpy may differ in the last bit of log/sin/cos; bf16 rounding
        # hides that except on the rare value sitting on a rounding boundary
        assert np.mean(c != n) < 1e-3
        assert np.max(np.abs(synth.bf16_to_f32(c) - synth.bf16_to_f32(n))) <= 2.0 ** -7 * 8 * sigma


def test_slices_are_independent_of_offset():
    full = synth.normal_bf16(3, 1, (10000,))
    part = synth.normal_bf16(3, 1, (3001,), first=4321)
    assert np.array_equal(full[4321:4321 + 3001], part)


def test_distribution_and_streams():
    x = synth.bf16_to_f32(synth.normal_bf16(1001, 0, (1 << 20,))).astype(np.float64)
    assert abs(x.mean()) < 5e-3 and abs(x.std() - 1.0) < 5e-3
    y = synth.bf16_to_f32(synth.normal_bf16(1001, 1, (1 << 20,))).astype(np.float64)
    assert abs(np.corrcoef(x, y)[0, 1]) < 5e-3
    z = synth.bf16_to_f32(synth.normal_bf16(5, 0, (1 << 18,), sigma=4.0)).astype(np.float64)
    assert abs(z.std() - 4.0) < 0.03


def test_bf16_rounding_is_nearest_even():
    vals = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9, -2.5, 0.0], dtype=np.float32)
    bits = synth.f32_to_bf16_bits(vals)
    back = synth.bf16_to_f32(bits)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: even mantissa wins (1.0)
    assert back.tolist() == [1.0, 1.0, 1.0 + 2 ** -6, 1.0, -2.5, 0.0]


def test_workload_recipes():
    w = synth.WORKLOADS["long_8192_d128"]
    assert w.flops == 4.0 * 4 * 32 * 8192 * 8192 * 128
    assert synth.WORKLOADS["long_8192_d128_causal"].flops == w.flops / 2
    s = synth.WORKLOADS["stress_32000_d128_causal"]
    assert (s.B, s.H, s.Nq, s.d, s.causal, s.sigma_q) == (1, 16, 32000, 128, True, 4.0)
    small = synth.WORKLOADS["single_head_256_d64"]
    q, k, v = small.make()
    assert q.shape == (1, 1, 256, 64) and q.dtype == np.uint16
    q2, _, _ = small.make()
    assert np.array_equal(q, q2)
