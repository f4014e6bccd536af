"""The seeded input generator: determinism, slicing, distributions and the 4-bit encoding."""
import math

import numpy as np

import oracle
import synth


def test_stream_is_deterministic_and_sliceable():
    a = synth.normal_f64(0, 3, 0, 5000)
    b = synth.normal_f64(0, 3, 0, 5000)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(synth.normal_f64(0, 3, 1234, 100), a[1234:1334])
    assert not np.array_equal(synth.normal_f64(1, 3, 0, 100), a[:100])
    assert not np.array_equal(synth.normal_f64(0, 4, 0, 100), a[:100])
    # threaded generation (large count) equals the serial one
    big = synth.normal_f64(7, 1, 0, 300_000)
    np.testing.assert_array_equal(big[200_000:200_100], synth.normal_f64(7, 1, 200_000, 100))


def test_normal_moments():
    z = synth.normal_f64(0, 1, 0, 1_000_000)
    assert abs(z.mean()) < 5e-3 and abs(z.std() - 1) < 5e-3
    assert abs(np.mean(z ** 4) - 3.0) < 0.05
    w = synth.normal_f32(0, 2, 0, 200_000, 0.0, 0.02)
    assert abs(w.std() - 0.02) < 2e-4


def test_bf16_rounding_nearest_even():
    vals = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 1e-40, 3.0e38])
    bits = synth.round_bf16(vals)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7 -> even (1.0); 1 + 3*2^-8 -> 1 + 2^-6 (even)
    assert bits[0] == 0x3F80 and bits[1] == 0x3F80 and bits[2] == 0x3F82 and bits[3] == 0xC020
    got = oracle.bf16_to_f64(bits)
    assert bits[4] == 0x0001 and got[4] == 2.0 ** -133     # subnormal: nearest multiple of 2^-133
    np.testing.assert_array_equal(synth.normal_bf16(0, 1, 0, 64), synth.round_bf16(synth.normal_f64(0, 1, 0, 64)))


def test_mxfp4_encoding_is_a_faithful_rounding():
    std = 1 / 64
    codes, scales = synth.mxfp4_blocks(0, 3, 0, 4000, std)
    w = synth.normal_f64(0, 3, 0, 4000 * 32, 0.0, std).reshape(4000, 32)
    dec = oracle.mxfp4_decode(codes.reshape(4000, 16), scales.reshape(4000, 1))
    amax = np.abs(w).max(axis=1)
    e = scales.astype(np.int64) - 127
    ratio = amax / np.ldexp(1.0, e)
    assert np.all((ratio >= 4.0) & (ratio < 8.0))            # shared exponent = floor(log2 amax) - 2
    q = w / np.ldexp(1.0, e)[:, None]
    qd = dec / np.ldexp(1.0, e)[:, None]
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    a = np.minimum(np.abs(q), 6.0)                            # saturate at the largest magnitude
    best = np.abs(a[..., None] - grid).min(-1)
    assert np.all(np.abs(np.abs(qd) - a) <= best + 1e-12)     # the chosen code is a nearest one
    assert np.all(np.isin(np.abs(qd), grid))
    assert np.all((np.sign(qd) == np.sign(q)) | (qd == 0))


def test_workloads_shapes_and_slices():
    w = synth.workload("tiny")
    x = w.x()
    assert x.shape == (16, 256) and x.dtype == np.uint16
    ex = w.experts()
    assert ex.gate.shape == (8, 512, 256) and ex.down.shape == (8, 256, 512)
    part = w.expert_slice(3, 5)
    np.testing.assert_array_equal(part.gate, ex.gate[3:5])
    np.testing.assert_array_equal(part.down, ex.down[3:5])
    v = synth.workload("verify")
    xv = oracle.bf16_to_f64(v.x())
    assert xv.shape == (48, 4096)
    # rows of one sequence are close to each other (x_seq + 0.1 noise), other sequences are not
    d_same = np.linalg.norm(xv[0] - xv[1]) / math.sqrt(4096)
    d_other = np.linalg.norm(xv[0] - xv[6]) / math.sqrt(4096)
    assert d_same < 0.2 and d_other > 1.0
    fz = synth.workload("fp4_zipf")
    b = fz.router_bias()
    assert b[0] == 0 and abs(b[1] + 1.1 * math.log(2)) < 1e-6
    sl = fz.expert_slice(5, 6)
    assert sl.gate.shape == (1, 1024, 2048) and sl.gate_scale.shape == (1, 1024, 128)
