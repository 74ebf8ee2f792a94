"""Pins of the oracle's sparse MLA decode attention (GLM-5.2 shared-Indexer KV
Cache Offload page §2.1; TokenSpeed engine audit, MLA section: one latent row
serves as K and V) against closed forms."""
import math

import numpy as np

from oracle import bf16_bits_to_f64, round_to_bf16_bits, sfa_decode


def _bits(x):
    """float values exactly representable in bf16 -> bit patterns."""
    f = np.asarray(x, dtype=np.float32)
    b = (f.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal((b.astype(np.uint32) << 16).view(np.float32), f)
    return b


def _rand_bf16(rng, shape):
    f = rng.standard_normal(shape).astype(np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def test_constant_rows_give_the_row():
    rng = np.random.default_rng(1)
    row = _rand_bf16(rng, (1, 576))
    rows = np.repeat(row, 37, axis=0)
    q = _rand_bf16(rng, (5, 576))
    scale = 1 / math.sqrt(576)
    out, lse = sfa_decode(q, rows, scale)
    v = bf16_bits_to_f64(row[0, :512])
    assert np.array_equal(out, np.broadcast_to(v, out.shape))
    s = scale * (bf16_bits_to_f64(q) @ bf16_bits_to_f64(row[0]))
    assert np.allclose(lse, s + math.log(37), rtol=0, atol=1e-12)


def test_single_row():
    rng = np.random.default_rng(2)
    rows = _rand_bf16(rng, (1, 576))
    q = _rand_bf16(rng, (3, 576))
    out, lse = sfa_decode(q, rows, 0.3)
    assert np.array_equal(out, np.broadcast_to(bf16_bits_to_f64(rows[0, :512]), out.shape))


def test_two_rows_sigmoid_weights():
    # q = a e_0, K_0[0] = x0, K_1[0] = x1, other dims of the rope part free:
    # s_j = scale a x_j, so row 0 gets weight sigmoid(scale a (x0 - x1)).
    rng = np.random.default_rng(3)
    rows_f = np.zeros((2, 576), np.float32)
    rows_f[:, 1:] = rng.standard_normal((2, 575)).astype(np.float32)
    rows_f[0, 0], rows_f[1, 0] = 1.5, -0.5
    rows_f = (((rows_f.view(np.uint32) >> 16) << 16)).view(np.float32)
    q_f = np.zeros((1, 576), np.float32)
    q_f[0, 0] = 2.0
    scale = 0.75
    out, lse = sfa_decode(_bits(q_f), _bits(rows_f), scale)
    w0 = 1.0 / (1.0 + math.exp(-scale * 2.0 * (1.5 - (-0.5))))
    want = w0 * rows_f[0, :512].astype(np.float64) + (1 - w0) * rows_f[1, :512].astype(np.float64)
    assert np.allclose(out[0], want, rtol=1e-14, atol=1e-15)
    want_lse = math.log(math.exp(scale * 3.0) + math.exp(scale * -1.0))
    assert abs(lse[0] - want_lse) < 1e-14


def test_row_permutation_invariance_and_zero_scale():
    rng = np.random.default_rng(4)
    rows = _rand_bf16(rng, (64, 576))
    q = _rand_bf16(rng, (8, 576))
    out, lse = sfa_decode(q, rows, 1 / 24)
    perm = rng.permutation(64)
    out2, lse2 = sfa_decode(q, rows[perm], 1 / 24)
    assert np.allclose(out, out2, rtol=1e-12, atol=1e-14)
    assert np.allclose(lse, lse2, rtol=1e-13, atol=1e-13)
    out0, _ = sfa_decode(q, rows, 0.0)
    mean = bf16_bits_to_f64(rows[:, :512]).mean(axis=0)
    assert np.allclose(out0, np.broadcast_to(mean, out0.shape), rtol=1e-13, atol=1e-15)


def test_round_to_bf16_ties_to_even():
    x = np.array([1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8 + 2 ** -30),
                  3.0, 0.0, -2.5], dtype=np.float64)
    got = round_to_bf16_bits(x).tolist()
    # 1+2^-8 is half way between 1 and 1+2^-7: even (1.0) wins; 1+3*2^-8 is
    # half way between 1+2^-7 and 1+2^-6: even (1+2^-6) wins; just past the
    # half way point rounds away.
    assert got == [0x3F80, 0x3F80, 0x3F82, 0xBF81, 0x4040, 0x0000, 0xC020]
    # a value that float32 would round first and then round again differently
    y = 1 + 2 ** -8 + 2 ** -40       # -> float32 gives 1+2^-8 (tie) -> 1.0; direct: up
    assert round_to_bf16_bits(np.array([y]))[0] == 0x3F81
