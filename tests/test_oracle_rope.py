"""Pins of the oracle's rotary position embedding (RoPE) that precedes the
FP8 quantiser (FlashAttention-3 deep-reading report §2.2 / §3.3: the block
quantisation fused into the memory-bound rotary-embedding kernel; RoPE as in
Su et al., "RoFormer", 2021).

* closed forms: a zero angle is the identity, a quarter turn maps the pair
  (a, b) to (-b, a) -- with both pair layouts, so a swapped layout, a wrong
  sign or a table indexed by the wrong axis fails;
* a different formulation: the complex product (a + ib)(cos + i sin) in
  float64, within the binary32 rounding bound of the oracle's evaluation;
* the two pair layouts are a column permutation of one another;
* the defining property: the dot product of a rotated query at position m
  and a rotated key at position n depends on m - n only, and equals the
  plain dot product at m = n;
* the FP8 prep with RoPE quantises exactly the RoPE'd values, and with the
  Hadamard rotation their rotated image.
"""
import numpy as np
import pytest

import oracle
from exact_attention_71_gb300 import synth


def _x(shape, seed=1):
    return synth.tensor_bf16(shape, seed=seed, stream=1)


@pytest.mark.parametrize("interleaved", [False, True])
def test_zero_angle_is_identity(interleaved):
    x = _x((2, 9, 3, 16))
    c = np.ones((9, 8), np.float32)
    s = np.zeros((9, 8), np.float32)
    r = oracle.rope(x, c, s, interleaved)
    np.testing.assert_array_equal(r, synth.bf16_bits_to_f32(x))


@pytest.mark.parametrize("interleaved", [False, True])
def test_quarter_turn_on_one_token(interleaved):
    """Token 3 turns by 90 degrees, every other token by 0."""
    B, N, H, d = 1, 6, 2, 8
    x = _x((B, N, H, d), seed=4)
    c = np.ones((N, d // 2), np.float32)
    s = np.zeros((N, d // 2), np.float32)
    c[3], s[3] = 0.0, 1.0
    r = oracle.rope(x, c, s, interleaved)
    xf = synth.bf16_bits_to_f32(x)
    want = xf.copy()
    for i in range(d // 2):
        ia, ib = (2 * i, 2 * i + 1) if interleaved else (i, i + d // 2)
        want[:, 3, :, ia] = -xf[:, 3, :, ib]
        want[:, 3, :, ib] = xf[:, 3, :, ia]
    np.testing.assert_array_equal(r, want)


@pytest.mark.parametrize("d", [8, 64, 128])
def test_matches_complex_product_within_binary32_rounding(d):
    B, N, H = 2, 50, 3
    x = _x((B, N, H, d), seed=d)
    c, s = synth.rope_tables(N, d)
    r = oracle.rope(x, c, s, interleaved=False).astype(np.float64)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    z = xf[..., : d // 2] + 1j * xf[..., d // 2:]
    w = c.astype(np.float64) + 1j * s.astype(np.float64)          # (N, d/2)
    exact = z * w[None, :, None, :]
    # each product and the sum rounded once: at most 2^-24 (|ac| + |bs|) twice
    bound_re = 2.0 ** -23 * (np.abs(z.real * w.real[None, :, None]) + np.abs(z.imag * w.imag[None, :, None]))
    bound_im = 2.0 ** -23 * (np.abs(z.real * w.imag[None, :, None]) + np.abs(z.imag * w.real[None, :, None]))
    assert np.all(np.abs(r[..., : d // 2] - exact.real) <= bound_re)
    assert np.all(np.abs(r[..., d // 2:] - exact.imag) <= bound_im)


def test_layouts_are_a_column_permutation():
    B, N, H, d = 1, 20, 2, 32
    x_int = _x((B, N, H, d), seed=7)
    order = np.concatenate([np.arange(0, d, 2), np.arange(1, d, 2)])   # half-split column k <- interleaved order[k]
    x_half = np.ascontiguousarray(x_int[..., order])
    c, s = synth.rope_tables(N, d)
    r_int = oracle.rope(x_int, c, s, interleaved=True)
    r_half = oracle.rope(x_half, c, s, interleaved=False)
    np.testing.assert_array_equal(r_half, r_int[..., order])


def test_scores_depend_on_relative_position_only():
    """The same query row at every position and the same key row at every
    position: <RoPE(q)_m, RoPE(k)_n> is a function of m - n, and at m = n it
    is the plain <q, k>."""
    N, d = 64, 64
    q1 = _x((1, 1, 1, d), seed=11)
    k1 = _x((1, 1, 1, d), seed=12)
    q = np.repeat(q1, N, axis=1)
    k = np.repeat(k1, N, axis=1)
    c, s = synth.rope_tables(N, d)
    rq = oracle.rope(q, c, s)[0, :, 0].astype(np.float64)
    rk = oracle.rope(k, c, s)[0, :, 0].astype(np.float64)
    S = rq @ rk.T
    qf = synth.bf16_bits_to_f32(q1).ravel().astype(np.float64)
    kf = synth.bf16_bits_to_f32(k1).ravel().astype(np.float64)
    tol = 2e-5 * np.linalg.norm(qf) * np.linalg.norm(kf)
    assert np.max(np.abs(np.diag(S) - qf @ kf)) <= tol
    for delta in (-17, -1, 1, 5, 30):
        diag = np.diagonal(S, offset=delta)
        assert np.max(np.abs(diag - diag[0])) <= tol
    # and it does depend on the offset
    assert abs(S[10, 0] - S[10, 10]) > 1e3 * tol


@pytest.mark.parametrize("interleaved", [False, True])
def test_rope_rows_keep_their_norm(interleaved):
    x = _x((2, 40, 2, 64), seed=3)
    c, s = synth.rope_tables(40, 64, base=500.0)
    r = oracle.rope(x, c, s, interleaved).astype(np.float64)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    n0, n1 = np.linalg.norm(xf, axis=-1), np.linalg.norm(r, axis=-1)
    assert np.max(np.abs(n1 - n0) / n0) < 1e-6


def test_fp8_prep_quantises_the_rope_values():
    B, N, H, d = 1, 300, 2, 64
    x = synth.tensor_bf16((B, N, H, d), seed=5, stream=2, outliers=True)
    c, s = synth.rope_tables(N, d)
    want = oracle.rope(x, c, s, interleaved=True)
    _, _, rot = oracle.fp8_quantize(x, oracle.MODE_BLOCK, rope=(c, s, True), return_rotated=True)
    np.testing.assert_array_equal(rot, want)
    M = oracle.rotation_matrix(d, 99)
    _, _, rot_h = oracle.fp8_quantize(x, oracle.MODE_BLOCK_HADAMARD, seed=99, rope=(c, s, True),
                                      return_rotated=True)
    ref = np.einsum("bnhc,ce->bnhe", want.astype(np.float64), M)
    assert np.max(np.abs(rot_h - ref)) <= 2.0 ** -23 * np.max(np.abs(ref))
    # and the codes are those of the plain quantiser applied to the RoPE'd values
    codes, scales = oracle.fp8_quantize(x, oracle.MODE_BLOCK, rope=(c, s, True))
    for blk in range(scales.shape[2]):
        sl = slice(blk * 128, min(N, (blk + 1) * 128))
        for h in range(H):
            amax = np.float32(np.max(np.abs(want[0, sl, h])))
            assert scales[0, h, blk] == np.float32(amax / np.float32(448.0))
            y = (want[0, sl, h] / scales[0, h, blk]).astype(np.float32)
            np.testing.assert_array_equal(codes[0, sl, h], oracle.e4m3_encode(y.astype(np.float64)).reshape(y.shape))


def test_rope_refused_for_values_and_bad_tables():
    x = _x((1, 8, 1, 16))
    c, s = synth.rope_tables(8, 16)
    with pytest.raises(ValueError):
        oracle.fp8_quantize(x, oracle.MODE_BLOCK, is_v=True, rope=(c, s, False))
    with pytest.raises(ValueError):
        oracle.fp8_quantize(x, oracle.MODE_BLOCK, rope=(c[:4], s[:4], False))
