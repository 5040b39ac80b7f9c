"""Pins of the oracle's FP8 pieces: the OCP E4M3 encoder, the splitmix64 signs,
the Hadamard rotation and the block quantiser.

* E4M3: the special values of the OCP OFP8 specification (golden file),
  torch's own float8_e4m3fn conversion as an independent library routine
  (decode of all 256 codes; round-to-nearest-even encode of every value in
  the finite range), exhaustive round trips, ties to even, saturation.
* signs: the published splitmix64 reference outputs for state 0.
* rotation: the textbook Sylvester H_4 (golden file), M M^T = I.
* quantiser: the error bound of E4M3 rounding, scale = amax / 448, the
  rotation equals a numpy matrix product.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from exact_attention_71_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def test_e4m3_special_values_from_ocp_spec():
    for val, bits in _golden_rows("e4m3_ocp.txt"):
        code = int(bits.replace(".", ""), 2)
        dec = oracle.e4m3_decode([code])[0]
        if val == "nan":
            assert np.isnan(dec)
            continue
        v = float(val)
        assert dec == v and np.signbit(dec) == np.signbit(v)
        assert oracle.e4m3_encode([v])[0] == code


def test_e4m3_decode_matches_torch_for_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])


def test_e4m3_round_trip_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle.e4m3_decode(codes)
    back = oracle.e4m3_encode(vals)
    finite = ~np.isnan(vals)
    assert np.array_equal(back[finite], codes[finite])
    assert np.all((back[~finite] & 0x7F) == 0x7F)


def test_e4m3_encode_matches_torch_rne_in_range():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(200000) * np.exp2(rng.uniform(-12, 9, 200000)),
        rng.uniform(-463.9, 463.9, 50000),
    ])
    x = x[np.abs(x) < 464.0]
    # every midpoint between neighbouring finite codes: the tie cases
    vals = np.unique(oracle.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8)))
    mids = (vals[:-1] + vals[1:]) / 2
    x = np.concatenate([x, mids, -mids]).astype(np.float32).astype(np.float64)
    ours = oracle.e4m3_encode(x)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_ties_go_to_even_mantissa():
    vals = oracle.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))
    for a, b in zip(vals[:-1], vals[1:]):
        code = oracle.e4m3_encode([(a + b) / 2])[0]
        assert code & 1 == 0


def test_e4m3_saturates_and_keeps_nan():
    out = oracle.e4m3_encode([448.0, 449.0, 480.0, 1e30, np.inf, -1e5, -np.inf])
    assert list(out) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]
    assert oracle.e4m3_encode([np.nan])[0] & 0x7F == 0x7F


def test_splitmix64_signs_follow_reference_outputs():
    outs = [int(r[0], 16) for r in _golden_rows("splitmix64_seed0.txt")]
    want = [-1.0 if (o >> 63) else 1.0 for o in outs]
    assert list(oracle.signs(3, 0)) == want
    s = oracle.signs(256, 99)
    assert set(np.unique(s)) <= {-1.0, 1.0}
    assert 80 < (s > 0).sum() < 176
    assert not np.array_equal(oracle.signs(64, 1), oracle.signs(64, 2))


def test_rotation_is_sign_flip_times_sylvester():
    H4 = np.array([[float(x) for x in r] for r in _golden_rows("hadamard_sylvester.txt")])
    s = oracle.signs(4, 7)
    M = oracle.rotation_matrix(4, 7)
    np.testing.assert_array_equal(M * 2.0, np.diag(s) @ H4)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_rotation_is_orthogonal(d):
    M = oracle.rotation_matrix(d, 12345)
    assert np.max(np.abs(M @ M.T - np.eye(d))) < 1e-15
    assert np.allclose(np.abs(M), 1 / np.sqrt(d), rtol=0, atol=1e-17)


def test_block_quantiser_scale_and_error_bound():
    x = synth.tensor_bf16((2, 300, 3, 64), seed=1, stream=1, outliers=True)
    codes, scales = oracle.fp8_quantize(x, oracle.MODE_BLOCK)
    assert scales.shape == (2, 3, 3)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    deq = oracle.e4m3_decode(codes).reshape(x.shape)
    for b in range(2):
        for h in range(3):
            for blk in range(3):
                sl = slice(blk * 128, min(300, (blk + 1) * 128))
                xb = xf[b, sl, h]
                amax = np.max(np.abs(xb))
                assert scales[b, h, blk] == np.float32(np.float32(amax) / np.float32(448.0))
                err = np.abs(deq[b, sl, h] * scales[b, h, blk] - xb)
                # E4M3 rounding: half an ulp, 2^-4 relative for normals,
                # 2^-10 absolute (times the scale) in the subnormal range;
                # plus the rounding of x / scale to binary32.
                bound = np.maximum(np.abs(xb) * 2.0**-4, 2.0**-10 * scales[b, h, blk]) * (1 + 1e-6)
                assert np.all(err <= bound)
                # the block maximum lands on +-448 exactly
                assert np.max(np.abs(deq[b, sl, h])) == 448.0


def test_per_tensor_mode_shares_one_scale():
    x = synth.tensor_bf16((1, 260, 2, 64), seed=3, stream=2, outliers=True)
    _, scales = oracle.fp8_quantize(x, oracle.MODE_PER_TENSOR)
    amax = np.max(np.abs(synth.bf16_bits_to_f32(x)))
    assert np.all(scales == np.float32(amax / np.float32(448.0)))


def test_zero_block_gets_unit_scale():
    x = np.zeros((1, 130, 1, 64), dtype=np.uint16)
    codes, scales = oracle.fp8_quantize(x, oracle.MODE_BLOCK_HADAMARD, seed=5)
    assert np.all(scales == 1.0) and np.all(codes == 0)


def test_hadamard_mode_rotates_q_k_but_not_v():
    x = synth.tensor_bf16((1, 200, 2, 128), seed=4, stream=1)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    M = oracle.rotation_matrix(128, 77)
    _, _, rot = oracle.fp8_quantize(x, oracle.MODE_BLOCK_HADAMARD, seed=77, return_rotated=True)
    want = np.einsum("bnhc,ce->bnhe", xf, M)
    assert np.max(np.abs(rot - want)) <= 2.0**-23 * np.max(np.abs(want))
    _, _, rot_v = oracle.fp8_quantize(x, oracle.MODE_BLOCK_HADAMARD, seed=77, is_v=True,
                                      return_rotated=True)
    np.testing.assert_array_equal(rot_v, xf.astype(np.float32))


def test_rotation_spreads_outliers():
    """Incoherent processing lowers the block amax / rms ratio of an
    outlier-heavy block (deep-reading report §2.2)."""
    x = synth.tensor_bf16((1, 128, 1, 128), seed=0, stream=1, outliers=True)
    _, _, r0 = oracle.fp8_quantize(x, oracle.MODE_BLOCK, return_rotated=True)
    _, _, r1 = oracle.fp8_quantize(x, oracle.MODE_BLOCK_HADAMARD, seed=1, return_rotated=True)
    ratio = lambda r: np.max(np.abs(r)) / np.sqrt(np.mean(r.astype(np.float64) ** 2))
    assert ratio(r1) < ratio(r0)
