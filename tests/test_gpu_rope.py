"""RoPE fused into the FP8 prep (attn_fp8_prep_rope) against the oracle.

* Without the Hadamard rotation (modes 0 and 2) the codes and scales are
  bit-exact: both sides turn each pair in float32 with every product and sum
  rounded, and take the quantisation decision on the same binary32 values.
* With the rotation (mode 1), codes agree except at e4m3 rounding midpoints,
  as for the plain prep.
* End to end: the FP8 forward on RoPE-prepped Q and K against the fp64
  oracle on the RoPE'd values (FlashAttention-3 deep-reading report §4.3
  error metric).
"""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_71_gb300 import api, synth
from tests.helpers import FP8_LSE, FP8_RMS, assert_codes_match_up_to_midpoints, dequant, gpu_rows, lse_rows, to_dev

pytestmark = pytest.mark.gpu

SEED = 4321


def _tables(N, d, base=10000.0):
    c, s = synth.rope_tables(N, d, base)
    return c, s, torch.from_numpy(c).cuda(), torch.from_numpy(s).cuda()


def _prep(x, ct, st, mode, interleaved):
    codes, scales = api.attn_fp8_prep_rope(to_dev(x), ct, st, mode=mode, sign_seed=SEED, interleaved=interleaved)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy()


@pytest.mark.parametrize("shape", [(1, 300, 2, 64), (2, 256, 3, 128), (1, 130, 2, 256)])
@pytest.mark.parametrize("mode", [0, 2])
@pytest.mark.parametrize("interleaved", [False, True])
def test_rope_prep_bit_exact_without_rotation(shape, mode, interleaved):
    B, N, H, d = shape
    x = synth.tensor_bf16(shape, seed=6, stream=1, outliers=True)
    c, s, ct, st = _tables(N, d)
    c_gpu, s_gpu = _prep(x, ct, st, mode, interleaved)
    c_ref, s_ref = oracle.fp8_quantize(x, mode, seed=SEED, rope=(c, s, interleaved))
    np.testing.assert_array_equal(s_gpu, s_ref)
    np.testing.assert_array_equal(c_gpu, c_ref)


@pytest.mark.parametrize("shape", [(1, 300, 2, 64), (2, 256, 3, 128), (1, 130, 2, 256)])
@pytest.mark.parametrize("interleaved", [False, True])
def test_rope_prep_with_hadamard(shape, interleaved):
    B, N, H, d = shape
    x = synth.tensor_bf16(shape, seed=7, stream=2, outliers=True)
    c, s, ct, st = _tables(N, d, base=500.0)
    c_gpu, s_gpu = _prep(x, ct, st, api.MODE_BLOCK_HADAMARD, interleaved)
    c_ref, s_ref, rot = oracle.fp8_quantize(x, oracle.MODE_BLOCK_HADAMARD, seed=SEED, rope=(c, s, interleaved),
                                            return_rotated=True)
    np.testing.assert_allclose(s_gpu, s_ref, rtol=2e-6, atol=0)
    assert_codes_match_up_to_midpoints(c_gpu, c_ref, s_ref, rot)


@pytest.mark.parametrize("interleaved", [False, True])
def test_rope_with_zero_angles_equals_plain_prep(interleaved):
    """cos = 1, sin = 0: the RoPE prep gives the plain prep's codes and
    scales bit for bit; real angles change most codes."""
    x = synth.tensor_bf16((1, 256, 2, 128), seed=8, stream=1)
    xd = to_dev(x)
    one = torch.ones((256, 64), dtype=torch.float32, device="cuda")
    zero = torch.zeros((256, 64), dtype=torch.float32, device="cuda")
    for mode in (api.MODE_BLOCK, api.MODE_BLOCK_HADAMARD):
        c_id, s_id = api.attn_fp8_prep_rope(xd, one, zero, mode=mode, sign_seed=SEED, interleaved=interleaved)
        c_pl, s_pl = api.attn_fp8_prep(xd, mode=mode, sign_seed=SEED)
        torch.cuda.synchronize()
        assert torch.equal(c_id, c_pl) and torch.equal(s_id, s_pl)
    c, s, ct, st = _tables(256, 128)
    c_rope, _ = _prep(x, ct, st, api.MODE_BLOCK, interleaved)
    assert np.mean(c_rope != c_pl.cpu().numpy()) > 0.5


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_forward_on_rope_inputs(causal):
    B, N, H, d = 1, 700, 2, 128
    q, k, v = synth.qkv_bf16(B, N, H, d, seed=9, outliers=True)
    c, s, ct, st = _tables(N, d)
    q8, k8, v8, qs, ks, vs = api.fp8_prepare_qkv(to_dev(q), to_dev(k), to_dev(v), api.MODE_BLOCK_HADAMARD, SEED,
                                                 rope=(ct, st, False))
    o, lse = api.attn_fwd_fp8(q8, k8, v8, qs, ks, vs, causal=causal)
    torch.cuda.synchronize()
    rows = np.arange(N, dtype=np.int32)
    qr = oracle.rope(q, c, s).astype(np.float64)
    kr = oracle.rope(k, c, s).astype(np.float64)
    vf = synth.bf16_bits_to_f32(v).astype(np.float64)
    o_ref, lse_ref = oracle.attention(qr, kr, vf, causal=causal, rows=rows)
    err = gpu_rows(o, rows) - o_ref
    rms = float(np.sqrt(np.mean(err ** 2)))
    assert rms <= FP8_RMS, rms
    # against the oracle on the dequantised codes: the kernel's own arithmetic
    o_dq, lse_dq = oracle.attention(dequant(q8, qs), dequant(k8, ks), dequant(v8, vs), causal=causal, rows=rows)
    rms_dq = float(np.sqrt(np.mean((gpu_rows(o, rows) - o_dq) ** 2)))
    lerr = float(np.max(np.abs(lse_rows(lse, rows) - lse_dq)))
    assert rms_dq <= 1e-2 and lerr <= FP8_LSE, (rms_dq, lerr)
    assert api.device_status()[0] == 0
