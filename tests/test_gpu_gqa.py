"""Grouped-query and multi-query attention (deep-reading report §3.4) on the
GPU against the fp64 oracle: query head h reads key/value head
h // (H // H_kv); K and V are stored once per key/value head."""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_71_gb300 import api, synth
from tests.helpers import FP8_LSE, assert_bf16_parity, errors, gpu_rows, lse_rows, to_dev

pytestmark = pytest.mark.gpu


def _qkv(B, N, H, Hkv, d, seed):
    q = synth.tensor_bf16((B, N, H, d), seed, synth.STREAM_Q)
    k = synth.tensor_bf16((B, N, Hkv, d), seed, synth.STREAM_K)
    v = synth.tensor_bf16((B, N, Hkv, d), seed, synth.STREAM_V)
    return q, k, v


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("H,Hkv,causal", [(8, 2, True), (8, 1, False), (6, 3, True)])
def test_gqa_parity(d, H, Hkv, causal):
    B, N = 2, 700
    q, k, v = _qkv(B, N, H, Hkv, d, seed=H * 10 + Hkv)
    o, lse = api.attn_fwd(to_dev(q), to_dev(k), to_dev(v), causal=causal)
    torch.cuda.synchronize()
    rows = np.arange(N, dtype=np.int32)
    o_ref, lse_ref = oracle.attention(q, k, v, causal=causal, rows=rows)
    assert_bf16_parity(errors(gpu_rows(o, rows), o_ref, lse_rows(lse, rows), lse_ref), f"GQA H={H} Hkv={Hkv} d={d}")
    assert api.device_status()[0] == 0


def test_gqa_window_full_size_sampled():
    """B=1, H=32, H_kv=8, N=16384, d=128, causal, 4096-token window."""
    B, N, H, Hkv, d = 1, 16384, 32, 8, 128
    q, k, v = _qkv(B, N, H, Hkv, d, seed=1)
    o, lse = api.attn_fwd(to_dev(q), to_dev(k), to_dev(v), causal=True, window=4096)
    torch.cuda.synchronize()
    rows = synth.sample_rows(N, 64, seed=2, must=(4095, 4096, 16383))
    o_ref, lse_ref = oracle.attention(q, k, v, causal=True, window=4096, rows=rows)
    assert_bf16_parity(errors(gpu_rows(o, rows), o_ref, lse_rows(lse, rows), lse_ref), "GQA window")


def test_gqa_fp8_matches_oracle_on_dequantised_codes():
    B, N, H, Hkv, d = 1, 600, 8, 2, 128
    q, k, v = _qkv(B, N, H, Hkv, d, seed=3)
    q8, qs = api.attn_fp8_prep(to_dev(q), api.MODE_BLOCK_HADAMARD, 99)
    k8, ks = api.attn_fp8_prep(to_dev(k), api.MODE_BLOCK_HADAMARD, 99)
    v8, vs = api.attn_fp8_prep(to_dev(v), api.MODE_BLOCK_HADAMARD, 99, is_v=True)
    o, lse = api.attn_fwd_fp8(q8, k8, v8, qs, ks, vs, causal=True)
    torch.cuda.synchronize()

    def deq(codes, scales):
        c = codes.cpu().numpy()
        sc = np.repeat(scales.cpu().numpy().astype(np.float64).transpose(0, 2, 1), 128, axis=1)[:, :c.shape[1]]
        return oracle.e4m3_decode(c.ravel()).reshape(c.shape) * sc[..., None]

    rows = np.arange(N, dtype=np.int32)
    o_ref, lse_ref = oracle.attention(deq(q8, qs), deq(k8, ks), deq(v8, vs), causal=True, rows=rows)
    err = np.abs(gpu_rows(o, rows) - o_ref)
    assert float(np.sqrt(np.mean(err ** 2))) <= 1e-2
    assert float(np.max(np.abs(lse_rows(lse, rows) - lse_ref))) <= FP8_LSE
    assert api.device_status()[0] == 0


def test_gqa_heads_must_divide():
    x = torch.zeros((1, 16, 6, 128), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((1, 16, 4, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        api.attn_fwd(x, y, y)
