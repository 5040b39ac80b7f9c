"""Attention backward (attn_bwd) on the GPU against the fp64 oracle.

The forward's O and LSE come from attn_fwd; the oracle computes dQ, dK, dV
from Q, K, V and dO alone (its own fp64 softmax), so the comparison covers
the whole chain.  Error measure (the pages state none for the backward):
relative RMS, ||g - g_ref||_2 / ||g_ref||_2, and the largest element error
relative to max |g_ref|, per gradient.  P and dS enter the tensor-core
products as bf16 (unit roundoff u = 2^-8) and the gradients are stored as
bf16.  The bf16 rounding of the stored gradients alone gives a relative RMS
of about u / sqrt(12) ~ 1.1e-3 per element for uniform rounding errors;
measured on GB300 the total is 2.2-2.7e-3 (relative max 2-4.4e-3) on every
case below.  The gates are 5e-3 relative RMS (1.3 u) and 1e-2 of the
largest magnitude.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_71_gb300 import api, synth
from tests.helpers import to_dev

pytestmark = pytest.mark.gpu

REL_RMS = 5e-3
REL_MAX = 1e-2


def _inputs(B, N, H, d, Hkv=None, seed=0):
    Hkv = Hkv or H
    q = synth.tensor_bf16((B, N, H, d), seed=seed, stream=synth.STREAM_Q)
    k = synth.tensor_bf16((B, N, Hkv, d), seed=seed, stream=synth.STREAM_K)
    v = synth.tensor_bf16((B, N, Hkv, d), seed=seed, stream=synth.STREAM_V)
    do = synth.tensor_bf16((B, N, H, d), seed=seed, stream=4)
    return q, k, v, do


def _gpu_grads(q, k, v, do, causal, window):
    qd, kd, vd, dod = (to_dev(x) for x in (q, k, v, do))
    o, lse = api.attn_fwd(qd, kd, vd, causal=causal, window=window)
    dq, dk, dv = api.attn_bwd(dod, qd, kd, vd, o, lse, causal=causal, window=window)
    torch.cuda.synchronize()
    assert api.device_status()[0] == 0
    return [t.float().cpu().numpy().astype(np.float64) for t in (dq, dk, dv)]


def _check(got, ref, label):
    out = {}
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        assert np.all(np.isfinite(g)), (label, name)
        rel_rms = float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30))
        rel_max = float(np.max(np.abs(g - r)) / max(np.max(np.abs(r)), 1e-30))
        out[name] = (rel_rms, rel_max)
    print(label, {k: f"{a:.2e}/{b:.2e}" for k, (a, b) in out.items()})
    for name, (a, b) in out.items():
        assert a <= REL_RMS and b <= REL_MAX, (label, name, a, b)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [64, 129, 300, 1000])
@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 97), (False, 200)])
def test_backward_matches_oracle(N, causal, window, d):
    B, H = 1, 2
    q, k, v, do = _inputs(B, N, H, d, seed=N)
    got = _gpu_grads(q, k, v, do, causal, window)
    ref = oracle.attention_bwd(q, k, v, do, causal=causal, window=window)
    _check(got, ref, f"d={d} N={N} causal={causal} W={window}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Hkv", [1, 2])
def test_backward_grouped_query(Hkv, d):
    B, N, H = 2, 257, 4
    q, k, v, do = _inputs(B, N, H, d, Hkv=Hkv, seed=7)
    got = _gpu_grads(q, k, v, do, True, 0)
    ref = oracle.attention_bwd(q, k, v, do, causal=True)
    _check(got, ref, f"GQA d={d} H={H} Hkv={Hkv}")


def test_backward_head_dim_64_full_size_heads():
    """B=1, H=32, N=8192, d=64, causal: two heads against the oracle."""
    B, N, H, d = 1, 8192, 32, 64
    q, k, v, do = _inputs(B, N, H, d, seed=5)
    dq, dk, dv = _gpu_grads(q, k, v, do, True, 0)
    for h in (0, 17):
        sl = slice(h, h + 1)
        ref = oracle.attention_bwd(q[:, :, sl], k[:, :, sl], v[:, :, sl], do[:, :, sl], causal=True)
        _check([dq[:, :, sl], dk[:, :, sl], dv[:, :, sl]], ref, f"d=64 N=8192 head {h}")


def test_backward_full_size_heads_and_invariants():
    """B=2, H=32, N=4096, causal (the forward's headline shape): two heads
    against the oracle, and for every head the sums that hold exactly in
    exact arithmetic: sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i."""
    B, N, H, d = 2, 4096, 32, 128
    q, k, v, do = _inputs(B, N, H, d, seed=0)
    dq, dk, dv = _gpu_grads(q, k, v, do, True, 0)
    for h in (0, 31):
        sl = slice(h, h + 1)
        ref = oracle.attention_bwd(q[:, :, sl], k[:, :, sl], v[:, :, sl], do[:, :, sl], causal=True)
        _check([dq[:, :, sl], dk[:, :, sl], dv[:, :, sl]], ref, f"C2 head {h}")
    dof = synth.bf16_bits_to_f32(do).astype(np.float64)
    sum_dv, want = dv.sum(axis=1), dof.sum(axis=1)
    assert np.max(np.abs(sum_dv - want)) <= 2e-2 * np.max(np.abs(want))
    # dK rows are O(|q| |dS|); their sum over 4096 keys cancels to rounding level.
    assert np.max(np.abs(dk.sum(axis=1))) <= 2e-2 * np.max(np.abs(dk)) * np.sqrt(N)


def test_backward_key_value_gradients_are_deterministic():
    B, N, H, d = 1, 700, 2, 128
    q, k, v, do = _inputs(B, N, H, d, seed=3)
    a = _gpu_grads(q, k, v, do, True, 0)
    b = _gpu_grads(q, k, v, do, True, 0)
    np.testing.assert_array_equal(a[1], b[1])
    np.testing.assert_array_equal(a[2], b[2])
    # dQ is a float32 sum over key tiles in arrival order: equal up to rounding.
    assert np.max(np.abs(a[0] - b[0])) <= 1e-2 * np.max(np.abs(a[0]))
