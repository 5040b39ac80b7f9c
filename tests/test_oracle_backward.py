"""Pins of the fp64 backward oracle against things other than itself
(FlashAttention-3 deep-reading report §3.4: the backward recomputes the
softmax from the forward's statistics, FA2 style).

* library routine: torch float64 autograd through an explicitly masked
  softmax attention, on small random inputs, every mask kind;
* finite differences of the (separately pinned) forward oracle: the
  derivative of L = sum(dO * O) along random directions in q, k and v;
* grouped-query heads: dK, dV of a key/value head are the sums over its
  group of the multi-head gradients with repeated K, V heads;
* invariants at any size: sum_j dK_j = 0 (each softmax row's dS sums to
  zero) and sum_j dV_j = sum_i dO_i (each P row sums to one);
* closed form: with Q = 0 every visible key gets equal weight, so
  dV_j = sum over the rows i that see j of dO_i / (number of keys row i sees).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_71_gb300 import synth


def _torch_grads(q, k, v, dout, causal, window, scale):
    N = q.shape[1]
    group = q.shape[2] // k.shape[2]
    qt, kt, vt = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    kk = kt.repeat_interleave(group, dim=2)
    vv = vt.repeat_interleave(group, dim=2)
    s = torch.einsum("bihc,bjhc->bhij", qt, kk) * scale
    m = torch.ones(N, N, dtype=torch.bool)
    if causal:
        m = torch.tril(m)
    if window > 0:
        m = m & torch.triu(torch.ones(N, N, dtype=torch.bool), diagonal=-(window - 1))
    s = s.masked_fill(~m, float("-inf"))
    p = torch.softmax(s, dim=-1)
    o = torch.einsum("bhij,bjhc->bihc", p, vv)
    o.backward(torch.tensor(dout))
    return qt.grad.numpy(), kt.grad.numpy(), vt.grad.numpy()


@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 3), (False, 4)])
@pytest.mark.parametrize("shape", [(1, 7, 2, 4, 2), (2, 12, 4, 8, 1), (1, 9, 3, 5, 3)])
def test_matches_torch_autograd_float64(shape, causal, window):
    B, N, H, d, Hkv = shape
    rng = np.random.default_rng(hash((shape, causal, window)) % (2 ** 32))
    q = rng.standard_normal((B, N, H, d)) * 1.3
    k = rng.standard_normal((B, N, Hkv, d)) * 1.3
    v = rng.standard_normal((B, N, Hkv, d))
    dout = rng.standard_normal((B, N, H, d))
    scale = 0.8 / math.sqrt(d)
    dq, dk, dv = oracle.attention_bwd(q, k, v, dout, causal=causal, scale=scale, window=window)
    rq, rk, rv = _torch_grads(q, k, v, dout, causal, window, scale)
    for a, b in ((dq, rq), (dk, rk), (dv, rv)):
        assert np.max(np.abs(a - b)) < 1e-12


@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 4)])
def test_directional_derivatives_match_finite_differences(causal, window):
    B, N, H, d = 1, 10, 2, 6
    rng = np.random.default_rng(17)
    q, k, v, dout = (rng.standard_normal((B, N, H, d)) for _ in range(4))

    def loss(q_, k_, v_):
        o, _ = oracle.attention(q_, k_, v_, causal=causal, window=window)     # (B, H, N, d)
        return float(np.sum(o.transpose(0, 2, 1, 3) * dout))

    dq, dk, dv = oracle.attention_bwd(q, k, v, dout, causal=causal, window=window)
    h = 1e-5
    for which, grad in ((0, dq), (1, dk), (2, dv)):
        for trial in range(3):
            u = rng.standard_normal((B, N, H, d))
            args_p = [q, k, v]
            args_m = [q, k, v]
            args_p[which] = args_p[which] + h * u
            args_m[which] = args_m[which] - h * u
            fd = (loss(*args_p) - loss(*args_m)) / (2 * h)
            an = float(np.sum(grad * u))
            assert abs(fd - an) <= 1e-7 * max(1.0, abs(an)), (which, fd, an)


def test_grouped_query_gradients_are_group_sums():
    B, N, H, d, Hkv = 1, 11, 6, 8, 2
    rng = np.random.default_rng(5)
    q = rng.standard_normal((B, N, H, d))
    k = rng.standard_normal((B, N, Hkv, d))
    v = rng.standard_normal((B, N, Hkv, d))
    dout = rng.standard_normal((B, N, H, d))
    dq, dk, dv = oracle.attention_bwd(q, k, v, dout, causal=True)
    g = H // Hkv
    rq, rk, rv = oracle.attention_bwd(q, np.repeat(k, g, axis=2), np.repeat(v, g, axis=2), dout, causal=True)
    np.testing.assert_allclose(dq, rq, rtol=0, atol=1e-13)
    np.testing.assert_allclose(dk, rk.reshape(B, N, Hkv, g, d).sum(axis=3), rtol=0, atol=1e-13)
    np.testing.assert_allclose(dv, rv.reshape(B, N, Hkv, g, d).sum(axis=3), rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 9)])
def test_key_gradients_sum_to_zero_and_value_gradients_to_dout(causal, window):
    q, k, v = synth.qkv_bf16(2, 70, 3, 16, seed=3)
    dout = synth.tensor_bf16((2, 70, 3, 16), seed=3, stream=4)
    dq, dk, dv = oracle.attention_bwd(q, k, v, dout, causal=causal, window=window)
    assert np.max(np.abs(dk.sum(axis=1))) < 1e-11
    dof = synth.bf16_bits_to_f32(dout).astype(np.float64)
    np.testing.assert_allclose(dv.sum(axis=1), dof.sum(axis=1), rtol=0, atol=1e-11)


@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 5)])
def test_constant_scores_value_gradient_closed_form(causal, window):
    B, N, H, d = 1, 15, 2, 4
    rng = np.random.default_rng(2)
    q = np.zeros((B, N, H, d))
    k, v, dout = (rng.standard_normal((B, N, H, d)) for _ in range(3))
    _, _, dv = oracle.attention_bwd(q, k, v, dout, causal=causal, window=window)
    want = np.zeros_like(dv)
    for i in range(N):
        lo = max(0, i - window + 1) if window > 0 else 0
        hi = i + 1 if causal else N
        want[:, lo:hi] += dout[:, i:i + 1] / (hi - lo)
    np.testing.assert_allclose(dv, want, rtol=0, atol=1e-13)


def test_bf16_entry_equals_f64_entry():
    q, k, v = synth.qkv_bf16(1, 40, 2, 8, seed=8)
    dout = synth.tensor_bf16((1, 40, 2, 8), seed=8, stream=4)
    a = oracle.attention_bwd(q, k, v, dout, causal=True, window=6)
    f = [synth.bf16_bits_to_f32(t).astype(np.float64) for t in (q, k, v, dout)]
    b = oracle.attention_bwd(*f, causal=True, window=6)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
