"""Pins of the fp64 attention oracle against things other than itself.

Each check is chosen so a plausible slip in the oracle (a dropped scale, a
transposed operand, a wrong mask direction or an off-by-one in the window,
a wrong log base in LSE) fails at least one of them:

* library routine: torch's float64 scaled_dot_product_attention with a
  boolean mask, and torch.logsumexp, on small random inputs;
* closed forms: constant scores (Q = 0) give the mean of the visible V rows
  and LSE = ln(#visible keys);
* one-hot scores select one V row;
* causal row 0 sees only key 0: O_0 = V_0, LSE_0 = scale * q_0 . k_0;
* softmax rows sum to one;
* rotation invariance: (QM)(KM)^T = QK^T for the orthogonal M = D H / sqrt(d)
  (FlashAttention-3 deep-reading report, §2.2, incoherent processing).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_71_gb300 import synth


def _mask(N, causal, window):
    """Visibility via torch's triangular helpers (keys j <= i, j > i - W)."""
    m = torch.ones(N, N, dtype=torch.bool)
    if causal:
        m = torch.tril(m)
    if window > 0:
        m = m & torch.triu(torch.ones(N, N, dtype=torch.bool), diagonal=-(window - 1))
    return m


def _sdpa(q, k, v, causal, window, scale):
    # (B,N,H,d) -> (B,H,N,d)
    qt, kt, vt = (torch.from_numpy(x).permute(0, 2, 1, 3) for x in (q, k, v))
    N = q.shape[1]
    m = _mask(N, causal, window)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=m, scale=scale)
    s = torch.matmul(qt, kt.transpose(-1, -2)) * scale
    s = s.masked_fill(~m, float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    return o.numpy(), lse.numpy()


@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 3), (False, 2), (True, 1)])
@pytest.mark.parametrize("shape", [(1, 7, 1, 4), (2, 16, 3, 8), (1, 13, 2, 5)])
def test_matches_torch_sdpa_float64(shape, causal, window):
    B, N, H, d = shape
    rng = np.random.default_rng(hash((shape, causal, window)) % (2**32))
    q, k, v = (rng.standard_normal(shape) * 1.5 for _ in range(3))
    scale = 0.7 / math.sqrt(d)
    o, lse = oracle.attention(q, k, v, causal=causal, scale=scale, window=window)
    o_ref, lse_ref = _sdpa(q, k, v, causal, window, scale)
    assert np.max(np.abs(o - o_ref)) < 1e-12
    assert np.max(np.abs(lse - lse_ref)) < 1e-12


def test_default_scale_is_inverse_sqrt_d():
    B, N, H, d = 1, 9, 2, 16
    rng = np.random.default_rng(5)
    q, k, v = (rng.standard_normal((B, N, H, d)) for _ in range(3))
    o, lse = oracle.attention(q, k, v)
    o_ref, lse_ref = _sdpa(q, k, v, False, 0, 1.0 / math.sqrt(d))
    assert np.max(np.abs(o - o_ref)) < 1e-12 and np.max(np.abs(lse - lse_ref)) < 1e-12


@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 5)])
def test_constant_scores_give_mean_of_visible_values(causal, window):
    B, N, H, d = 2, 19, 2, 8
    rng = np.random.default_rng(11)
    q = np.zeros((B, N, H, d))
    k = rng.standard_normal((B, N, H, d))
    v = rng.standard_normal((B, N, H, d))
    o, lse = oracle.attention(q, k, v, causal=causal, window=window)
    for i in range(N):
        lo = max(0, i - window + 1) if window > 0 else 0
        hi = i + 1 if causal else N
        want = v[:, lo:hi].mean(axis=1)                      # (B, H, d)
        assert np.max(np.abs(o[:, :, i] - want)) < 1e-13
        assert np.max(np.abs(lse[:, :, i] - math.log(hi - lo))) < 1e-13


def test_one_hot_scores_select_a_value_row():
    N = d = 8
    perm = np.array([3, 0, 7, 1, 6, 2, 5, 4])
    c = 60.0
    k = (c * np.eye(N))[None, :, None, :]
    q = np.eye(d)[perm][None, :, None, :]
    v = np.random.default_rng(3).standard_normal((1, N, 1, d))
    o, lse = oracle.attention(q, k, v, scale=1.0)
    np.testing.assert_allclose(o[0, 0], v[0, perm, 0], atol=1e-20 + 1e-24, rtol=1e-12)
    # LSE = c + log(1 + 7 exp(-c)) ~ c
    assert np.max(np.abs(lse - c)) < 1e-12


def test_causal_row_zero_is_first_value_row():
    q, k, v = synth.qkv_bf16(1, 37, 3, 64, seed=4)
    o, lse = oracle.attention(q, k, v, causal=True)
    qf, kf, vf = (synth.bf16_bits_to_f32(t).astype(np.float64) for t in (q, k, v))
    for h in range(3):
        np.testing.assert_array_equal(o[0, h, 0], vf[0, 0, h])
        dot = float(np.dot(qf[0, 0, h], kf[0, 0, h]))
        assert abs(lse[0, h, 0] - dot / 8.0) < 1e-12


@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 4)])
def test_probability_rows_sum_to_one(causal, window):
    rng = np.random.default_rng(8)
    q, k, v = (rng.standard_normal((1, 24, 2, 16)) * 2 for _ in range(3))
    for i in (0, 1, 7, 23):
        p = oracle.row_probs(q, k, v, 0, 1, i, causal=causal, window=window)
        assert abs(p.sum() - 1.0) < 1e-14
        assert np.all(p >= 0)
        if causal:
            assert np.all(p[i + 1:] == 0)
        if window:
            assert np.all(p[:max(0, i - window + 1)] == 0)


def test_rotation_leaves_attention_unchanged():
    B, N, H, d = 1, 40, 2, 32
    rng = np.random.default_rng(21)
    q, k, v = (rng.standard_normal((B, N, H, d)) for _ in range(3))
    M = oracle.rotation_matrix(d, seed=1234)
    o0, l0 = oracle.attention(q, k, v, causal=True)
    o1, l1 = oracle.attention(q @ M, k @ M, v, causal=True)
    assert np.max(np.abs(o0 - o1)) < 1e-12 and np.max(np.abs(l0 - l1)) < 1e-12


def test_bf16_entry_equals_f64_entry_on_the_same_values():
    q, k, v = synth.qkv_bf16(2, 50, 3, 16, seed=9)
    o_b, l_b = oracle.attention(q, k, v, causal=True, window=7)
    qf, kf, vf = (synth.bf16_bits_to_f32(t).astype(np.float64) for t in (q, k, v))
    o_f, l_f = oracle.attention(qf, kf, vf, causal=True, window=7)
    np.testing.assert_array_equal(o_b, o_f)
    np.testing.assert_array_equal(l_b, l_f)


def test_sampled_rows_equal_full_rows():
    q, k, v = synth.qkv_bf16(1, 300, 2, 32, seed=2)
    rows = synth.sample_rows(300, 40, seed=0)
    o_full, l_full = oracle.attention(q, k, v, causal=True)
    o_s, l_s = oracle.attention(q, k, v, causal=True, rows=rows)
    np.testing.assert_array_equal(o_s, o_full[:, :, rows])
    np.testing.assert_array_equal(l_s, l_full[:, :, rows])


def test_bad_rows_rejected():
    q, k, v = synth.qkv_bf16(1, 10, 1, 8, seed=2)
    with pytest.raises(ValueError):
        oracle.attention(q, k, v, rows=[0, 10])


@pytest.mark.parametrize("Hkv", [1, 2, 3])
def test_grouped_query_heads_equal_repeated_key_value_heads(Hkv):
    """GQA/MQA (deep-reading report §3.4): query head h reads key/value head
    h // group; pinned against the plain multi-head oracle on K and V whose
    heads are repeated group times with numpy."""
    B, N, H, d = 2, 21, 6, 8
    rng = np.random.default_rng(Hkv)
    q = rng.standard_normal((B, N, H, d))
    k = rng.standard_normal((B, N, Hkv, d))
    v = rng.standard_normal((B, N, Hkv, d))
    o, lse = oracle.attention(q, k, v, causal=True, window=5)
    group = H // Hkv
    o_ref, lse_ref = oracle.attention(q, np.repeat(k, group, axis=2), np.repeat(v, group, axis=2),
                                      causal=True, window=5)
    np.testing.assert_array_equal(o, o_ref)
    np.testing.assert_array_equal(lse, lse_ref)


def test_grouped_heads_must_divide():
    q = np.zeros((1, 4, 6, 8)); k = np.zeros((1, 4, 4, 8))
    with pytest.raises(ValueError):
        oracle.attention(q, k, k)
