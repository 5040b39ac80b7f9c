"""Pins of the oracle's block-sparse key mask (the practitioner's FA3 post,
§3.3: the caller decides per query block and key block, 128 x 128 here,
whether the pair takes part; ANDed with the causal and window masks).

* an all-ones mask is no mask (bit for bit);
* torch float64 scaled_dot_product_attention with the element mask the
  block mask expands to, on ragged lengths and every mask kind;
* a block-diagonal mask is attention inside each 128-token chunk alone;
* a row that sees no key gets O = 0 and LSE = -inf.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_71_gb300 import synth


def _element_mask(block, N, causal, window):
    T = block.shape[-1]
    m = np.kron(block.astype(bool), np.ones((128, 128), dtype=bool))[..., :N, :N]
    i = np.arange(N)[:, None]
    j = np.arange(N)[None, :]
    vis = np.ones((N, N), dtype=bool)
    if causal:
        vis &= j <= i
    if window > 0:
        vis &= j > i - window
    return m & vis


def test_all_ones_mask_is_no_mask():
    q, k, v = synth.qkv_bf16(2, 300, 3, 16, seed=1)
    ones = np.ones((2, 3, 3, 3), dtype=np.uint8)
    a = oracle.attention(q, k, v, causal=True, window=150)
    b = oracle.attention(q, k, v, causal=True, window=150, block_mask=ones)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 170), (False, 90)])
@pytest.mark.parametrize("N", [130, 300])
def test_matches_torch_sdpa_with_expanded_mask(N, causal, window):
    B, H, d = 1, 2, 8
    rng = np.random.default_rng(N + window)
    q, k, v = (rng.standard_normal((B, N, H, d)) for _ in range(3))
    T = (N + 127) // 128
    block = (rng.random((B, H, T, T)) < 0.6).astype(np.uint8)
    o, lse = oracle.attention(q, k, v, causal=causal, window=window, block_mask=block)
    m = torch.from_numpy(_element_mask(block, N, causal, window))            # (B, H, N, N)
    qt, kt, vt = (torch.from_numpy(x).permute(0, 2, 1, 3) for x in (q, k, v))
    scale = 1.0 / np.sqrt(d)
    s = (qt @ kt.transpose(-1, -2) * scale).masked_fill(~m, float("-inf"))
    seen = m.any(dim=-1).numpy()                                              # (B, H, N)
    ref_o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=m, scale=scale).numpy()
    ref_l = torch.logsumexp(s, dim=-1).numpy()
    np.testing.assert_allclose(o[seen], ref_o[seen], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[seen], ref_l[seen], rtol=0, atol=1e-12)
    assert np.all(o[~seen] == 0.0) and np.all(np.isneginf(lse[~seen]))


def test_block_diagonal_mask_is_chunked_attention():
    B, N, H, d = 1, 384, 2, 16
    q, k, v = synth.qkv_bf16(B, N, H, d, seed=4)
    diag = np.zeros((B, H, 3, 3), dtype=np.uint8)
    for t in range(3):
        diag[:, :, t, t] = 1
    o, lse = oracle.attention(q, k, v, block_mask=diag)
    for t in range(3):
        sl = slice(128 * t, 128 * t + 128)
        oc, lc = oracle.attention(q[:, sl], k[:, sl], v[:, sl])
        np.testing.assert_array_equal(o[:, :, sl], oc)
        np.testing.assert_array_equal(lse[:, :, sl], lc)


def test_empty_mask_rows():
    q, k, v = synth.qkv_bf16(1, 200, 1, 8, seed=5)
    block = np.array([[[[1, 0], [0, 0]]]], dtype=np.uint8)
    o, lse = oracle.attention(q, k, v, block_mask=block)
    assert np.all(o[:, :, 128:] == 0) and np.all(np.isneginf(lse[:, :, 128:]))
    assert np.all(np.isfinite(lse[:, :, :128]))


def test_bad_mask_shape_rejected():
    q, k, v = synth.qkv_bf16(1, 200, 1, 8, seed=5)
    with pytest.raises(ValueError):
        oracle.attention(q, k, v, block_mask=np.ones((1, 1, 3, 3), dtype=np.uint8))
