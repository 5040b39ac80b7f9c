"""Block-sparse forward (attn_fwd_sparse) against the fp64 oracle with the
same block mask (bf16 parity bar: max-abs <= 1e-2, RMS <= 2e-3, LSE <= 1e-3
on rows that see a key; rows that see none: O = 0, LSE = -inf exactly)."""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_71_gb300 import api, synth
from tests.helpers import assert_bf16_parity, errors, gpu_rows, lse_rows, to_dev

pytestmark = pytest.mark.gpu


def _mask(B, H, N, density, seed):
    T = (N + 127) // 128
    rng = np.random.default_rng(seed)
    return (rng.random((B, H, T, T)) < density).astype(np.uint8)


def _run(B, N, H, d, block, causal=False, window=0, Hkv=None, seed=0, rows=None):
    Hkv = Hkv or H
    q = synth.tensor_bf16((B, N, H, d), seed, synth.STREAM_Q)
    k = synth.tensor_bf16((B, N, Hkv, d), seed, synth.STREAM_K)
    v = synth.tensor_bf16((B, N, Hkv, d), seed, synth.STREAM_V)
    o, lse = api.attn_fwd_sparse(to_dev(q), to_dev(k), to_dev(v), torch.from_numpy(block).cuda(), causal=causal,
                                 window=window)
    torch.cuda.synchronize()
    assert api.device_status()[0] == 0
    if rows is None:
        rows = np.arange(N, dtype=np.int32)
    o_ref, lse_ref = oracle.attention(q, k, v, causal=causal, window=window, rows=rows, block_mask=block)
    og, lg = gpu_rows(o, rows), lse_rows(lse, rows)
    empty = np.isneginf(lse_ref)
    assert np.all(og[empty] == 0.0) and np.all(np.isneginf(lg[empty])), "rows without keys"
    seen = ~empty
    if seen.any():
        e = errors(og[seen], o_ref[seen], lg[seen], lse_ref[seen])
        assert_bf16_parity(e, f"sparse N={N} d={d} causal={causal} W={window}")
    return empty.mean()


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("density", [0.5, 0.2])
@pytest.mark.parametrize("causal", [False, True])
def test_random_block_masks(d, density, causal):
    B, N, H = 1, 1000, 2
    _run(B, N, H, d, _mask(B, H, N, density, seed=int(density * 100) + d), causal=causal, seed=1)


def test_sparse_with_window_and_grouped_heads():
    B, N, H, Hkv, d = 2, 777, 4, 2, 128
    _run(B, N, H, d, _mask(B, H, N, 0.6, seed=9), causal=True, window=300, Hkv=Hkv, seed=2)


def test_rows_that_see_no_key():
    B, N, H, d = 1, 640, 2, 128
    block = _mask(B, H, N, 0.5, seed=3)
    block[:, :, 2, :] = 0            # query block 2 sees nothing
    block[:, 1, :, :] = 0            # head 1 sees nothing at all
    frac = _run(B, N, H, d, block, causal=False, seed=3)
    assert frac >= 0.5


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_many_items_per_cta_with_inactive_tiles(d, causal):
    """640 work items (about four per CTA on a 152-SM part): a CTA's key walk
    runs on from one item into the next, carrying the last P V of each tile.
    Random masks, query tiles that see no key block (inactive tiles), and
    heads that see nothing at all (items with no key step) between active
    items."""
    B, N, H = 2, 2048, 40
    block = _mask(B, H, N, 0.35, seed=40 + d)
    T = block.shape[2]
    block[:, :, ::5, :] = 0              # every fifth query tile sees no key
    block[:, 3::7, :, :] = 0             # every seventh head sees nothing
    rows = synth.sample_rows(N, 48, seed=8, must=(0, 127, 128, 255, 256, 640, 767, N - 1))
    frac = _run(B, N, H, d, block, causal=causal, seed=4, rows=rows)
    assert 0.1 < frac < 0.9


def test_all_ones_mask_equals_dense_forward():
    B, N, H, d = 1, 1000, 2, 128
    q, k, v = synth.qkv_bf16(B, N, H, d, seed=6)
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    ones = torch.ones((B, H, 8, 8), dtype=torch.uint8, device="cuda")
    for causal, window in ((False, 0), (True, 0), (True, 300)):
        o1, l1 = api.attn_fwd_sparse(qd, kd, vd, ones, causal=causal, window=window)
        o2, l2 = api.attn_fwd(qd, kd, vd, causal=causal, window=window)
        torch.cuda.synchronize()
        # Same arithmetic in the same order (one issuer instead of two changes no value).
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_full_size_band_plus_strided_pattern_sampled_rows():
    """B=1, H=16, N=16384, d=128, non-causal: a band of +-8 key blocks around
    the diagonal plus every 8th key block (about 24 % of the blocks)."""
    B, N, H, d = 1, 16384, 16, 128
    T = N // 128
    i = np.arange(T)[:, None]
    j = np.arange(T)[None, :]
    block = ((np.abs(i - j) <= 8) | (j % 8 == 0)).astype(np.uint8)
    block = np.broadcast_to(block, (B, H, T, T)).copy()
    rows = synth.sample_rows(N, 64, seed=5, must=(0, 127, 128, 8191, 16383))
    _run(B, N, H, d, block, rows=rows, seed=0)
