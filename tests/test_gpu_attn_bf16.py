"""bf16 fused forward vs the fp64 oracle on the same seeded inputs, through
the C ABI (max-abs <= 1e-2, RMS <= 2e-3, LSE <= 1e-3)."""
import functools

import numpy as np
import pytest
import torch

import oracle
from exact_attention_71_gb300 import api, synth
from tests.helpers import assert_bf16_parity, errors, gpu_rows, lse_rows, to_dev

pytestmark = pytest.mark.gpu


def run_case(B, N, H, d, causal=False, window=0, seed=0, rows=None, scale=None):
    q, k, v = synth.qkv_bf16(B, N, H, d, seed=seed)
    o, lse = api.attn_fwd(to_dev(q), to_dev(k), to_dev(v), causal=causal, window=window, scale=scale)
    torch.cuda.synchronize()
    if rows is None:
        rows = np.arange(N, dtype=np.int32)
    o_ref, lse_ref = oracle.attention(q, k, v, causal=causal, window=window, rows=rows, scale=scale)
    e = errors(gpu_rows(o, rows), o_ref, lse_rows(lse, rows), lse_ref)
    rc, site = api.device_status()
    assert rc == 0, f"device status {rc} site {site:#x}"
    return e


def test_config1_small_noncausal():
    """B=1, H=2, N=256, d=64, non-causal, scale 1/sqrt(d), seed 0."""
    e = run_case(1, 256, 2, 64, causal=False)
    assert_bf16_parity(e, "C1")


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_ragged_multi_tile(d, causal):
    e = run_case(1, 1000, 2, d, causal=causal, seed=1)
    assert_bf16_parity(e, f"N=1000 d={d} causal={causal}")


@pytest.mark.parametrize("N", [1, 5, 77, 128, 129, 255, 256, 257, 383])
def test_short_and_boundary_lengths(N):
    for causal in (False, True):
        e = run_case(2, N, 3, 128, causal=causal, seed=N)
        assert_bf16_parity(e, f"N={N} causal={causal}")


@pytest.mark.parametrize("N", [1, 5, 63, 64, 65, 127, 128, 129, 200])
def test_short_and_boundary_lengths_head_dim_256(N):
    """d = 256 runs the one-tile kernel with 64-key tiles and an S pipeline:
    items of a single key tile (the ring then carries a stage with neither K
    nor V), tails shorter than a tile and a pipeline shorter than its depth."""
    for causal in (False, True):
        e = run_case(2, N, 3, 256, causal=causal, seed=N + 1)
        assert_bf16_parity(e, f"d=256 N={N} causal={causal}")


@pytest.mark.parametrize("window", [1, 127, 128, 129, 300, 5000])
def test_sliding_window(window):
    e = run_case(1, 1500, 2, 128, causal=True, window=window, seed=3)
    assert_bf16_parity(e, f"window={window}")


@pytest.mark.parametrize("window", [1, 63, 64, 65, 300])
def test_sliding_window_head_dim_256(window):
    e = run_case(1, 900, 2, 256, causal=True, window=window, seed=6)
    assert_bf16_parity(e, f"d=256 window={window}")


def test_window_without_causal():
    e = run_case(1, 700, 2, 64, causal=False, window=200, seed=4)
    assert_bf16_parity(e, "non-causal window")


def test_explicit_scale():
    e = run_case(1, 300, 2, 128, causal=True, seed=5, scale=0.05)
    assert_bf16_parity(e, "scale=0.05")


def test_config2_full_size_sampled_rows():
    """B=2, H=32, N=4096, d=128, causal (the benchmark workload)."""
    rows = synth.sample_rows(4096, 96, seed=0, must=(4095, 2047, 2048))
    e = run_case(2, 4096, 32, 128, causal=True, rows=rows)
    assert_bf16_parity(e, "C2")


def test_config5_long_window_sampled_rows():
    """B=1, H=8, N=32768, d=128, causal, 4096-token window."""
    rows = synth.sample_rows(32768, 512, seed=5, must=(0, 127, 128, 4095, 4096, 4097, 32767))
    e = run_case(1, 32768, 8, 128, causal=True, window=4096, rows=rows)
    assert_bf16_parity(e, "C5")


def test_empty_problem_is_a_noop():
    x = torch.empty((1, 0, 2, 128), dtype=torch.bfloat16, device="cuda")
    o, lse = api.attn_fwd(x, x, x)
    assert o.numel() == 0 and lse.numel() == 0


def test_outputs_written_exactly_once_and_nothing_outside():
    """NaN-prefilled outputs inside larger guard buffers: every element of O
    and LSE is written, nothing past them is touched."""
    B, N, H, d = 1, 300, 2, 128
    q, k, v = synth.qkv_bf16(B, N, H, d, seed=6)
    guard = 4096
    ob = torch.full((B * N * H * d + guard,), float("nan"), dtype=torch.bfloat16, device="cuda")
    lb = torch.full((B * H * N + guard,), float("nan"), dtype=torch.float32, device="cuda")
    o = ob[: B * N * H * d].view(B, N, H, d)
    lse = lb[: B * H * N].view(B, H, N)
    api.attn_fwd(to_dev(q), to_dev(k), to_dev(v), causal=True, out=o, lse=lse)
    torch.cuda.synchronize()
    assert not torch.isnan(o).any() and not torch.isnan(lse).any()
    assert torch.isnan(ob[B * N * H * d:]).all() and torch.isnan(lb[B * H * N:]).all()


@pytest.mark.parametrize("B,H,N,d", [
    (1, 19, 4096, 64),     # 304 causal items: two whole rounds of 152 CTAs
    (1, 10, 4096, 128),    # 160: one round and a partial one
    (2, 100, 256, 64),     # one query block per head
    (1, 7, 4000, 128),     # fewer items than CTAs, ragged last tile
    (3, 37, 1792, 128),    # 777: five rounds and 17 items
    (1, 12, 2048, 256),    # head dim 256 (one 128-row tile per item)
])
def test_causal_item_order_covers_every_row(B, H, N, d):
    """The causal work order (rounds cut out of a head-major sequence, the
    lightest items last) must hand every (query block, head) to exactly one
    CTA: NaN-prefilled outputs are all written, and sampled rows of every head
    match the oracle."""
    q, k, v = synth.qkv_bf16(B, N, H, d, seed=12)
    o = torch.full((B, N, H, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
    api.attn_fwd(to_dev(q), to_dev(k), to_dev(v), causal=True, out=o, lse=lse)
    torch.cuda.synchronize()
    assert not torch.isnan(o).any() and not torch.isnan(lse).any()
    rows = np.array(sorted({0, 127, 128, 255, N // 2, N - 1} & set(range(N))))
    o_ref, lse_ref = oracle.attention(q, k, v, causal=True, rows=rows)
    assert_bf16_parity(errors(gpu_rows(o, rows), o_ref, lse_rows(lse, rows), lse_ref), f"order B{B} H{H} N{N} d{d}")


def test_repeat_is_bitwise_deterministic():
    q, k, v = (to_dev(t) for t in synth.qkv_bf16(1, 900, 4, 128, seed=7))
    o1, l1 = api.attn_fwd(q, k, v, causal=True)
    o2, l2 = api.attn_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@functools.lru_cache(maxsize=1)
def _sweep_inputs(N, d):
    """The sweep point's Q, K, V (the causal and non-causal cases share them)."""
    return synth.qkv_bf16(16384 // N, N, 2048 // d, d, seed=11)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("N", [512, 1024, 2048, 4096, 8192, 16384])
def test_config3_sweep_sampled_rows(N, d, causal):
    """16384 tokens, hidden 2048: B = 16384 / N, H = 2048 / d; every point of
    the sweep, 256 sampled query rows of every head (first and last rows,
    tile-boundary rows, the rows around each 1024-row boundary and seeded
    picks)."""
    B, H = 16384 // N, 2048 // d
    q, k, v = _sweep_inputs(N, d)
    must = [r for x in range(1024, N, 1024) for r in (x - 1, x)]
    rows = synth.sample_rows(N, 256, seed=N + d, must=must)
    o, lse = api.attn_fwd(to_dev(q), to_dev(k), to_dev(v), causal=causal)
    torch.cuda.synchronize()
    assert api.device_status()[0] == 0
    o_ref, lse_ref = oracle.attention(q, k, v, causal=causal, rows=rows)
    e = errors(gpu_rows(o, rows), o_ref, lse_rows(lse, rows), lse_ref)
    assert_bf16_parity(e, f"C3 N={N} d={d} causal={causal}")


def _growing_scores(N, H, d, seed):
    """Scores that grow by ~16 log2-units per 128-key tile for most rows (the
    running maximum jumps every tile, so the accumulator is rescaled), plus
    rows whose scores shrink (never rescaled)."""
    rng = np.random.default_rng(seed)
    u = np.sign(rng.standard_normal(d))
    a = rng.uniform(0.25, 1.5, size=(N, H)) * np.where(rng.random((N, H)) < 0.8, 1.0, -1.0)
    b = np.arange(N)[:, None] / 128.0 + 0.5 * rng.standard_normal((N, H))
    q = a[None, :, :, None] * u
    k = b[None, :, :, None] * u + 0.3 * rng.standard_normal((1, N, H, d))
    v = rng.standard_normal((1, N, H, d))
    return tuple(synth.to_bf16_bits(x) for x in (q, k, v))


@pytest.mark.parametrize("d", [128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_growing_scores_exercise_rescaling(causal, d):
    """Scores that grow along the keys move the reference maximum often: the
    O rescale (at d = 256 after waiting for the previous P V) is exercised."""
    N, H = 1100, 2
    q, k, v = _growing_scores(N, H, d, seed=3)
    o, lse = api.attn_fwd(to_dev(q), to_dev(k), to_dev(v), causal=causal)
    torch.cuda.synchronize()
    rows = np.arange(N, dtype=np.int32)
    o_ref, lse_ref = oracle.attention(q, k, v, causal=causal, rows=rows)
    e = errors(gpu_rows(o, rows), o_ref, lse_rows(lse, rows), lse_ref)
    # LSE here reaches ~100: the tolerance is relative to its magnitude
    assert e["rms"] <= 2e-3 and e["max_excess"] <= 1e-2, e
    assert np.max(np.abs(lse_rows(lse, rows) - lse_ref) / np.maximum(1.0, np.abs(lse_ref))) <= 1e-5, e


@pytest.mark.parametrize("d", [64, 128, 256])
def test_window_rows_whose_first_key_tile_is_masked_with_very_negative_scores(d):
    """Causal, W = 200, N = 640: rows 583..639 see none of the keys of their
    query tile's first key tile.  Every score is -16 sqrt(d) (q = 4, k = -4),
    far below 0, so the row's first visible scores must set its running
    maximum (a maximum left at 0 would underflow every P).  Constant scores:
    O_i is the mean of the visible V rows (and the oracle agrees)."""
    B, N, H, W = 1, 640, 1, 200
    q = np.full((B, N, H, d), synth.to_bf16_bits(np.array([4.0]))[0], dtype=np.uint16)
    k = np.full((B, N, H, d), synth.to_bf16_bits(np.array([-4.0]))[0], dtype=np.uint16)
    v = synth.tensor_bf16((B, N, H, d), seed=3, stream=3)
    o, lse = api.attn_fwd(to_dev(q), to_dev(k), to_dev(v), causal=True, window=W)
    torch.cuda.synchronize()
    rows = np.arange(N, dtype=np.int32)
    o_ref, lse_ref = oracle.attention(q, k, v, causal=True, window=W, rows=rows)
    vf = synth.bf16_bits_to_f32(v).astype(np.float64)
    for i in (0, 582, 583, 600, 639):
        np.testing.assert_allclose(o_ref[0, 0, i], vf[0, max(0, i - W + 1):i + 1, 0].mean(axis=0), atol=1e-12)
    e = errors(gpu_rows(o, rows), o_ref, lse_rows(lse, rows), lse_ref)
    assert_bf16_parity(e, f"masked first tile d={d}")
    assert api.device_status()[0] == 0
