"""attn_bwd_noalloc: the backward for callers that cannot allocate device
memory (a framework's own memory pool, a fixed memory budget, a layer that
must not own buffers).  It uses the library's built-in scratch buffer instead
of a caller workspace; its results must match attn_bwd's, and both must match
the fp64 oracle within the backward's parity gates.

Each test makes a large call and then a smaller one, so the second call covers
only part of the scratch region the first one wrote: nothing the first call
left there may leak into the second's gradients.  The cases cover both head
dimensions, grouped-query heads and a sliding window.

This file is collected last on purpose (its name), so that a run stopping at
the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from exact_attention_71_gb300 import api, synth
from tests.helpers import to_dev

REL_RMS = 5e-3     # the backward parity gates of the other GPU tests
REL_MAX = 1e-2

# (B, N, H, H_kv, causal, window, seed): a large call, then a smaller one.
CALLS = ((2, 1000, 4, 4, True, 0, 11),
         (1, 300, 4, 2, False, 97, 12))


def _inputs(B, N, H, Hkv, d, seed):
    q = synth.tensor_bf16((B, N, H, d), seed, synth.STREAM_Q)
    k = synth.tensor_bf16((B, N, Hkv, d), seed, synth.STREAM_K)
    v = synth.tensor_bf16((B, N, Hkv, d), seed, synth.STREAM_V)
    do = synth.tensor_bf16((B, N, H, d), seed, 4)
    return q, k, v, do


def _close(got, want, name):
    """Relative RMS and relative largest error of `got` against `want`."""
    got, want = np.asarray(got, dtype=np.float64), np.asarray(want, dtype=np.float64)
    assert np.all(np.isfinite(got)), name
    rel_rms = float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-30))
    rel_max = float(np.max(np.abs(got - want)) / max(np.max(np.abs(want)), 1e-30))
    assert rel_rms <= REL_RMS and rel_max <= REL_MAX, (name, rel_rms, rel_max)


@pytest.mark.gpu
@pytest.mark.parametrize("d", [64, 128])
def test_no_alloc_backward_matches_workspace_entry_and_oracle_large_then_small(d):
    """Two calls in a row on different inputs and sizes, each compared with
    attn_bwd (its own workspace) and with the fp64 oracle."""
    for B, N, H, Hkv, causal, window, seed in CALLS:
        q, k, v, do = _inputs(B, N, H, Hkv, d, seed)
        qd, kd, vd, dod = (to_dev(x) for x in (q, k, v, do))
        o, lse = api.attn_fwd(qd, kd, vd, causal=causal, window=window)
        want = api.attn_bwd(dod, qd, kd, vd, o, lse, causal=causal, window=window)
        got = api.attn_bwd_noalloc(dod, qd, kd, vd, o, lse, causal=causal, window=window)
        torch.cuda.synchronize()
        assert api.device_status()[0] == 0
        ref = oracle.attention_bwd(q, k, v, do, causal=causal, window=window)
        label = f"d={d} B={B} N={N} H={H} H_kv={Hkv} causal={causal} W={window}"
        for g, w, r, name in zip(got, want, ref, ("dq", "dk", "dv")):
            g64 = g.float().cpu().numpy()
            _close(g64, w.float().cpu().numpy(), f"{name} vs attn_bwd, {label}")
            _close(g64, r, f"{name} vs oracle, {label}")


def test_no_alloc_backward_rejects_problems_beyond_its_buffer():
    """No device work is needed to refuse: the size check comes first."""
    L = api.library()
    cap = L.attn_bwd_noalloc_max_scratch()
    assert cap == 256 << 20
    fake = ctypes.c_void_p(1 << 20)
    B, H, N, d = 4, 32, 8192, 128
    assert api.bwd_workspace_bytes(B, H, N, d) > cap
    rc = L.attn_bwd_noalloc(fake, fake, fake, fake, fake, fake, fake, fake, fake, B, H, H, N, d, 0, 0.0, 0, None)
    assert rc == -1
    assert b"scratch" in L.attn_last_error_string()
