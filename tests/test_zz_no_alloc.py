"""attn_bwd_noalloc: the backward for callers that cannot allocate device
memory (a framework's own memory pool, a fixed memory budget, a layer that
must not own buffers).  It uses the library's built-in scratch buffer instead
of a caller workspace; its results must match attn_bwd's.

This file is collected last on purpose (its name), so that a run stopping at
the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from exact_attention_71_gb300 import api, synth
from tests.helpers import to_dev

REL_RMS = 5e-3     # the backward parity gates of the other GPU tests
REL_MAX = 1e-2


def _inputs(B, N, H, d, seed):
    q = synth.tensor_bf16((B, N, H, d), seed, synth.STREAM_Q)
    k = synth.tensor_bf16((B, N, H, d), seed, synth.STREAM_K)
    v = synth.tensor_bf16((B, N, H, d), seed, synth.STREAM_V)
    do = synth.tensor_bf16((B, N, H, d), seed, 4)
    return [to_dev(x) for x in (q, k, v, do)]


def _close(a, b, name):
    a, b = a.float(), b.float()
    rel_rms = float(torch.linalg.norm(a - b) / torch.linalg.norm(b))
    rel_max = float((a - b).abs().max() / b.abs().max())
    assert rel_rms <= REL_RMS and rel_max <= REL_MAX, (name, rel_rms, rel_max)


@pytest.mark.gpu
def test_no_alloc_backward_matches_the_workspace_entry_point_twice_in_a_row():
    """Two calls in a row on different inputs (the second must not see the
    first's scratch contents), each against attn_bwd with its own workspace."""
    B, N, H, d = 2, 1000, 4, 128
    for seed, causal in ((11, True), (12, False)):
        q, k, v, do = _inputs(B, N, H, d, seed)
        o, lse = api.attn_fwd(q, k, v, causal=causal)
        want = api.attn_bwd(do, q, k, v, o, lse, causal=causal)
        got = api.attn_bwd_noalloc(do, q, k, v, o, lse, causal=causal)
        torch.cuda.synchronize()
        assert api.device_status()[0] == 0
        for g, w, name in zip(got, want, ("dq", "dk", "dv")):
            _close(g, w, f"{name} seed={seed}")


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
