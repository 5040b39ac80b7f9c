"""Failure detection on the GPU without a GPU fault.

Every barrier wait inside the forward kernel is bounded.  The test makes
the waits run out by setting a one-cycle wait limit: the kernel must give
up, record the site in the library's status word and return (no hang), the
host must see ATTN_ERR_DEVICE_TIMEOUT, and the CUDA context must stay usable
so that the next call, with the default limit, is correct.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_71_gb300 import api, synth
from tests.helpers import assert_bf16_parity, errors, gpu_rows, lse_rows, to_dev

pytestmark = pytest.mark.gpu

ATTN_ERR_DEVICE_TIMEOUT = -4
KNOWN_SITES = {0x11, 0x12, 0x21, 0x22, 0x23, 0x24, 0x31, 0x32, 0x41}


def test_wait_timeout_is_reported_and_the_context_survives():
    B, N, H, d = 1, 1024, 2, 128
    q, k, v = synth.qkv_bf16(B, N, H, d, seed=8)
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    lib = api.library()
    assert api.device_status()[0] == 0
    assert lib.attn_set_wait_limit(1) == 0
    try:
        api.attn_fwd(qd, kd, vd, causal=True)
        rc, site = api.device_status()
        msg = lib.attn_last_error_string()
    finally:
        lib.attn_set_wait_limit(0)
    assert rc == ATTN_ERR_DEVICE_TIMEOUT, (rc, site)
    assert site in KNOWN_SITES, hex(site)
    assert b"gave up" in msg
    # status word cleared, context usable, results correct again
    assert api.device_status()[0] == 0
    o, lse = api.attn_fwd(qd, kd, vd, causal=True)
    torch.cuda.synchronize()
    rows = np.arange(N, dtype=np.int32)
    o_ref, lse_ref = oracle.attention(q, k, v, causal=True)
    assert_bf16_parity(errors(gpu_rows(o, rows), o_ref, lse_rows(lse, rows), lse_ref), "after timeout")
    assert api.device_status()[0] == 0
