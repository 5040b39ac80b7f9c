"""Failure detection on the GPU without a GPU fault.

Every barrier wait inside the kernels (forward, backward, FP8 prep) is
bounded.  The tests make the waits run out by setting a one-cycle wait
limit: the kernel must give up, record the site in the library's status word
and return (no hang), the host must see ATTN_ERR_DEVICE_TIMEOUT, and the CUDA
context must stay usable so that the next call, with the default limit, is
correct.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_71_gb300 import api, synth
from tests.helpers import assert_bf16_parity, errors, gpu_rows, lse_rows, to_dev

pytestmark = pytest.mark.gpu

ATTN_ERR_DEVICE_TIMEOUT = -4
FWD_SITES = {0x11, 0x12, 0x21, 0x22, 0x23, 0x24, 0x31, 0x32, 0x41}
BWD_SITES = {0x51, 0x52, 0x61, 0x62, 0x63, 0x64, 0x65, 0x66, 0x71, 0x72, 0x73, 0x74, 0x81, 0x82}
PREP_SITES = {0x91, 0x92, 0x93, 0x94}   # CUDA-core prep load; tensor-core prep load, MMA, producer
KNOWN_SITES = FWD_SITES


@pytest.mark.parametrize("d", [128, 256])
def test_wait_timeout_is_reported_and_the_context_survives(d):
    """d = 128 runs the two-tile kernel, d = 256 the one-tile kernel with
    the S pipeline in tensor memory."""
    B, N, H = 1, 1024, 2
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


def _timeout_then_recover(run):
    lib = api.library()
    assert api.device_status()[0] == 0
    assert lib.attn_set_wait_limit(1) == 0
    try:
        run()
        rc, site = api.device_status()
    finally:
        lib.attn_set_wait_limit(0)
    assert api.device_status()[0] == 0
    return rc, site


def test_backward_wait_timeout_is_reported_and_the_context_survives():
    B, N, H, d = 1, 700, 2, 128
    q, k, v = synth.qkv_bf16(B, N, H, d, seed=9)
    do = synth.tensor_bf16((B, N, H, d), seed=9, stream=4)
    qd, kd, vd, dod = (to_dev(x) for x in (q, k, v, do))
    o, lse = api.attn_fwd(qd, kd, vd, causal=True)
    want = api.attn_bwd(dod, qd, kd, vd, o, lse, causal=True)
    torch.cuda.synchronize()
    rc, site = _timeout_then_recover(lambda: api.attn_bwd(dod, qd, kd, vd, o, lse, causal=True))
    assert rc in (0, ATTN_ERR_DEVICE_TIMEOUT), rc
    if rc != 0:
        assert site in BWD_SITES, hex(site)
    got = api.attn_bwd(dod, qd, kd, vd, o, lse, causal=True)
    torch.cuda.synchronize()
    assert api.device_status()[0] == 0
    assert torch.equal(got[1], want[1]) and torch.equal(got[2], want[2])
    assert float((got[0].float() - want[0].float()).abs().max()) <= 1e-2 * float(want[0].float().abs().max())


@pytest.mark.parametrize("d", [128, 256])
def test_prep_wait_timeout_is_reported_and_the_context_survives(d):
    """d = 128 runs the tensor-core prep, d = 256 the CUDA-core one."""
    x = synth.tensor_bf16((2, 4096, 4, d), seed=3, stream=1)
    xd = to_dev(x)
    want = api.attn_fp8_prep(xd, mode=api.MODE_BLOCK_HADAMARD, sign_seed=7)
    torch.cuda.synchronize()
    rc, site = _timeout_then_recover(lambda: api.attn_fp8_prep(xd, mode=api.MODE_BLOCK_HADAMARD, sign_seed=7))
    assert rc in (0, ATTN_ERR_DEVICE_TIMEOUT), rc
    if rc != 0:
        assert site in PREP_SITES, hex(site)
    got = api.attn_fp8_prep(xd, mode=api.MODE_BLOCK_HADAMARD, sign_seed=7)
    torch.cuda.synchronize()
    assert torch.equal(got[0], want[0]) and torch.equal(got[1], want[1])


def test_fp8_head_dim_256_wait_timeout_is_reported_and_the_context_survives():
    B, N, H, d = 1, 1024, 2, 256
    q, k, v = synth.qkv_bf16(B, N, H, d, seed=10)
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    q8, k8, v8, qs, ks, vs = api.fp8_prepare_qkv(qd, kd, vd, api.MODE_BLOCK_HADAMARD, 3)
    want, want_lse = api.attn_fwd_fp8(q8, k8, v8, qs, ks, vs, causal=True)
    torch.cuda.synchronize()
    rc, site = _timeout_then_recover(lambda: api.attn_fwd_fp8(q8, k8, v8, qs, ks, vs, causal=True))
    assert rc == ATTN_ERR_DEVICE_TIMEOUT, (rc, site)
    assert site in FWD_SITES, hex(site)
    got, got_lse = api.attn_fwd_fp8(q8, k8, v8, qs, ks, vs, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int16), want.view(torch.int16)) and torch.equal(got_lse, want_lse)
    assert api.device_status()[0] == 0


def test_fused_qkv_prep_wait_timeout_is_reported_and_the_context_survives():
    B, N, H, Hkv, d = 2, 2048, 4, 2, 128
    q = to_dev(synth.tensor_bf16((B, N, H, d), seed=5, stream=1))
    k = to_dev(synth.tensor_bf16((B, N, Hkv, d), seed=5, stream=2))
    v = to_dev(synth.tensor_bf16((B, N, Hkv, d), seed=5, stream=3))
    want = api.attn_fp8_prep_qkv(q, k, v, api.MODE_BLOCK_HADAMARD, 11)
    torch.cuda.synchronize()
    rc, site = _timeout_then_recover(lambda: api.attn_fp8_prep_qkv(q, k, v, api.MODE_BLOCK_HADAMARD, 11))
    assert rc in (0, ATTN_ERR_DEVICE_TIMEOUT), rc
    if rc != 0:
        assert site in PREP_SITES, hex(site)
    got = api.attn_fp8_prep_qkv(q, k, v, api.MODE_BLOCK_HADAMARD, 11)
    torch.cuda.synchronize()
    for a, b in zip(got, want):
        assert torch.equal(a, b)
