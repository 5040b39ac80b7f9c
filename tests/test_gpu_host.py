"""attn_fwd_host (the forward on host buffers, chunked through two device
staging slots) returns exactly what attn_fwd returns on the same data, for
ragged chunkings, grouped heads, masks and back-to-back calls that overlap."""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_71_gb300 import api, synth

pytestmark = pytest.mark.gpu


def host_qkv(B, N, H, Hkv, d, seed, pin=True):
    q = synth.tensor_bf16((B, N, H, d), seed=seed, stream=1)
    k = synth.tensor_bf16((B, N, Hkv, d), seed=seed, stream=2)
    v = synth.tensor_bf16((B, N, Hkv, d), seed=seed, stream=3)
    t = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    out = tuple(t(a) for a in (q, k, v))
    return tuple(x.pin_memory() for x in out) if pin else out


@pytest.mark.parametrize("B,N,H,Hkv,d,causal,window", [
    (3, 1000, 4, 2, 128, True, 0),      # 3 chunks of 1 sequence, grouped heads, ragged N
    (5, 777, 2, 2, 64, False, 0),       # chunks of 2, 2, 1
    (1, 300, 2, 1, 256, True, 100),     # one chunk, multi-query, sliding window
    (9, 512, 8, 8, 128, True, 0),       # chunks of 3
])
def test_host_forward_matches_device_forward(B, N, H, Hkv, d, causal, window):
    q, k, v = host_qkv(B, N, H, Hkv, d, seed=B * 100 + d)
    o, lse = api.attn_fwd_host(q, k, v, causal=causal, window=window)
    torch.cuda.synchronize()
    dev = torch.device("cuda:0")
    o_ref, lse_ref = api.attn_fwd(q.to(dev), k.to(dev), v.to(dev), causal=causal, window=window)
    torch.cuda.synchronize()
    assert api.device_status() == (0, 0)
    assert torch.equal(o.view(torch.int16), o_ref.cpu().view(torch.int16))
    assert torch.equal(lse, lse_ref.cpu())


def test_host_forward_against_oracle():
    B, N, H, d = 2, 200, 2, 64
    q, k, v = host_qkv(B, N, H, H, d, seed=7)
    o, lse = api.attn_fwd_host(q, k, v, causal=True)
    torch.cuda.synchronize()
    as_np = lambda t: t.view(torch.int16).numpy().view(np.uint16)
    o_ref, lse_ref = oracle.attention(as_np(q), as_np(k), as_np(v), causal=True)
    err = np.abs(o.float().permute(0, 2, 1, 3).double().numpy() - o_ref)
    assert err.max() <= 1e-2 and np.sqrt(np.mean(err ** 2)) <= 2e-3
    assert np.abs(lse.double().numpy() - lse_ref).max() <= 1e-3


def test_back_to_back_calls_and_pageable_memory():
    """Calls queued without a synchronisation in between share the staging
    slots (their copies overlap); each still gets its own result.  Pageable
    host memory works too (the copies then do not overlap)."""
    dev = torch.device("cuda:0")
    B, N, H, d = 4, 640, 4, 128
    ws = torch.empty(api.fwd_host_workspace_bytes(B, H, H, N, d), dtype=torch.uint8, device=dev)
    runs = []
    for i in range(5):
        q, k, v = host_qkv(B, N, H, H, d, seed=50 + i, pin=(i != 3))
        runs.append(((q, k, v), api.attn_fwd_host(q, k, v, causal=bool(i & 1), workspace=ws)))
    torch.cuda.synchronize()
    for i, ((q, k, v), (o, lse)) in enumerate(runs):
        o_ref, lse_ref = api.attn_fwd(q.to(dev), k.to(dev), v.to(dev), causal=bool(i & 1))
        assert torch.equal(o.view(torch.int16), o_ref.cpu().view(torch.int16)), i
        assert torch.equal(lse, lse_ref.cpu()), i
    assert api.device_status() == (0, 0)


def test_two_streams_and_changing_shapes_share_a_workspace():
    """Calls in flight on two streams share one workspace, and calls of
    different shapes (different staging layouts) follow each other without a
    synchronisation; every result matches the device forward."""
    dev = torch.device("cuda:0")
    shapes = [(2, 1024, 8, 128), (3, 500, 4, 64), (2, 1024, 8, 128), (1, 2048, 2, 256), (4, 256, 8, 128)]
    ws = torch.empty(max(api.fwd_host_workspace_bytes(B, H, H, N, d) for B, N, H, d in shapes),
                     dtype=torch.uint8, device=dev)
    streams = [torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)]
    runs = []
    for i, (B, N, H, d) in enumerate(shapes * 2):
        q, k, v = host_qkv(B, N, H, H, d, seed=200 + i)
        runs.append(((q, k, v), i, api.attn_fwd_host(q, k, v, causal=bool(i % 3), workspace=ws,
                                                      stream=streams[i & 1])))
    torch.cuda.synchronize()
    for (q, k, v), i, (o, lse) in runs:
        o_ref, lse_ref = api.attn_fwd(q.to(dev), k.to(dev), v.to(dev), causal=bool(i % 3))
        assert torch.equal(o.view(torch.int16), o_ref.cpu().view(torch.int16)), i
        assert torch.equal(lse, lse_ref.cpu()), i
    assert api.device_status() == (0, 0)


@pytest.mark.parametrize("B,N,H,Hkv,d,causal,mode", [
    (3, 1000, 4, 2, 128, True, api.MODE_BLOCK_HADAMARD),
    (5, 777, 2, 2, 64, False, api.MODE_BLOCK),
    (2, 512, 2, 1, 256, True, api.MODE_BLOCK_HADAMARD),
])
def test_fp8_host_forward_matches_device_path(B, N, H, Hkv, d, causal, mode):
    """attn_fwd_fp8_host = attn_fp8_prep of Q, K, V + attn_fwd_fp8 on the
    device, bit for bit (block scales are per sequence, so chunking does not
    change them)."""
    q, k, v = host_qkv(B, N, H, Hkv, d, seed=300 + d)
    o, lse = api.attn_fwd_fp8_host(q, k, v, mode=mode, sign_seed=99, causal=causal)
    torch.cuda.synchronize()
    dev = torch.device("cuda:0")
    q8, k8, v8, qs, ks, vs = api.fp8_prepare_qkv(q.to(dev), k.to(dev), v.to(dev), mode, 99)
    o_ref, lse_ref = api.attn_fwd_fp8(q8, k8, v8, qs, ks, vs, causal=causal)
    torch.cuda.synchronize()
    assert api.device_status() == (0, 0)
    assert torch.equal(o.view(torch.int16), o_ref.cpu().view(torch.int16))
    assert torch.equal(lse, lse_ref.cpu())


def test_fp8_and_bf16_host_calls_interleave():
    """FP8 and bf16 host calls of different layouts, in flight on two streams
    with one shared workspace, each return their own device-path result."""
    dev = torch.device("cuda:0")
    B, N, H, d = 4, 640, 4, 128
    ws = torch.empty(api.fwd_fp8_host_workspace_bytes(B, H, H, N, d), dtype=torch.uint8, device=dev)
    streams = [torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)]
    runs = []
    for i in range(6):
        q, k, v = host_qkv(B, N, H, H, d, seed=400 + i)
        if i % 2:
            res = api.attn_fwd_fp8_host(q, k, v, sign_seed=5, causal=True, workspace=ws, stream=streams[i % 2])
        else:
            res = api.attn_fwd_host(q, k, v, causal=True, workspace=ws, stream=streams[i % 2])
        runs.append(((q, k, v), i, res))
    torch.cuda.synchronize()
    for (q, k, v), i, (o, lse) in runs:
        qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
        if i % 2:
            q8, k8, v8, qs, ks, vs = api.fp8_prepare_qkv(qd, kd, vd, api.MODE_BLOCK_HADAMARD, 5)
            o_ref, lse_ref = api.attn_fwd_fp8(q8, k8, v8, qs, ks, vs, causal=True)
        else:
            o_ref, lse_ref = api.attn_fwd(qd, kd, vd, causal=True)
        assert torch.equal(o.view(torch.int16), o_ref.cpu().view(torch.int16)), i
        assert torch.equal(lse, lse_ref.cpu()), i
    assert api.device_status() == (0, 0)


@pytest.mark.parametrize("B,N,H,Hkv,d,causal", [(3, 700, 4, 2, 128, True), (5, 384, 2, 2, 64, False)])
def test_bwd_host_matches_device_backward(B, N, H, Hkv, d, causal):
    """attn_bwd_host = attn_bwd on the device: dK and dV bit for bit (one CTA
    owns each key block); dQ up to the order of its float32 accumulation
    (bulk adds from several CTAs), checked against the oracle as well."""
    dev = torch.device("cuda:0")
    q, k, v = host_qkv(B, N, H, Hkv, d, seed=500 + d)
    do = torch.from_numpy(synth.tensor_bf16((B, N, H, d), seed=500 + d, stream=4).view(np.int16)).view(
        torch.bfloat16).pin_memory()
    o_d, lse_d = api.attn_fwd(q.to(dev), k.to(dev), v.to(dev), causal=causal)
    o, lse = o_d.cpu().pin_memory(), lse_d.cpu().pin_memory()
    dq, dk, dv = api.attn_bwd_host(do, q, k, v, o, lse, causal=causal)
    torch.cuda.synchronize()
    rq, rk, rv = api.attn_bwd(do.to(dev), q.to(dev), k.to(dev), v.to(dev), o_d, lse_d, causal=causal)
    torch.cuda.synchronize()
    assert api.device_status() == (0, 0)
    assert torch.equal(dk.view(torch.int16), rk.cpu().view(torch.int16))
    assert torch.equal(dv.view(torch.int16), rv.cpu().view(torch.int16))
    diff = (dq.float() - rq.cpu().float()).abs().max().item()
    assert diff <= 2e-2 * rq.float().abs().max().item()
    as_np = lambda t: t.view(torch.int16).numpy().view(np.uint16)
    refs = oracle.attention_bwd(as_np(q), as_np(k), as_np(v), as_np(do), causal=causal)
    for g, r in zip((dq, dk, dv), refs):
        g = g.float().double().numpy()
        assert np.linalg.norm(g - r) / np.linalg.norm(r) <= 5e-3


def test_binding_allocated_workspace_survives_reuse_pressure():
    """A workspace the binding allocates is released while the library's
    streams still use it; it is recorded on the caller's stream, so fresh
    allocations (filled right away) cannot take its memory early."""
    dev = torch.device("cuda:0")
    s = torch.cuda.Stream(device=dev)
    B, N, H, d = 3, 1024, 8, 128
    q, k, v = host_qkv(B, N, H, H, d, seed=600)
    with torch.cuda.stream(s):
        o, lse = api.attn_fwd_host(q, k, v, causal=True, stream=s)
        junk = [torch.full((1 << 22,), 7.0, device=dev) for _ in range(16)]   # 256 MB of new allocations
    o2, lse2 = api.attn_fwd_host(q, k, v, causal=True, stream=s.cuda_stream)  # stream as a raw handle
    torch.cuda.synchronize()
    o_ref, lse_ref = api.attn_fwd(q.to(dev), k.to(dev), v.to(dev), causal=True)
    torch.cuda.synchronize()
    for a, b_ in ((o, o_ref), (o2, o_ref)):
        assert torch.equal(a.view(torch.int16), b_.cpu().view(torch.int16))
    assert torch.equal(lse, lse_ref.cpu()) and torch.equal(lse2, lse_ref.cpu())
    del junk
