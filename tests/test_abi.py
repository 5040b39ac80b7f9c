"""The C ABI library: it builds, loads without a GPU, exports every entry
point include/attn.h declares, and rejects bad arguments before any launch."""
import ctypes
import os
import re

import pytest

from exact_attention_71_gb300 import api, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:int|size_t|const char\*)\s+(attn_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return api.library()


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("attn_fwd", "attn_fwd_fp8", "attn_fp8_prep", "attn_last_error_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


FAKE = ctypes.c_void_p(1 << 20)   # never dereferenced: the checks fail first


@pytest.mark.parametrize("d", [32, 96, 512])
def test_unsupported_head_dim_rejected(lib, d):
    rc = lib.attn_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 16, d, 0, 0.0, 0, None)
    assert rc == -2
    assert b"head_dim" in lib.attn_last_error_string()


def test_negative_sizes_and_window_rejected(lib):
    assert lib.attn_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, -1, 1, 16, 128, 0, 0.0, 0, None) == -1
    assert lib.attn_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 16, 128, 0, 0.0, -5, None) == -1


def test_null_and_misaligned_pointers_rejected(lib):
    assert lib.attn_fwd(None, FAKE, FAKE, FAKE, FAKE, 1, 1, 16, 128, 0, 0.0, 0, None) == -1
    odd = ctypes.c_void_p((1 << 20) + 8)
    assert lib.attn_fwd(FAKE, odd, FAKE, FAKE, FAKE, 1, 1, 16, 128, 0, 0.0, 0, None) == -1
    assert b"aligned" in lib.attn_last_error_string()


def test_empty_problem_is_ok_without_launch(lib):
    assert lib.attn_fwd(None, None, None, None, None, 0, 4, 16, 128, 1, 0.0, 0, None) == 0
    assert lib.attn_fwd(None, None, None, None, None, 2, 4, 0, 128, 1, 0.0, 0, None) == 0


def test_fp8_arguments_checked(lib):
    assert lib.attn_fwd_fp8(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 16, 96, 0, 0.0, 0, FAKE, FAKE, FAKE, None) == -2
    assert lib.attn_fwd_fp8(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 16, 128, 0, 0.0, 0, None, FAKE, FAKE, None) == -1


def test_prep_arguments_checked(lib):
    assert lib.attn_fp8_prep(FAKE, FAKE, FAKE, 1, 1, 16, 128, 64, 1, 0, 0, None) == -2
    assert lib.attn_fp8_prep(FAKE, FAKE, FAKE, 1, 1, 16, 128, 128, 3, 0, 0, None) == -1
    assert lib.attn_fp8_prep(FAKE, FAKE, FAKE, 1, 1, 16, 96, 128, 1, 0, 0, None) == -2
    assert lib.attn_fp8_prep(None, None, None, 1, 1, 0, 128, 128, 1, 0, 0, None) == 0


def test_wait_limit_setter(lib):
    assert lib.attn_set_wait_limit(0) == 0


def test_gqa_head_count_checked(lib):
    assert lib.attn_fwd_gqa(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 6, 4, 16, 128, 0, 0.0, 0, None) == -1
    assert b"divide" in lib.attn_last_error_string()
    assert lib.attn_fwd_gqa(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 6, 0, 16, 128, 0, 0.0, 0, None) == -1
    assert lib.attn_fwd_fp8_gqa(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 8, 3, 16, 128, 0, 0.0, 0, FAKE, FAKE, FAKE,
                                None) == -1


def test_rope_prep_arguments_checked(lib):
    f = lib.attn_fp8_prep_rope
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 16, 96, 128, 1, 0, 0, None) == -2       # head_dim
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 16, 128, 64, 1, 0, 0, None) == -2       # block rows
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 16, 128, 128, 5, 0, 0, None) == -1      # mode
    assert f(FAKE, FAKE, FAKE, None, FAKE, 1, 1, 16, 128, 128, 1, 0, 0, None) == -1      # no cos table
    assert b"null" in lib.attn_last_error_string()
    odd = ctypes.c_void_p((1 << 20) + 4)
    assert f(FAKE, FAKE, FAKE, FAKE, odd, 1, 1, 16, 128, 128, 1, 0, 0, None) == -1       # unaligned sin
    assert b"aligned" in lib.attn_last_error_string()
    assert f(None, None, None, None, None, 0, 1, 16, 128, 128, 1, 0, 0, None) == 0       # empty


def test_backward_arguments_checked(lib):
    f = lib.attn_bwd
    ws = lib.attn_bwd_workspace_size(1, 2, 100, 128)
    # (2 x float32 per padded row) + float32 dQ accumulator, 256-byte aligned parts
    assert ws == 2 * 1024 + 2 * 128 * 128 * 4
    assert lib.attn_bwd_workspace_size(-1, 2, 100, 128) == 0
    args = lambda d=128, hkv=2, wsp=FAKE, wsb=ws: (FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, wsp, wsb,
                                                   1, 2, hkv, 100, d, 1, 0.0, 0, None)
    assert f(*args(d=256)) == -2
    assert f(*args(hkv=3)) == -1
    assert f(*args(wsp=None)) == -1
    assert f(*args(wsp=ctypes.c_void_p((1 << 20) + 16))) == -1
    assert b"256-byte" in lib.attn_last_error_string()
    assert f(*args(wsb=ws - 1)) == -1
    assert b"smaller" in lib.attn_last_error_string()


def test_sparse_arguments_checked(lib):
    f = lib.attn_fwd_sparse
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, None, 1, 2, 2, 100, 128, 0, 0.0, 0, None) == -1
    assert b"mask" in lib.attn_last_error_string()
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 2, 3, 100, 128, 0, 0.0, 0, None) == -1
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 2, 2, 100, 96, 0, 0.0, 0, None) == -2
    assert f(None, None, None, None, None, None, 1, 2, 2, 0, 128, 0, 0.0, 0, None) == 0


def test_host_forward_workspace_and_arguments(lib):
    """attn_fwd_host: two staging slots of whole-sequence chunks (at most four
    chunks per call); its argument checks run before any CUDA call."""
    size = lib.attn_fwd_host_workspace_size
    # B=3 -> 3 chunks of 1 sequence: Q, K, V, O, LSE parts rounded to 256 bytes
    q_seq, kv_seq, l_seq = 100 * 2 * 128 * 2, 100 * 1 * 128 * 2, 2 * 100 * 4
    up = lambda x: (x + 255) // 256 * 256
    slot = 2 * up(q_seq) + 2 * up(kv_seq) + up(l_seq)
    assert size(3, 2, 1, 100, 128) == 2 * slot
    # B=10 -> chunks of ceil(10 / 4) = 3 sequences
    assert size(10, 2, 1, 100, 128) == 2 * (2 * up(3 * q_seq) + 2 * up(3 * kv_seq) + up(3 * l_seq))
    assert size(-1, 2, 1, 100, 128) == 0 and size(1, 2, 0, 100, 128) == 0
    f = lib.attn_fwd_host
    ws = size(3, 2, 1, 100, 128)
    args = lambda d=128, hkv=1, wsp=FAKE, wsb=ws: (FAKE, FAKE, FAKE, FAKE, FAKE, 3, 2, hkv, 100, d, 1, 0.0, 0, wsp,
                                                   wsb, None)
    assert f(*args(d=96)) == -2
    assert f(*args(hkv=3)) == -1
    assert f(*args(wsp=None)) == -1
    assert f(*args(wsp=ctypes.c_void_p((1 << 20) + 16))) == -1
    assert b"256-byte" in lib.attn_last_error_string()
    assert f(*args(wsb=ws - 1)) == -1
    assert f(None, None, None, None, None, 0, 2, 1, 100, 128, 0, 0.0, 0, None, 0, None) == 0


def test_fp8_host_forward_workspace_and_arguments(lib):
    """attn_fwd_fp8_host: the slots of attn_fwd_host plus each chunk's e4m3
    codes and block scales; the per-tensor mode is refused (its one scale
    would span chunks)."""
    size = lib.attn_fwd_fp8_host_workspace_size
    up = lambda x: (x + 255) // 256 * 256
    B, H, Hkv, N, d = 3, 2, 1, 100, 128
    bf16_slot = lib.attn_fwd_host_workspace_size(B, H, Hkv, N, d) // 2
    nblk = 1
    codes = up(N * H * d) + 2 * up(N * Hkv * d)
    scales = up(H * nblk * 4) + 2 * up(Hkv * nblk * 4)
    assert size(B, H, Hkv, N, d) == 2 * (bf16_slot + codes + scales)
    assert size(0, H, Hkv, N, d) == 0
    f = lib.attn_fwd_fp8_host
    ws = size(B, H, Hkv, N, d)
    args = lambda mode=1, d=128, wsb=ws: (FAKE, FAKE, FAKE, FAKE, FAKE, B, H, Hkv, N, d, 0, 0.0, 0, mode, 7, FAKE,
                                          wsb, None)
    assert f(*args(mode=2)) == -1
    assert b"mode" in lib.attn_last_error_string()
    assert f(*args(d=96)) == -2
    assert f(*args(wsb=ws - 1)) == -1


def test_bwd_host_workspace_and_arguments(lib):
    """attn_bwd_host: per slot Q, K, V, O, LSE, dO in and dQ, dK, dV out for
    one chunk, plus that chunk's backward workspace."""
    size = lib.attn_bwd_host_workspace_size
    up = lambda x: (x + 255) // 256 * 256
    B, H, Hkv, N, d = 3, 2, 1, 100, 128
    q_seq, kv_seq, l_seq = N * H * d * 2, N * Hkv * d * 2, H * N * 4
    parts = [q_seq, kv_seq, kv_seq, q_seq, l_seq, q_seq, q_seq, kv_seq, kv_seq]
    slot = sum(up(x) for x in parts) + up(lib.attn_bwd_workspace_size(1, H, N, d))
    assert size(B, H, Hkv, N, d) == 2 * slot
    assert size(B, H, 0, N, d) == 0
    f = lib.attn_bwd_host
    ws = size(B, H, Hkv, N, d)
    args = lambda d=128, wsb=ws: (FAKE,) * 9 + (B, H, Hkv, N, d, 1, 0.0, 0, FAKE, wsb, None)
    assert f(*args(d=256)) == -2
    assert f(*args(wsb=ws - 1)) == -1


def test_host_bindings_check_their_arguments(lib):
    """The host-buffer bindings reject device tensors, wrong dtypes, shapes
    and outputs before calling the library (no GPU needed)."""
    import torch
    q = torch.zeros(2, 16, 4, 64, dtype=torch.bfloat16)
    k = torch.zeros(2, 16, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        api.attn_fwd_host(q.float(), k, k)                      # dtype
    with pytest.raises(ValueError):
        api.attn_fwd_host(q, k, k[:, :8])                       # k / v shapes differ
    with pytest.raises(ValueError):
        api.attn_fwd_host(q, torch.zeros(2, 16, 3, 64, dtype=torch.bfloat16),
                          torch.zeros(2, 16, 3, 64, dtype=torch.bfloat16))   # 3 does not divide 4
    with pytest.raises(ValueError):
        api.attn_fwd_host(q, k, k, out=torch.zeros(2, 16, 4, 32, dtype=torch.bfloat16))
    with pytest.raises(ValueError):
        api.attn_fwd_fp8_host(q, k, k, lse=torch.zeros(2, 4, 8))
    with pytest.raises(ValueError):
        api.attn_bwd_host(q[:, :8], q, k, k, q, torch.zeros(2, 4, 16))     # dout shaped unlike q
    with pytest.raises(ValueError):
        api.attn_bwd_host(q, q, k, k, q, torch.zeros(2, 4, 16), dk=torch.zeros(2, 16, 4, 64, dtype=torch.bfloat16))


@pytest.mark.parametrize("nmb,bh,grid", [(16, 64, 152), (64, 16, 152), (16, 19, 152), (1, 200, 152),
                                          (7, 111, 152), (16, 128, 152), (3, 5, 7), (32, 64, 152)])
def test_causal_work_order(lib, nmb, bh, grid):
    """The causal forward's host-built work order: a permutation of the
    items; every full round numbered heaviest query block first; the last,
    partial round holds the lightest items; the zigzag over rounds balances
    the per-CTA work (query block q of a head costs 4q + 3 key blocks of 128);
    and a full round touches few heads."""
    order = api.fwd_work_order(nmb, bh, grid)
    n = nmb * bh
    assert order is not None and len(order) == n
    assert sorted(order) == sorted((m, h) for h in range(bh) for m in range(nmb))
    full = n // grid * grid
    per_head = nmb - -(-(n - full) // bh)           # fewest items a head keeps outside the last round
    for r in range(0, full, grid):
        mbs = [m for m, _ in order[r:r + grid]]
        assert mbs == sorted(mbs, reverse=True)
        heads = {h for _, h in order[r:r + grid]}
        assert len(heads) <= -(-grid // max(per_head, 1)) + 1
    tail = order[full:]
    if tail and full:
        assert max((m, h) for m, h in tail) < min((m, h) for m, h in order[:full])
    load = [0] * grid
    for i, (m, _) in enumerate(order):
        rnd, c = divmod(i, grid)
        load[c if rnd % 2 == 0 else grid - 1 - c] += 4 * m + 3
    # No CTA's work exceeds the mean by a whole heaviest item (items are
    # indivisible; 3-7 % above the mean for the larger shapes here).
    assert max(load) - sum(load) / grid <= 4 * (nmb - 1) + 3


def test_causal_work_order_beyond_the_table(lib):
    assert api.fwd_work_order(64, 40, 152) is None      # 2560 items: the closed-form order
    assert lib.attn_fwd_work_order(4, 4, 4, None, 16) == 0
