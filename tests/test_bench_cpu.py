"""Host logic of bench.py (no GPU): the attended-pair and FLOP conventions
the throughput figures rest on, against brute-force counts, and the keys of
the sweep workloads."""
import numpy as np
import pytest

import bench


def brute_pairs(N, causal, window, block=None):
    """(query, key) pairs that take part: key j is visible to query i when
    j <= i (causal), j > i - window (window > 0) and the 128 x 128 block
    (i // 128, j // 128) is set (block mask)."""
    count = 0
    for i in range(N):
        for j in range(N):
            if causal and j > i:
                continue
            if window > 0 and j <= i - window:
                continue
            if block is not None and not block[i // 128, j // 128]:
                continue
            count += 1
    return count


@pytest.mark.parametrize("N", [1, 7, 128, 300])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("window", [0, 1, 5, 64])
def test_attended_pairs_match_a_brute_force_count(N, causal, window):
    assert bench.attended_pairs(N, causal, window) == brute_pairs(N, causal, window)


def test_flop_conventions():
    w = dict(B=2, H=3, N=256, d=64, causal=False, window=0, dtype="bf16")
    full = 4 * 2 * 3 * 256 * 256 * 64
    assert bench.flops_per_step(w) == full
    assert bench.flops_per_step(dict(w, causal=True)) == full / 2
    assert bench.flops_per_step(dict(w, direction="bwd")) == 2.5 * full
    assert bench.flops_per_step(dict(w, causal=True, window=50)) == 4 * 2 * 3 * 64 * brute_pairs(256, True, 50)


def test_block_sparse_pairs_match_a_brute_force_count():
    w = dict(B=1, H=2, N=1100, d=64, causal=True, window=0, dtype="bf16", sparse="band8_stride8")
    block = bench.block_mask(w)[0, 0].astype(bool)
    pairs = brute_pairs(1100, True, 0, block)
    assert bench.visible_pairs(w) == 2 * pairs
    assert bench.flops_per_step(w) == 4 * 64 * 2 * pairs
    rows = np.array([0, 127, 128, 600, 1099])
    assert bench.visible_pairs(w, rows) == 2 * sum(
        1 for i in rows for j in range(i + 1) if block[i // 128, j // 128])


def test_sweep_workload_keys():
    w = bench.workload("c3:4096:128:1")
    assert (w["B"], w["H"], w["N"], w["d"], w["causal"], w["dtype"]) == (4, 16, 4096, 128, True, "bf16")
    w = bench.workload("fp8:512:256:0")
    assert (w["B"], w["H"], w["N"], w["d"], w["causal"], w["dtype"]) == (32, 8, 512, 256, False, "fp8")
    w = bench.workload("bwd:16384:1:64")
    assert (w["B"], w["H"], w["N"], w["d"], w["causal"], w.get("direction")) == (1, 32, 16384, 64, True, "bwd")
    with pytest.raises(SystemExit):
        bench.workload("no-such-workload")
