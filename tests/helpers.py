"""Shared helpers of the parity tests (no attention arithmetic here)."""
import numpy as np
import torch

from exact_attention_71_gb300 import synth

# Tolerances against the fp64 oracle for the bf16 path (max-abs, RMS, LSE).
BF16_MAX_ABS = 1e-2
BF16_RMS = 2e-3
LSE_ABS = 1e-3
FP8_RMS = 3e-2
# FP8 path, LSE against the oracle run on the dequantised codes.  P's
# exponentials use FP16 intermediates: the argument (which carries the V
# block factor's log2, <= 4, so the keys that carry the weight have arguments
# up to 8.8) is rounded to f16, at most 2^-8 absolute there, i.e. <= 2.7e-3
# relative in P; the f16 result adds ~2^-10; the row sum is kept in f16
# partial sums of 16 terms (~4 * 2^-11 / sqrt(3) ~ 1.1e-3 random-walk,
# 16 * 2^-11 ~ 7.8e-3 worst case).  ln l is off by their sum, ~5e-3 in the
# worst rows of a large sample; gated at 1e-2.
FP8_LSE = 1e-2


def to_dev(bits: np.ndarray, device="cuda") -> torch.Tensor:
    """uint16 bf16 bit pattern array -> bf16 CUDA tensor."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def gpu_rows(o: torch.Tensor, rows) -> np.ndarray:
    """(B, N, H, d) device output -> float64 (B, H, R, d) for the given rows."""
    idx = torch.as_tensor(np.asarray(rows, dtype=np.int64), device=o.device)
    return o.index_select(1, idx).permute(0, 2, 1, 3).double().cpu().numpy()


def lse_rows(lse: torch.Tensor, rows) -> np.ndarray:
    idx = torch.as_tensor(np.asarray(rows, dtype=np.int64), device=lse.device)
    return lse.index_select(2, idx).double().cpu().numpy()


def bf16_half_ulp(x: np.ndarray) -> np.ndarray:
    """Half a bf16 ulp at |x| (the output-rounding floor)."""
    a = np.maximum(np.abs(x), 2.0 ** -126)
    e = np.floor(np.log2(a))
    return np.exp2(e - 8)


def errors(o_gpu, o_ref, lse_gpu, lse_ref):
    err = np.abs(o_gpu - o_ref)
    return dict(max_abs=float(err.max()), rms=float(np.sqrt(np.mean(err ** 2))),
                lse=float(np.max(np.abs(lse_gpu - lse_ref))),
                # error beyond the bf16 rounding of the exact output
                max_excess=float(np.max(err - bf16_half_ulp(o_ref))))


def assert_bf16_parity(e, label=""):
    """The bf16 bar: max-abs <= 1e-2, RMS <= 2e-3, LSE <= 1e-3 against fp64.

    Elements whose exact value is >= 4 in magnitude have a bf16 half-ulp of
    2^-6 > 1e-2, so the output cast alone can exceed 1e-2 there; such a case
    is reported (max_excess = error beyond half an ulp) rather than hidden:
    the assertion then requires max_excess <= 1e-2 instead.
    """
    msg = f"{label}: {e}"
    assert e["rms"] <= BF16_RMS, msg
    assert e["lse"] <= LSE_ABS, msg
    if e["max_abs"] > BF16_MAX_ABS:
        assert e["max_excess"] <= BF16_MAX_ABS, msg
        print(f"[cast floor] {label}: max-abs {e['max_abs']:.3e} exceeds 1e-2 only through the bf16 "
              f"output rounding (error beyond half an ulp {e['max_excess']:.3e})")


def assert_codes_match_up_to_midpoints(c_gpu, c_ref, s_ref, rot, block_rows=128, max_frac=1e-3):
    """e4m3 codes of a rotated tensor: equal to the oracle's, except where the
    oracle's exact quotient rot / scale lies within 1e-5 (relative) of a
    rounding midpoint between two e4m3 values -- the float32 butterflies and
    the oracle's double product may round to either side there -- and then
    only to a neighbouring code."""
    import oracle
    vals = np.unique(np.abs(oracle.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))))
    mids = (vals[:-1] + vals[1:]) / 2
    N = c_ref.shape[1]
    sc = np.repeat(s_ref.transpose(0, 2, 1), block_rows, axis=1)[:, :N]      # (B, N, H)
    y = rot.astype(np.float64) / sc[..., None]
    a = np.abs(y).ravel()
    pos = np.searchsorted(mids, a)
    near = np.minimum(np.abs(a - mids[np.clip(pos - 1, 0, len(mids) - 1)]),
                      np.abs(a - mids[np.clip(pos, 0, len(mids) - 1)])) <= 1e-5 * np.maximum(a, 2.0 ** -9)
    cg, cr = c_gpu.ravel(), c_ref.ravel()
    same = cg == cr
    assert np.all(same | near), f"{np.sum(~(same | near))} codes differ away from a rounding midpoint"
    diff = ~same
    mg, mr = (cg[diff] & 0x7F).astype(int), (cr[diff] & 0x7F).astype(int)
    same_sign = (cg[diff] & 0x80) == (cr[diff] & 0x80)
    assert np.all((np.abs(mg - mr) == 1) & (same_sign | (np.minimum(mg, mr) == 0)))
    assert diff.mean() < max_frac


def dequant(codes, scales, block_rows=128):
    """e4m3 codes (B,N,H,d) torch tensor x block scales (B,H,nblk) -> float64 values."""
    import oracle
    c = codes.cpu().numpy()
    s = scales.cpu().numpy().astype(np.float64)
    N = c.shape[1]
    vals = oracle.e4m3_decode(c.ravel()).reshape(c.shape)
    sc = np.repeat(s.transpose(0, 2, 1), block_rows, axis=1)[:, :N]
    return vals * sc[..., None]
