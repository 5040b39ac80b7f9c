"""Shared helpers of the parity tests (no attention arithmetic here)."""
import numpy as np
import torch

from exact_attention_71_gb300 import synth

# Tolerances against the fp64 oracle for the bf16 path (max-abs, RMS, LSE).
BF16_MAX_ABS = 1e-2
BF16_RMS = 2e-3
LSE_ABS = 1e-3
FP8_RMS = 3e-2


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
