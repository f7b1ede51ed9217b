"""Shared helpers of the GPU parity tests: tolerances, error metric and the
host copies handed to the oracle."""
import numpy as np
import torch

# Tolerances on max|x_gpu - x_ref| / rms(x_ref), over the compared tensor:
# fp32 inputs 1e-4, bf16 inputs with an fp32 state 2e-2.  They apply to the
# fp32 result of the kernel; a bf16 `out` is checked separately to be the
# round-to-nearest-even of that fp32 result, bit for bit (the store rounding
# alone reaches half a bf16 ulp of max|o|, about 2e-2 of rms(o) on these inputs).
TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


def rel_err(x, ref):
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = np.sqrt(np.mean(ref ** 2))
    if rms == 0.0:
        return float(np.max(np.abs(x - ref))) if x.size else 0.0
    return float(np.max(np.abs(x - ref)) / rms) if x.size else 0.0


def host64(t):
    return None if t is None else t.detach().to("cpu", torch.float64).numpy()


def bf16_rne(t32):
    """Round an fp32 tensor to bf16 (torch's cast is round-to-nearest-even)."""
    return t32.to(torch.bfloat16)
