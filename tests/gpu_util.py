"""Shared helpers of the GPU parity tests: put a synthetic checkpoint on the device, run the
library through its C ABI, and compare with the CPU oracle."""
import numpy as np
import torch

import oracle
from weight_only_quantized_gb300 import gptq, synth

# GEMM tolerance: max |y_gpu - y_ref| <= REL_TOL * max |y_ref| (fp32 accumulation, one rounding of
# y to fp16/bf16; bf16 output rounding alone is up to 2^-9 ~ 1.95e-3 of |y|).
REL_TOL = 4e-3


def to_device(ck: synth.Checkpoint, dev="cuda"):
    return dict(qweight=ck.qweight.to(dev), qzeros=ck.qzeros.to(dev), scales=ck.scales.to(dev),
                g_idx=None if ck.g_idx is None else ck.g_idx.to(dev))


def repack(ck: synth.Checkpoint) -> gptq.Handle:
    d = to_device(ck)
    h = gptq.gptq_repack(d["qweight"], d["qzeros"], d["scales"], d["g_idx"], ck.spec.bits, ck.spec.group_size)
    torch.cuda.synchronize()
    return h


def run_gemm(h, x_cpu: torch.Tensor, N: int, path=gptq.PATH_AUTO) -> torch.Tensor:
    x = x_cpu.cuda()
    y = torch.full((x.shape[0], N), float("nan"), dtype=x.dtype, device="cuda")
    gptq.gptq_gemm_path(h, x, y, path)
    torch.cuda.synchronize()
    return y.cpu()


def oracle_y(ck: synth.Checkpoint, x_cpu, rows=None, cols=None) -> np.ndarray:
    s = ck.spec
    return oracle.linear(ck.qweight, ck.qzeros, ck.scales, ck.g_idx, s.bits, s.group_size, s.dtype, x_cpu, rows, cols)


def compare(y_gpu: torch.Tensor, y_ref: np.ndarray, tol=REL_TOL) -> dict:
    g = y_gpu.double().numpy()
    assert g.shape == y_ref.shape
    assert np.all(np.isfinite(g)), "non-finite outputs"
    scale = float(np.max(np.abs(y_ref)))
    err = float(np.max(np.abs(g - y_ref)))
    # error that rounding y_ref to the output dtype alone implies, reported apart from arithmetic error
    rounded = torch.from_numpy(y_ref).to(y_gpu.dtype).double().numpy()
    round_err = float(np.max(np.abs(rounded - y_ref)))
    info = dict(max_abs_err=err, max_ref=scale, rel=err / max(scale, 1e-30), output_rounding=round_err / max(scale, 1e-30))
    assert err <= tol * scale, info
    return info
