"""GPU parity on the five workload configurations at their own sizes, through gptq_gemm (the call the
benchmark times, with the same gptq_reserve), against the CPU oracle.

  decode   K=4096  N=14336 4-bit g128, symmetric zero 8, bf16          M = 1, 8, 16
  gate     K=8192  N=28672 4-bit g128 act-order, asymmetric, fp16      M = 1, 2, 4, 16, 64
  prefill  K=8192  N=28672 4-bit g128, asymmetric, bf16                M = 512, 4096
  sweep    K=N=4096: bits 2/3/8 at g128, bits 4 at g-1/32/64 (fp16)    M = 1, 32, 256

These are the Llama-3-8B MLP and Llama-3-70B gate_proj shapes of mlinterviewnotes "Formats and
kernels: FP8, INT8, INT4, Marlin, Machete" (opening section: the 28672 x 8192 gate_proj layer).
The full products are too large for the oracle, so each case is checked on sampled outputs that
cover every part of the grid: the first and last 128 columns (first and last tiles, both ends of a
K-split and of a CTA's tile run) plus 256 random columns, and rows 0, M-1 and, for large M, two
seeded rows of every 128-row x tile.  Tolerance: max|y - y_ref| <= 4e-3 max|y_ref| on the sample.
Where a configuration exists to exercise one kernel variant, the test asserts that variant through
gptq_gemm_plan before it compares.
"""
import functools

import numpy as np
import pytest
import torch

import oracle
from weight_only_quantized_gb300 import gptq, synth

from gpu_util import compare

pytestmark = pytest.mark.gpu

DECODE = "llama3-8b-decode-4096x14336-b4g128-sym"
GATE = "llama3-70b-gate-8192x28672-b4g128-descact"
PREFILL = "prefill-8192x28672-b4g128"


@functools.lru_cache(maxsize=1)
def _layer(name):
    """(spec, checkpoint, handle) of one named workload; one layer at a time stays on the device."""
    spec, _ = synth.workload(name)
    return _build(spec, seed=11)


def _build(spec, seed):
    ck = synth.make_checkpoint(spec, seed=seed)
    d = [t.cuda() if t is not None else None for t in (ck.qweight, ck.qzeros, ck.scales, ck.g_idx)]
    h = gptq.gptq_repack(d[0], d[1], d[2], d[3], spec.bits, spec.group_size)
    torch.cuda.synchronize()
    return spec, ck, h


def _samples(M, N, seed):
    rng = np.random.default_rng(seed)
    cols = np.concatenate([np.arange(128), np.arange(N - 128, N), rng.choice(N, 256, replace=False)])
    rows = [0, M - 1]
    if M > 16:
        for t0 in range(0, M, 128):
            rows += list(rng.integers(t0, min(M, t0 + 128), 2))
    else:
        rows += list(range(M))
    return np.unique(np.array(rows, np.int32)), np.unique(cols.astype(np.int32))


def _check(spec, ck, h, M, seed):
    gptq.gptq_reserve(h, M)
    x = synth.make_x(M, spec.K, spec.dtype, seed=seed)
    dt = torch.float16 if spec.dtype == "fp16" else torch.bfloat16
    xd = x.cuda()
    y = torch.full((M, spec.N), float("nan"), dtype=dt, device="cuda")
    gptq.gptq_gemm(h, xd, y)
    torch.cuda.synchronize()
    gptq.gptq_device_status(h)
    rows, cols = _samples(M, spec.N, seed)
    yg = y[torch.from_numpy(rows).long().cuda()][:, torch.from_numpy(cols).long().cuda()].cpu()
    ref = oracle.linear(ck.qweight, ck.qzeros, ck.scales, ck.g_idx, spec.bits, spec.group_size, spec.dtype, x,
                        rows, cols)
    compare(yg, ref)
    assert torch.isfinite(y.float()).all(), "an output outside the sample was never written"


@pytest.mark.parametrize("M", [1, 8, 16])
def test_decode_layer(M):
    spec, ck, h = _layer(DECODE)
    _check(spec, ck, h, M, seed=100 + M)


@pytest.mark.parametrize("M", [1, 2, 4, 16, 64])
def test_gate_layer_act_order(M):
    spec, ck, h = _layer(GATE)
    plan = gptq.gptq_gemm_plan(h, M)
    if M <= 2:
        # the variant behind the M = 1 target: a long CTA (more than three tiles per SM) with 16
        # consumer warps, x permuted in shared memory, no gather pre-pass
        assert plan.path == gptq.PATH_SMALL_M and plan.consumer_warps == 16 and plan.act_order_in_kernel == 1
        assert plan.launches == 1
    elif M <= 16:
        assert plan.path == gptq.PATH_SMALL_M and plan.act_order_in_kernel == 0 and plan.launches == 2
    else:
        assert plan.path == gptq.PATH_LARGE_M
    _check(spec, ck, h, M, seed=200 + M)


@pytest.mark.parametrize("M", [512, 4096])
def test_prefill_layer(M):
    spec, ck, h = _layer(PREFILL)
    plan = gptq.gptq_gemm_plan(h, M)
    assert plan.path == gptq.PATH_LARGE_M and plan.m_tiles == 256
    _check(spec, ck, h, M, seed=300 + M)


def _sweep_id(s):
    return f"b{s.bits}g{s.group_size}{'-descact' if s.desc_act else ''}"


@pytest.mark.parametrize("spec", synth.format_sweep(), ids=_sweep_id)
def test_format_sweep(spec):
    _, ck, h = _build(spec, seed=spec.bits * 1000 + abs(spec.group_size))
    for M in synth.SWEEP_M:
        _check(spec, ck, h, M, seed=400 + M)
    h.close()


def test_gate_layer_plan_is_what_gptq_gemm_launches():
    """The plan query and the launch counter agree on every M of the gate layer."""
    spec, ck, h = _layer(GATE)
    for M in (1, 2, 3, 4, 16, 28, 29, 64):
        assert gptq.gptq_gemm_plan(h, M).launches == gptq.gptq_gemm_launches(h, M)
