"""GPU parity of the large-M kernel's K split against the oracle, on layers whose grid would leave
SMs idle: the K ranges of an output tile are the CTAs of one thread-block cluster, each keeps its
fp32 partial in its shared memory, and CTA z sums the z-th slice of the tile's rows over all ranges
in range order (distributed shared memory reads)."""
import numpy as np
import pytest
import torch

import oracle
from weight_only_quantized_gb300 import gptq, synth

from gpu_util import compare, oracle_y, repack, run_gemm

pytestmark = pytest.mark.gpu

SPECS = [
    synth.LayerSpec(2048, 256, 4, 128, False, False, "bf16"),
    synth.LayerSpec(4096, 384, 4, 128, True, False, "fp16"),      # act-order: groups cross the ranges
    synth.LayerSpec(3072, 288, 3, 64, True, False, "bf16"),
    synth.LayerSpec(4096, 256, 8, 32, False, False, "fp16"),
    synth.LayerSpec(4096, 512, 2, -1, False, True, "bf16"),
]


def _id(s):
    return f"K{s.K}N{s.N}b{s.bits}g{s.group_size}{'da' if s.desc_act else ''}{s.dtype}"


@pytest.mark.parametrize("spec", SPECS, ids=_id)
@pytest.mark.parametrize("M", [1, 40, 64, 65, 129, 300])
def test_split_parity_and_determinism(spec, M):
    ck = synth.make_checkpoint(spec, seed=spec.K + M)
    h = repack(ck)
    splits = gptq.gptq_gemm_k_splits(h, M, gptq.PATH_LARGE_M)
    assert splits > 1                                   # no workspace needed for the split
    gptq.gptq_reserve(h, 300)                           # (act-order: the permuted x above M = 32)
    assert gptq.gptq_gemm_k_splits(h, M, gptq.PATH_LARGE_M) == splits
    assert gptq.gptq_gemm_plan(h, M, gptq.PATH_LARGE_M).k_splits == splits
    x = synth.make_x(M, spec.K, spec.dtype, seed=M)
    y1 = run_gemm(h, x, spec.N, gptq.PATH_LARGE_M)
    compare(y1, oracle_y(ck, x))
    assert torch.equal(y1, run_gemm(h, x, spec.N, gptq.PATH_LARGE_M))   # same sum order every call


def test_split_with_bias_awq_and_fp8():
    K, N = 4096, 256
    b = torch.randn(N, generator=torch.Generator().manual_seed(2)) * 0.1
    ck = synth.make_awq_checkpoint(K, N, 128, "fp16", seed=3)
    h = gptq.gptq_repack_awq(ck.qweight.cuda(), ck.qzeros.cuda(), ck.scales.cuda(), 128)
    gptq.gptq_set_bias(h, b.half().cuda())
    assert gptq.gptq_gemm_k_splits(h, 64) > 1
    x = synth.make_x(64, K, "fp16", seed=4)
    y_ref = oracle.awq_linear(ck.qweight, ck.qzeros, ck.scales, 128, "fp16", x) + b.half().double().numpy()[None, :]
    compare(run_gemm(h, x, N, gptq.PATH_LARGE_M), y_ref)
    f8 = synth.make_fp8_checkpoint(K, N, "bf16", seed=5)
    h8 = gptq.gptq_repack_fp8(f8.weight.cuda(), f8.scale_inv.cuda(), torch.bfloat16)
    assert gptq.gptq_gemm_k_splits(h8, 64) > 1
    x8 = synth.make_x(64, K, "bf16", seed=6)
    compare(run_gemm(h8, x8, N, gptq.PATH_LARGE_M), oracle.fp8_linear(f8.weight, f8.scale_inv, "bf16", x8))


def test_split_back_to_back_calls_and_graphs():
    """Many calls in a row, alternating M and captured in a CUDA graph (the next call's clusters start
    while this call's finish): every result stays right."""
    spec = synth.LayerSpec(4096, 256, 4, 128, False, False, "bf16")
    ck = synth.make_checkpoint(spec, seed=7)
    h = repack(ck)
    assert gptq.gptq_gemm_k_splits(h, 40) > 1 and gptq.gptq_gemm_k_splits(h, 128) > 1
    xs = {M: synth.make_x(M, spec.K, "bf16", seed=M).cuda() for M in (40, 128)}
    ys = {M: torch.empty(M, spec.N, dtype=torch.bfloat16, device="cuda") for M in xs}
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(3):
            for M in (40, 128):
                gptq.gptq_gemm_path(h, xs[M], ys[M], gptq.PATH_LARGE_M)
    for _ in range(4):
        g.replay()
    torch.cuda.synchronize()
    for M in (40, 128):
        compare(ys[M].cpu(), oracle_y(ck, xs[M].cpu()))
