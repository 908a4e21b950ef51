"""GPU parity of the large-M (tcgen05 / TMEM / TMA) kernel against the CPU oracle.

The path is forced with gptq_gemm_path so it is checked at small M too.  Shapes cover every bit
width, both dtypes, act-order (x gathered into the workspace), padded K, ragged N and M tails
that leave part of an x tile (64, 128 or 256 rows, chosen by M) empty.
"""
import numpy as np
import pytest
import torch

import oracle
from weight_only_quantized_gb300 import gptq, synth

from gpu_util import compare, oracle_y, repack, run_gemm

pytestmark = pytest.mark.gpu

SPECS = [
    synth.LayerSpec(256, 256, 4, 128, False, False, "bf16"),
    synth.LayerSpec(512, 512, 4, 128, False, False, "fp16"),
    synth.LayerSpec(512, 288, 4, 128, True, False, "bf16"),        # act-order, ragged N tile
    synth.LayerSpec(320, 256, 2, 64, False, False, "fp16"),        # K padded to 384
    synth.LayerSpec(384, 320, 3, 128, True, False, "bf16"),
    synth.LayerSpec(384, 256, 3, 128, False, False, "fp16"),
    synth.LayerSpec(256, 256, 8, 32, True, False, "bf16"),
    synth.LayerSpec(256, 512, 8, 64, False, False, "fp16"),
    synth.LayerSpec(1024, 256, 4, -1, False, True, "bf16"),
    synth.LayerSpec(1024, 512, 4, 96, False, False, "fp16"),       # groups of 96, padded
]


def _id(s):
    return f"K{s.K}N{s.N}b{s.bits}g{s.group_size}{'da' if s.desc_act else ''}{s.dtype}"


@pytest.mark.parametrize("spec", SPECS, ids=_id)
@pytest.mark.parametrize("M", [1, 17, 64, 65, 128, 129, 200, 300])
def test_large_path_parity(spec, M):
    ck = synth.make_checkpoint(spec, seed=spec.K + spec.N + spec.bits)
    h = repack(ck)
    gptq.gptq_reserve(h, 300)
    x = synth.make_x(M, spec.K, spec.dtype, seed=M + 7)
    compare(run_gemm(h, x, spec.N, gptq.PATH_LARGE_M), oracle_y(ck, x))
    gptq.gptq_device_status(h)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_large_path_one_hot_exact(dtype):
    """x = e_k on the tcgen05 path gives round(W[n, k]) exactly: the weight is rounded once when it
    is dequantised and the single non-zero product is exact in fp32."""
    spec = synth.LayerSpec(512, 256, 4, 64, True, False, dtype)
    ck = synth.make_checkpoint(spec, seed=33)
    h = repack(ck)
    gptq.gptq_reserve(h, 256)
    W = oracle.dequant(ck.qweight, ck.qzeros, ck.scales, ck.g_idx, 4, 64, dtype)
    ks = list(range(0, 512, 37))
    tdt = torch.float16 if dtype == "fp16" else torch.bfloat16
    x = torch.zeros(len(ks), spec.K, dtype=tdt)
    for i, k in enumerate(ks):
        x[i, k] = 1.0
    y = run_gemm(h, x, spec.N, gptq.PATH_LARGE_M).float().numpy()
    for i, k in enumerate(ks):
        assert np.array_equal(y[i], torch.from_numpy(W[:, k]).to(tdt).float().numpy()), k


def test_launch_counts_per_path():
    spec = synth.LayerSpec(256, 256, 4, 128)
    h = repack(synth.make_checkpoint(spec))
    assert gptq.gptq_gemm_launches(h, 16) == 1
    assert gptq.gptq_gemm_launches(h, 28) == 1          # small-M kernel, four m-tiles
    assert gptq.gptq_gemm_launches(h, 29) == 1          # tcgen05 kernel
    assert gptq.gptq_gemm_launches(h, 17, gptq.PATH_LARGE_M) == 1
    spec = synth.LayerSpec(256, 256, 4, 128, True)
    h = repack(synth.make_checkpoint(spec))
    assert gptq.gptq_gemm_launches(h, 64) == 2          # gather pre-pass + tcgen05 kernel
    assert gptq.gptq_gemm_launches(h, 1) == 1           # small-M kernel gathers x itself at M <= 2
    assert gptq.gptq_gemm_launches(h, 5) == 2           # pre-pass above that
