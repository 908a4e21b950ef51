"""Seeded synthetic checkpoints and activations shaped like the workloads of the GPTQ pages.

This module draws random numbers and nothing else: it holds none of the method's
arithmetic (no packing, unpacking or dequantisation).  Both the CUDA path and the
CPU oracle consume what it produces.

Why random int32 words are valid checkpoint tensors: in the AutoGPTQ "cuda" pack
(tensref.org, "GPTQ packed checkpoint", section GptqLayer) every bit of a qweight
or qzeros word belongs to exactly one code, for bits 2, 4 and 8 and also for 3
(32 codes fill exactly 3 words).  Independent uniform words therefore carry
independent codes uniform over [0, 2^bits - 1], which is the codes distribution
the workloads ask for.  The asymmetric zero points are "uniform over [0,
2^bits-1]" and are stored minus one (masked), which is again a uniform field, so
uniform words serve for qzeros as well.  A symmetric zero of 2^(bits-1) is stored
as 2^(bits-1) - 1 in every field; ``symmetric_zero_word`` gives that constant
word pattern for bits 2, 4 and 8 (the pattern repeats every byte or nibble).

Draw order per layer is fixed: qweight words, qzeros words, scales, desc_act
permutation, x.  Everything is drawn on the CPU with torch.Generator.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

_DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16}


@dataclasses.dataclass
class LayerSpec:
    """One GPTQ linear layer: in_features K, out_features N and its quantize_config."""
    K: int
    N: int
    bits: int = 4
    group_size: int = 128
    desc_act: bool = False
    sym: bool = False
    dtype: str = "fp16"          # dtype of scales, x and y
    scale_lo: float = 0.002
    scale_hi: float = 0.01

    @property
    def G(self) -> int:
        return 1 if self.group_size == -1 else -(-self.K // self.group_size)


@dataclasses.dataclass
class Checkpoint:
    spec: LayerSpec
    qweight: torch.Tensor        # int32 [K*bits/32, N]
    qzeros: torch.Tensor         # int32 [G, N*bits/32]
    scales: torch.Tensor         # fp16/bf16 [G, N]
    g_idx: Optional[torch.Tensor]  # int32 [K], None for sequential k // group_size


def symmetric_zero_word(bits: int) -> int:
    """int32 word whose every field holds 2^(bits-1) - 1 (zero 2^(bits-1) stored minus one)."""
    if bits == 2:
        return 0x55555555          # field value 1 in every 2-bit slot
    if bits == 4:
        return 0x77777777          # field value 7 in every nibble
    if bits == 8:
        return 0x7F7F7F7F          # field value 127 in every byte
    raise ValueError("symmetric zero words are generated for bits 2, 4 and 8")


def _as_int32(u: torch.Tensor) -> torch.Tensor:
    """int64 holding 32-bit patterns -> int32 with the same bits."""
    return torch.where(u >= 2 ** 31, u - 2 ** 32, u).to(torch.int32)


def random_words(gen: torch.Generator, shape) -> torch.Tensor:
    return _as_int32(torch.randint(0, 2 ** 32, shape, generator=gen, dtype=torch.int64))


def make_checkpoint(spec: LayerSpec, seed: int = 0) -> Checkpoint:
    gen = torch.Generator().manual_seed(seed)
    K, N, b, G = spec.K, spec.N, spec.bits, spec.G
    qweight = random_words(gen, (K * b // 32, N))
    if spec.sym:
        qzeros = torch.full((G, N * b // 32), symmetric_zero_word(b), dtype=torch.int64)
        qzeros = _as_int32(qzeros)
    else:
        qzeros = random_words(gen, (G, N * b // 32))
    scales = (torch.rand((G, N), generator=gen, dtype=torch.float64) * (spec.scale_hi - spec.scale_lo)
              + spec.scale_lo).to(_DTYPES[spec.dtype])
    g_idx = None
    if spec.desc_act:
        gs = K if spec.group_size == -1 else spec.group_size
        order = torch.randperm(K, generator=gen)
        g_idx = (torch.arange(K) // gs)[order].to(torch.int32)
    return Checkpoint(spec, qweight, qzeros, scales, g_idx)


@dataclasses.dataclass
class AwqCheckpoint:
    """An AutoAWQ GEMM layer (4-bit, codes packed eight to a word along the output dimension)."""
    K: int
    N: int
    group_size: int
    dtype: str                   # dtype of scales, x and y (the format ships fp16 scales)
    qweight: torch.Tensor        # int32 [K, N/8]
    qzeros: torch.Tensor         # int32 [G, N/8]
    scales: torch.Tensor         # fp16/bf16 [G, N]

    @property
    def G(self) -> int:
        return 1 if self.group_size == -1 else -(-self.K // self.group_size)


def make_awq_checkpoint(K: int, N: int, group_size: int = 128, dtype: str = "fp16", seed: int = 0,
                        scale_lo: float = 0.002, scale_hi: float = 0.01) -> AwqCheckpoint:
    """Uniform random words again carry uniform independent 4-bit codes and zeros: in the AWQ
    packing every nibble of a qweight or qzeros word is one field (only their order along the
    output dimension differs from GPTQ).  Draw order: qweight words, qzeros words, scales."""
    gen = torch.Generator().manual_seed(seed)
    G = 1 if group_size == -1 else -(-K // group_size)
    qweight = random_words(gen, (K, N // 8))
    qzeros = random_words(gen, (G, N // 8))
    scales = (torch.rand((G, N), generator=gen, dtype=torch.float64) * (scale_hi - scale_lo)
              + scale_lo).to(_DTYPES[dtype])
    return AwqCheckpoint(K, N, group_size, dtype, qweight, qzeros, scales)


@dataclasses.dataclass
class Fp8Checkpoint:
    """An FP8 block-scaled layer: float8_e4m3fn weight [N, K] (held as its bytes) and one float32
    factor per 128 x 128 block."""
    K: int
    N: int
    dtype: str                   # dtype of x and y
    weight: torch.Tensor         # uint8 [N, K], e4m3 bit patterns
    scale_inv: torch.Tensor      # float32 [ceil(N/128), ceil(K/128)]


def make_fp8_checkpoint(K: int, N: int, dtype: str = "bf16", seed: int = 0, scale_lo: float = 1e-4,
                        scale_hi: float = 1e-3) -> Fp8Checkpoint:
    """Weight bytes uniform over the 254 e4m3 codes that are numbers (0x7F and 0xFF, the NaNs,
    left out): every magnitude from the subnormals to 448 occurs, both signs.  Draw order:
    weight bytes, scales."""
    gen = torch.Generator().manual_seed(seed)
    b = torch.randint(0, 254, (N, K), generator=gen, dtype=torch.int32)
    b = b + (b >= 0x7F).to(torch.int32)                  # skip 0x7F; 0xFF is never reached
    scale_inv = (torch.rand((-(-N // 128), -(-K // 128)), generator=gen, dtype=torch.float64)
                 * (scale_hi - scale_lo) + scale_lo).float()
    return Fp8Checkpoint(K, N, dtype, b.to(torch.uint8), scale_inv)


def make_x(M: int, K: int, dtype: str, seed: int = 1) -> torch.Tensor:
    gen = torch.Generator().manual_seed(seed)
    return torch.randn((M, K), generator=gen, dtype=torch.float32).to(_DTYPES[dtype])


def sequential_g_idx(K: int, group_size: int) -> torch.Tensor:
    """g_idx of a checkpoint without act-order: input feature k belongs to group k // group_size."""
    gs = K if group_size == -1 else group_size
    return (torch.arange(K) // gs).to(torch.int32)


# The five workloads, named by what they are.
def workload(name: str) -> tuple[LayerSpec, list[int]]:
    """Layer shape and the batch sizes M that each named workload is run at."""
    if name == "tiny-256x256-b4g128":
        return LayerSpec(256, 256, 4, 128, False, False, "fp16", 0.005, 0.02), [4]
    if name == "llama3-8b-decode-4096x14336-b4g128-sym":
        return LayerSpec(4096, 14336, 4, 128, False, True, "bf16", 0.002, 0.01), [1, 8, 16]
    if name == "llama3-70b-gate-8192x28672-b4g128-descact":
        return LayerSpec(8192, 28672, 4, 128, True, False, "fp16", 0.002, 0.01), [1, 4, 16, 64]
    if name == "prefill-8192x28672-b4g128":
        return LayerSpec(8192, 28672, 4, 128, False, False, "bf16", 0.002, 0.01), [512, 2048, 4096]
    raise KeyError(name)


def format_sweep() -> list[LayerSpec]:
    """K = N = 4096 sweep: bits 2/3/8 at group 128 and bits 4 at groups -1/32/64.

    desc_act is on for half the cases (b3-g128, b8-g128, b4-g32); never for group
    -1, whose single group makes the permutation a no-op.
    """
    mk = lambda b, gs, da: LayerSpec(4096, 4096, b, gs, da, False, "fp16", 0.002, 0.02)
    return [mk(2, 128, False), mk(3, 128, True), mk(8, 128, True),
            mk(4, -1, False), mk(4, 32, True), mk(4, 64, False)]


SWEEP_M = [1, 32, 256]
