"""Pins of the oracle's format extensions: gptq_v2 zero fields, the optional bias, and the
rounding of float32 scales to the layer's dtype.

What fixes each check: numpy's and torch's own float32 -> float16 / bfloat16 conversions (round
to nearest even) over a large stride of all float32 bit patterns plus the boundary cases; the
v1/v2 relation (a v2 field holds the zero, a v1 field the zero minus one) against the pinned v1
reader; x = 0 giving exactly the bias; and a float64 matrix product.
"""
import numpy as np
import pytest
import torch

import oracle
from weight_only_quantized_gb300 import synth


def _sample_fp32_patterns():
    pats = np.arange(0, 2 ** 32, 257, dtype=np.uint64).astype(np.uint32)
    # boundaries: fp16 subnormal/normal edge, largest finite, overflow threshold, ties at every
    # binade edge of fp16 and bf16, the smallest fp32 subnormals
    edges = []
    for base in (0x33000000, 0x387FC000, 0x38800000, 0x477FE000, 0x477FEFFF, 0x477FF000, 0x7F7F8000,
                 0x7F7FFFFF, 0x3F808000, 0x3F818000, 0x3F801000, 0x3F803000, 0x00000001, 0x007FFFFF):
        edges.extend(range(base - 3, base + 4))
    e = np.array(edges, np.int64) & 0x7FFFFFFF
    e = np.concatenate([e, e | 0x80000000]).astype(np.uint32)
    return np.concatenate([pats, e])


def test_round_fp32_to_fp16_matches_numpy():
    u = _sample_fp32_patterns()
    v = u.view(np.float32)
    with np.errstate(over="ignore", invalid="ignore"):
        ref = v.astype(np.float16).view(np.uint16)
    got = oracle.round_fp32(v, "fp16")
    nan = np.isnan(v)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.all((got[nan] & 0x7C00) == 0x7C00) and np.all((got[nan] & 0x3FF) != 0)


def test_round_fp32_to_bf16_matches_torch():
    u = _sample_fp32_patterns()
    v = u.view(np.float32)
    ref = torch.from_numpy(v.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.round_fp32(v, "bf16")
    nan = np.isnan(v)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.all((got[nan] & 0x7F80) == 0x7F80) and np.all((got[nan] & 0x7F) != 0)


@pytest.mark.parametrize("bits", [2, 3, 4, 8])
def test_v2_fields_hold_the_zero(bits):
    """A v2 field f reads as zero f; the v1 field of the same zero is f - 1 (zeros 1 .. 2^bits - 1)."""
    K, N, gs = 128, 64, 32
    spec = synth.LayerSpec(K, N, bits, gs, dtype="bf16")
    ck = synth.make_checkpoint(spec, seed=bits)
    gen = torch.Generator().manual_seed(bits + 1)
    z = torch.randint(1, 2 ** bits, (spec.G, N), generator=gen, dtype=torch.int32).numpy()
    qz_v1 = oracle.pack_zeros(z, bits)            # fields z - 1
    qz_v2 = oracle.pack_zeros(z + 1, bits)        # fields z
    W1 = oracle.dequant(ck.qweight, qz_v1, ck.scales, None, bits, gs, "bf16")
    W2 = oracle.dequant(ck.qweight, qz_v2, ck.scales, None, bits, gs, "bf16", zero_offset=0)
    assert np.array_equal(W1, W2)
    x = synth.make_x(3, K, "bf16", seed=2)
    y1 = oracle.linear(ck.qweight, qz_v1, ck.scales, None, bits, gs, "bf16", x)
    y2 = oracle.linear(ck.qweight, qz_v2, ck.scales, None, bits, gs, "bf16", x, zero_offset=0)
    assert np.array_equal(y1, y2)


def test_v2_code_equal_to_field_is_zero_weight():
    K, N, gs, bits = 64, 32, 32, 4
    gen = torch.Generator().manual_seed(9)
    f = torch.randint(0, 16, (K // gs, N), generator=gen, dtype=torch.int32).numpy()
    codes = np.repeat(f, gs, axis=0).astype(np.uint8)
    qw = oracle.pack_codes(codes, bits)
    qz = oracle.pack_zeros(f + 1, bits)           # v2 fields = f (pack_zeros stores its argument minus one)
    sc = synth.make_checkpoint(synth.LayerSpec(K, N, bits, gs), seed=1).scales
    assert np.array_equal(oracle.dequant(qw, qz, sc, None, bits, gs, "fp16", zero_offset=0), np.zeros((N, K), np.float32))


@pytest.mark.parametrize("kind", [torch.float16, torch.bfloat16, torch.float32])
def test_bias_alone_when_x_is_zero(kind):
    K, N = 128, 64
    ck = synth.make_checkpoint(synth.LayerSpec(K, N, 4, 32, dtype="fp16"), seed=3)
    b = (torch.randn(N, generator=torch.Generator().manual_seed(4)) * 3).to(kind)
    x = torch.zeros(2, K, dtype=torch.float16)
    y = oracle.linear(ck.qweight, ck.qzeros, ck.scales, None, 4, 32, "fp16", x, bias=b)
    assert np.array_equal(y, np.tile(b.double().numpy(), (2, 1)))


def test_bias_adds_to_the_product():
    K, N, M = 256, 96, 5
    ck = synth.make_checkpoint(synth.LayerSpec(K, N, 4, 128, True, dtype="bf16"), seed=5)
    x = synth.make_x(M, K, "bf16", seed=6)
    b = torch.randn(N, generator=torch.Generator().manual_seed(7)).to(torch.bfloat16)
    W = oracle.dequant(ck.qweight, ck.qzeros, ck.scales, ck.g_idx, 4, 128, "bf16").astype(np.float64)
    ref = x.double().numpy() @ W.T + b.double().numpy()[None, :]
    y = oracle.linear(ck.qweight, ck.qzeros, ck.scales, ck.g_idx, 4, 128, "bf16", x, bias=b)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)
    cols = np.array([95, 0, 40])
    ys = oracle.linear(ck.qweight, ck.qzeros, ck.scales, ck.g_idx, 4, 128, "bf16", x, cols=cols, bias=b)
    assert np.array_equal(ys, y[:, cols])
