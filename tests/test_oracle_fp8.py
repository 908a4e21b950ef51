"""Pins of the oracle's FP8 block-scaled reader ([P4] ch. 39, section "FP8 checkpoints").

What fixes each check: torch's own float8_e4m3fn type (all 256 codes), the page's statement that
448 is the largest E4M3 value, block invariants of the 128 x 128 scales (a factor reaches only its
own block; scale 1 reads the bare codes), the float64 product, and a decode-back of the runtime
layout (reading each byte out of it, the inverse of how the layout function writes them).
"""
import numpy as np
import pytest
import torch

import oracle
from weight_only_quantized_gb300 import synth


def test_e4m3_decoder_matches_torch_on_all_codes():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).float().numpy()
    got = oracle.e4m3_to_float(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2          # 0x7F and 0xFF
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))   # -0 at 0x80


def test_largest_e4m3_value_is_448():
    v = oracle.e4m3_to_float(np.arange(256, dtype=np.uint8))
    assert np.nanmax(v) == 448.0 and v[0x7E] == 448.0 and v[0xFE] == -448.0
    assert v[0x01] == 2.0 ** -9 and v[0x08] == 2.0 ** -6                  # smallest subnormal, normal


def test_scale_one_reads_the_bare_codes():
    ck = synth.make_fp8_checkpoint(256, 160, seed=1)
    W = oracle.fp8_dequant(ck.weight, np.ones_like(ck.scale_inv.numpy()))
    assert np.array_equal(W, oracle.e4m3_to_float(ck.weight))


def test_each_factor_reaches_only_its_block():
    K, N = 384, 288                                        # ragged blocks on both axes
    ck = synth.make_fp8_checkpoint(K, N, seed=2)
    base = oracle.fp8_dequant(ck.weight, ck.scale_inv)
    for bi, bj in ((0, 0), (2, 1), (1, 2)):
        s = ck.scale_inv.clone()
        s[bi, bj] *= 2.0
        W = oracle.fp8_dequant(ck.weight, s)
        changed = W != base
        rows, cols = np.nonzero(changed)
        assert rows.min() >= 128 * bi and rows.max() < min(N, 128 * (bi + 1))
        assert cols.min() >= 128 * bj and cols.max() < min(K, 128 * (bj + 1))
        blk = (slice(128 * bi, min(N, 128 * (bi + 1))), slice(128 * bj, min(K, 128 * (bj + 1))))
        assert np.array_equal(W[blk], base[blk] * 2.0)       # a power of two: exact


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_fp8_linear_is_x_times_dense_weight(dtype):
    K, N, M = 256, 96, 4
    ck = synth.make_fp8_checkpoint(K, N, dtype, seed=3)
    x = synth.make_x(M, K, dtype, seed=4)
    W = oracle.fp8_dequant(ck.weight, ck.scale_inv).astype(np.float64)
    y = oracle.fp8_linear(ck.weight, ck.scale_inv, dtype, x)
    assert np.allclose(y, x.double().numpy() @ W.T, rtol=1e-12, atol=1e-12)
    rows, cols = np.array([3, 1]), np.array([95, 0, 64])
    assert np.array_equal(oracle.fp8_linear(ck.weight, ck.scale_inv, dtype, x, rows, cols), y[np.ix_(rows, cols)])


def test_synthetic_weights_hold_no_nan_and_every_number():
    ck = synth.make_fp8_checkpoint(1024, 512, seed=5)
    seen = np.unique(ck.weight.numpy())
    assert 0x7F not in seen and 0xFF not in seen and len(seen) == 254


@pytest.mark.parametrize("K,N", [(256, 256), (320, 96), (512, 288)])
def test_fp8_layout_decodes_back(K, N):
    """Every byte read out of the layout (pair p of lane word p // 2 in its 16-bit half p % 2, the
    even k in the low byte) lands at weight[n, perm[j]]; pad rows and columns hold 0."""
    ck = synth.make_fp8_checkpoint(K, N, seed=K + N)
    L = oracle.runtime_layout_fp8(ck.weight)
    Kr, Np = L["Kr"], L["Np"]
    assert Kr % 128 == 0 and Np % 256 == 0
    perm = L["perm"]
    assert np.array_equal(perm[perm >= 0], np.arange(K))              # sequential groups: k order kept
    assert np.all(L["cgid"][:(K + 31) // 32] == np.arange((K + 31) // 32) * 32 // 128)
    words = L["wr"].view(np.uint32)
    j = np.arange(Kr)
    B, r = j // 128, j % 128
    c, t, e = r // 32, (r % 32) // 8, r % 8
    p, h = 4 * c + e // 2, e % 2
    q = 8 * t + p // 2
    V = q // 4
    n = np.arange(Np)[None, :]
    pos = n // 32 * 32 + (n % 32 + (2 * (V // 2))[:, None]) % 32
    idx = ((B * 8 + V)[:, None] * Np + pos) * 4 + (q % 4)[:, None]
    got = (words[idx] >> (16 * (p % 2) + 8 * h)[:, None]) & 0xFF
    w = ck.weight.numpy().astype(np.int64)
    ref = np.zeros((Kr, Np), np.int64)
    real = perm >= 0
    ref[np.ix_(real, np.arange(N))] = w[:, perm[real]].T
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_fp8_linear_matches_a_product_built_from_torch_float8(dtype):
    """The whole FP8 path against one built only from torch: float8_e4m3fn decoding of the bytes,
    the 128 x 128 factors expanded by repeat_interleave, float32 products, a float64 matmul."""
    K, N, M = 384, 160, 3
    ck = synth.make_fp8_checkpoint(K, N, dtype, seed=21)
    x = synth.make_x(M, K, dtype, seed=22)
    w = ck.weight.view(torch.float8_e4m3fn).float()
    s = ck.scale_inv.repeat_interleave(128, 0)[:N].repeat_interleave(128, 1)[:, :K]
    W = (w * s).double()                                      # float32 products, as dequantize_blocks
    ref = (x.double() @ W.T).numpy()
    y = oracle.fp8_linear(ck.weight, ck.scale_inv, dtype, x)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)
