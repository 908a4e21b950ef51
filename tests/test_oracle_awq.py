"""Pins of the oracle's AutoAWQ GEMM reader (4-bit, codes packed along the output dimension).

What fixes each check: the printed interleaved order and the bits-16-19 statement (golden
words), the inverse relation of packing and unpacking, the special cases code == zero and
code == zero + 1, agreement with the already-pinned GPTQ reader on the same integers (an AWQ
zero z equals a GPTQ zero field z - 1), and a float64 matrix product.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from weight_only_quantized_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _u32(a):
    return np.asarray(a).astype(np.int64) & 0xFFFFFFFF


def test_awq_order_golden_words():
    """Each output column's nibble position, one-hot, plus the ascending-codes word."""
    with open(os.path.join(GOLDEN, "awq_order_words.json")) as f:
        cases = json.load(f)["cases"]
    for case in cases:
        codes = np.array([case["codes"] * 4], np.uint8)          # one row, 32 outputs
        w = oracle.awq_pack(codes)
        assert w.shape == (1, 4)
        assert all(int(_u32(v)) == int(case["word_hex"], 16) for v in w[0]), case
        assert np.array_equal(oracle.awq_unpack(w), codes)


def test_output_one_sits_in_bits_16_to_19():
    codes = np.zeros((1, 8), np.uint8)
    for v in range(16):
        codes[0, 1] = v
        assert (int(_u32(oracle.awq_pack(codes)[0, 0])) >> 16) & 0xF == v
        assert int(_u32(oracle.awq_pack(codes)[0, 0])) & ~(0xF << 16) & 0xFFFFFFFF == 0


def test_awq_pack_unpack_round_trip():
    gen = torch.Generator().manual_seed(3)
    words = synth.random_words(gen, (64, 12)).numpy()
    assert np.array_equal(oracle.awq_pack(oracle.awq_unpack(words)), words)
    codes = torch.randint(0, 16, (40, 96), generator=gen, dtype=torch.uint8).numpy()
    assert np.array_equal(oracle.awq_unpack(oracle.awq_pack(codes)), codes)


def _awq_from_integers(codes, zeros, scales):
    """AWQ tensors for given integer codes [K, N], zeros [G, N] and scales [G, N]."""
    return oracle.awq_pack(codes), oracle.awq_pack(zeros), scales


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_code_equal_zero_gives_zero_weight(dtype):
    K, N, gs = 64, 32, 32
    gen = torch.Generator().manual_seed(4)
    zeros = torch.randint(0, 16, (K // gs, N), generator=gen, dtype=torch.uint8).numpy()
    codes = np.repeat(zeros, gs, axis=0)
    sc = synth.make_awq_checkpoint(K, N, gs, dtype, seed=4).scales
    qw, qz, sc = _awq_from_integers(codes, zeros, sc)
    assert np.array_equal(oracle.awq_dequant(qw, qz, sc, gs, dtype), np.zeros((N, K), np.float32))


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_code_one_above_zero_reads_the_scale(dtype):
    """No +1 on the AWQ zero: code z + 1 dequantises to exactly scale (code z to 0 above)."""
    K, N, gs = 64, 32, 16
    gen = torch.Generator().manual_seed(5)
    zeros = torch.randint(0, 15, (K // gs, N), generator=gen, dtype=torch.uint8).numpy()
    codes = np.repeat(zeros, gs, axis=0) + 1
    sc = synth.make_awq_checkpoint(K, N, gs, dtype, seed=5).scales
    qw, qz, _ = _awq_from_integers(codes, zeros, sc)
    W = oracle.awq_dequant(qw, qz, sc, gs, dtype)
    s = sc.float().numpy()                                       # [G, N]
    assert np.array_equal(W, np.repeat(s, gs, axis=0).T)


@pytest.mark.parametrize("gs", [32, 128, -1])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_awq_dequant_equals_gptq_reader_on_same_integers(gs, dtype):
    """Zeros drawn in 1..15 so that the GPTQ zero field (stored minus one) can hold them."""
    K, N = 256, 64
    ck = synth.make_awq_checkpoint(K, N, gs, dtype, seed=6)
    gen = torch.Generator().manual_seed(7)
    zeros = torch.randint(1, 16, (ck.G, N), generator=gen, dtype=torch.uint8).numpy()
    codes = oracle.awq_unpack(ck.qweight)
    qw, qz, sc = _awq_from_integers(codes, zeros, ck.scales)
    W_awq = oracle.awq_dequant(qw, qz, sc, gs, dtype)
    W_gptq = oracle.dequant(oracle.pack_codes(codes, 4), oracle.pack_zeros(zeros.astype(np.int32), 4),
                            sc, None, 4, gs, dtype)
    assert np.array_equal(W_awq, W_gptq)


def test_gptq_field_conversion_keeps_codes_and_raw_zeros():
    ck = synth.make_awq_checkpoint(128, 64, 32, "fp16", seed=8)
    qwg, qzg = oracle.awq_to_gptq_fields(ck.qweight, ck.qzeros, 32)
    assert np.array_equal(oracle.unpack_codes(qwg, 4), oracle.awq_unpack(ck.qweight))
    # unpack_zeros adds GPTQ's +1 to the raw field; the raw field is the AWQ zero itself.
    assert np.array_equal(oracle.unpack_zeros(qzg, 64, 4) - 1, oracle.awq_unpack(ck.qzeros).astype(np.int32))


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_awq_linear_is_x_times_dense_weight(dtype):
    K, N, M, gs = 128, 64, 5, 32
    ck = synth.make_awq_checkpoint(K, N, gs, dtype, seed=9)
    x = synth.make_x(M, K, dtype, seed=10)
    W = oracle.awq_dequant(ck.qweight, ck.qzeros, ck.scales, gs, dtype).astype(np.float64)
    y_ref = x.double().numpy() @ W.T
    y = oracle.awq_linear(ck.qweight, ck.qzeros, ck.scales, gs, dtype, x)
    assert np.allclose(y, y_ref, rtol=1e-12, atol=1e-12)
    rows, cols = np.array([4, 0]), np.array([63, 2, 17])
    part = oracle.awq_linear(ck.qweight, ck.qzeros, ck.scales, gs, dtype, x, rows, cols)
    assert np.array_equal(part, y[np.ix_(rows, cols)])


def test_awq_rejects_bad_shapes():
    w = np.zeros((32, 3), np.int32)                              # N = 24 is not a multiple of 32
    with pytest.raises(Exception):
        oracle.awq_dequant(w, np.zeros((1, 3), np.int32), np.zeros((1, 24), np.float16), -1, "fp16")
