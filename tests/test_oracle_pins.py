"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test states what it pins.  None re-types the oracle's own formulas: the
checks are printed/closed-form values, an independent bit-string decoding,
invariants, special cases that reduce to library routines, and brute force.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from weight_only_quantized_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
BITS = [2, 3, 4, 8]


def _u32(a):
    return np.asarray(a).astype(np.int64) & 0xFFFFFFFF


# ---------------------------------------------------------------- bit order
def test_bit_order_golden_words():
    """Low-bits-first packing along K: printed statement -> closed-form words (golden file)."""
    with open(os.path.join(GOLDEN, "bit_order_words.json")) as f:
        cases = json.load(f)["cases"]
    for case in cases:
        b, codes = case["bits"], case["codes"]
        pack = 32 // b
        col = np.zeros((32, 1), np.uint8)           # one 32-row K block, one column
        col[:pack, 0] = codes
        qw = oracle.pack_codes(np.tile(col, (1, 32)), b)
        assert int(_u32(qw[0, 0])) == int(case["word_hex"], 16), case
        back = oracle.unpack_codes(qw, b)
        assert np.array_equal(back[:pack, 0], np.array(codes, np.uint8))


def _bitstream_decode(words_col, bits, count):
    """Independent decoding: the column's int32 words concatenated little-endian into one
    integer; code i is bits [bits*i, bits*i + bits) of it.  For bits 2/4/8 this is the
    Reader's per-word shift; for bits 3 it is the 10 / split / 10 reading (32 codes in 96
    contiguous bits, fields straddling words at codes 10 and 21)."""
    big = 0
    for i, w in enumerate(_u32(words_col).tolist()):
        big |= int(w) << (32 * i)
    mask = (1 << bits) - 1
    return np.array([(big >> (bits * i)) & mask for i in range(count)], np.uint8)


@pytest.mark.parametrize("bits", BITS)
def test_unpack_matches_bitstream_decoding(bits):
    gen = torch.Generator().manual_seed(11)
    K, N = 96, 32
    qw = synth.random_words(gen, (K * bits // 32, N)).numpy()
    codes = oracle.unpack_codes(qw, bits)
    for n in (0, 7, 31):
        assert np.array_equal(codes[:, n], _bitstream_decode(qw[:, n], bits, K))
    # zeros pack along N with the same scheme
    G = 3
    qz = synth.random_words(gen, (G, N * bits // 32)).numpy()
    z = oracle.unpack_zeros(qz, N, bits)
    for g in range(G):
        assert np.array_equal(z[g] - 1, _bitstream_decode(qz[g], bits, N).astype(np.int32))


def test_three_bit_straddling_fields():
    """Codes 10 and 21 of a 32-code block straddle words (the 10 / split / 10 reading)."""
    codes = np.zeros((32, 32), np.uint8)
    codes[10, :] = 0b101
    codes[21, :] = 0b011
    qw = _u32(oracle.pack_codes(codes, 3))
    # code 10: bits 0-1 -> word0 bits 30-31, bit 2 -> word1 bit 0
    assert qw[0, 0] == (0b01 << 30) and qw[1, 0] & 1 == 1
    # code 21: bit 0 -> word1 bit 31, bits 1-2 -> word2 bits 0-1
    assert (qw[1, 0] >> 31) & 1 == 1 and qw[2, 0] & 3 == 0b01


# ---------------------------------------------------------------- round trips
@pytest.mark.parametrize("bits", BITS)
def test_pack_unpack_round_trip_random(bits):
    rng = np.random.default_rng(bits)
    codes = rng.integers(0, 2 ** bits, size=(128, 64), dtype=np.uint8)
    assert np.array_equal(oracle.unpack_codes(oracle.pack_codes(codes, bits), bits), codes)


@pytest.mark.parametrize("bits", BITS)
def test_pack_unpack_round_trip_exhaustive(bits):
    """Every code value at every position inside a 32-row block."""
    vals = np.arange(2 ** bits, dtype=np.uint8)
    codes = np.zeros((32, 32 * len(vals)), np.uint8)
    for i, v in enumerate(vals):
        codes[:, 32 * i:32 * (i + 1)] = v
    codes[:, ::3] = ((codes[:, ::3].astype(np.int64) + np.arange(32)[:, None]) % (2 ** bits)).astype(np.uint8)
    assert np.array_equal(oracle.unpack_codes(oracle.pack_codes(codes, bits), bits), codes)


@pytest.mark.parametrize("bits", BITS)
def test_zero_points_stored_minus_one(bits):
    """GPTQ-006: the writer stores z - 1, the reader adds 1 back, with no wrap."""
    N = 64
    z = np.tile(np.arange(1, 2 ** bits, dtype=np.int32), N)[:N][None, :]   # z in [1, 2^b - 1]
    assert np.array_equal(oracle.unpack_zeros(oracle.pack_zeros(z, bits), N, bits), z)
    # an intended zero of 0 is stored masked (all ones) and reads back as 2^b
    z0 = np.zeros((1, N), np.int32)
    back = oracle.unpack_zeros(oracle.pack_zeros(z0, bits), N, bits)
    assert np.all(back == 2 ** bits)


def test_symmetric_zero_word_reads_eight():
    """A symmetric 4-bit layer (zero 8) stores 7 in every nibble: 0x77777777."""
    qz = np.full((2, 32 * 4 // 32), 0x77777777, np.int64).astype(np.int32)
    assert np.all(oracle.unpack_zeros(qz, 32, 4) == 8)
    for b in (2, 8):
        w = synth.symmetric_zero_word(b)
        qz = np.full((1, 32 * b // 32), w, np.int64).astype(np.int32)
        assert np.all(oracle.unpack_zeros(qz, 32, b) == 2 ** (b - 1))


# ---------------------------------------------------------------- scalar decoders
def test_fp16_decoder_exhaustive():
    """All 65536 binary16 patterns agree with numpy's float16 -> float32 conversion."""
    lib = oracle.lib()
    pats = np.arange(65536, dtype=np.uint32)
    ref = pats.astype(np.uint16).view(np.float16).astype(np.float32)
    got = np.array([lib.oracle_half_to_float(int(p), 0) for p in pats], np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_bf16_decoder_exhaustive():
    lib = oracle.lib()
    pats = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    ref = pats.view(torch.bfloat16).float().numpy()
    got = np.array([lib.oracle_half_to_float(int(p) & 0xFFFF, 1) for p in pats.tolist()], np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


# ---------------------------------------------------------------- groups
def test_group_count():
    assert oracle.num_groups(4096, -1) == 1
    assert oracle.num_groups(4096, 128) == 32
    assert oracle.num_groups(4100 - 4, 96) == 43      # ceil(4096 / 96)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_group_size_minus_one_is_one_group(dtype):
    """group_size -1: one group over all of in_features, identical to g_idx == 0 everywhere."""
    spec = synth.LayerSpec(256, 64, 4, -1, dtype=dtype)
    ck = synth.make_checkpoint(spec, seed=3)
    assert ck.qzeros.shape[0] == 1 and ck.scales.shape[0] == 1
    Wa = oracle.dequant(ck.qweight, ck.qzeros, ck.scales, None, 4, -1, dtype)
    Wb = oracle.dequant(ck.qweight, ck.qzeros, ck.scales, np.zeros(256, np.int32), 4, -1, dtype)
    assert np.array_equal(Wa, Wb)


@pytest.mark.parametrize("bits", BITS)
def test_sequential_g_idx_equals_default(bits):
    spec = synth.LayerSpec(512, 64, bits, 128)
    ck = synth.make_checkpoint(spec, seed=4)
    Wa = oracle.dequant(ck.qweight, ck.qzeros, ck.scales, None, bits, 128, "fp16")
    Wb = oracle.dequant(ck.qweight, ck.qzeros, ck.scales, synth.sequential_g_idx(512, 128), bits, 128, "fp16")
    assert np.array_equal(Wa, Wb)


@pytest.mark.parametrize("bits", BITS)
def test_desc_act_checkpoint_gives_same_dense_weight(bits):
    """Act-order: a checkpoint written from the same (codes, zeros, scales) with its
    columns visited in a permuted order (ch. 39 gptq_quantize: codes[:, inverse] and
    g_idx = (arange // group_size)[inverse]) dequantises to the sequential W with its
    columns permuted back -- bit-exactly -- and gives the same y."""
    K, N, gs = 512, 64, 64
    G = K // gs
    rng = np.random.default_rng(7 + bits)
    codes_v = rng.integers(0, 2 ** bits, size=(K, N), dtype=np.uint8)   # [k in visit order, n]
    z = rng.integers(1, 2 ** bits, size=(G, N), dtype=np.int32)
    s = torch.from_numpy(rng.uniform(0.002, 0.02, size=(G, N))).to(torch.float16)
    perm = rng.permutation(K)
    inverse = np.argsort(perm)
    qz = oracle.pack_zeros(z, bits)
    seq_qw = oracle.pack_codes(codes_v, bits)
    act_qw = oracle.pack_codes(codes_v[inverse, :], bits)                # original column k = visit inverse[k]
    g_idx = (np.arange(K) // gs)[inverse].astype(np.int32)
    W_seq = oracle.dequant(seq_qw, qz, s, None, bits, gs, "fp16")
    W_act = oracle.dequant(act_qw, qz, s, g_idx, bits, gs, "fp16")
    assert np.array_equal(W_act[:, perm], W_seq)
    x = torch.randn(3, K, generator=torch.Generator().manual_seed(1)).to(torch.float16)
    y_act = oracle.linear(act_qw, qz, s, g_idx, bits, gs, "fp16", x)
    y_seq = oracle.linear(seq_qw, qz, s, None, bits, gs, "fp16", x[:, torch.from_numpy(perm)])
    assert np.allclose(y_act, y_seq, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- brute force
@pytest.mark.parametrize("bits", BITS)
@pytest.mark.parametrize("K", [32, 64])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_linear_brute_force_tiny(bits, K, dtype):
    """Tiny layers: oracle.linear against a dense float64 product built from an independent
    bit-string decoding of the checkpoint and torch's own fp16/bf16 -> float conversion."""
    N, M, gs = 32, 3, 32
    spec = synth.LayerSpec(K, N, bits, gs, desc_act=(K == 64), dtype=dtype)
    ck = synth.make_checkpoint(spec, seed=bits * 10 + K)
    x = synth.make_x(M, K, dtype, seed=5)
    qw, qz = ck.qweight.numpy(), ck.qzeros.numpy()
    q = np.stack([_bitstream_decode(qw[:, n], bits, K) for n in range(N)], axis=1).astype(np.float64)
    zz = np.stack([_bitstream_decode(qz[g], bits, N) for g in range(spec.G)]).astype(np.float64) + 1.0
    sc = ck.scales.double().numpy()
    gi = np.arange(K) // gs if ck.g_idx is None else ck.g_idx.numpy()
    W = np.empty((N, K))
    for k in range(K):
        W[:, k] = (q[k, :] - zz[gi[k], :]) * sc[gi[k], :]
    y_ref = x.double().numpy() @ W.T
    y = oracle.linear(ck.qweight, ck.qzeros, ck.scales, ck.g_idx, bits, gs, dtype, x)
    assert np.allclose(y, y_ref, rtol=1e-12, atol=1e-12)


def test_linear_sampled_rows_and_columns_match_full():
    spec = synth.LayerSpec(256, 96, 4, 128, dtype="bf16")
    ck = synth.make_checkpoint(spec, seed=9)
    x = synth.make_x(7, 256, "bf16", seed=2)
    full = oracle.linear(ck.qweight, ck.qzeros, ck.scales, None, 4, 128, "bf16", x)
    rows, cols = np.array([6, 0, 3]), np.array([95, 1, 40, 41])
    part = oracle.linear(ck.qweight, ck.qzeros, ck.scales, None, 4, 128, "bf16", x, rows, cols)
    assert np.array_equal(part, full[np.ix_(rows, cols)])


def test_one_hot_input_reads_one_weight_column():
    """x = e_k picks column k of the dense W exactly."""
    spec = synth.LayerSpec(128, 64, 4, 32, desc_act=True)
    ck = synth.make_checkpoint(spec, seed=12)
    W = oracle.dequant(ck.qweight, ck.qzeros, ck.scales, ck.g_idx, 4, 32, "fp16")
    x = torch.zeros(4, 128, dtype=torch.float16)
    ks = [0, 31, 77, 127]
    for i, k in enumerate(ks):
        x[i, k] = 1.0
    y = oracle.linear(ck.qweight, ck.qzeros, ck.scales, ck.g_idx, 4, 32, "fp16", x)
    for i, k in enumerate(ks):
        assert np.array_equal(y[i], W[:, k].astype(np.float64))


# ---------------------------------------------------------------- reject rules
def test_example_header_passes_shape_rules():
    with open(os.path.join(GOLDEN, "example_header_small_gptq.json")) as f:
        hdr = json.load(f)
    t, d = hdr["tensors"], hdr["derived"]
    qw, qz, sc = t["gptq.qweight"]["shape"], t["gptq.qzeros"]["shape"], t["gptq.scales"]["shape"]
    in_f = t["gptq.g_idx"]["shape"][0]
    assert in_f == qw[0] * 32 // d["bits"] and qw[1] == d["out_features"]
    assert qz[0] == d["groups"] == oracle.num_groups(in_f, d["group_size"])
    g_idx = (np.arange(in_f) // d["group_size"]).astype(np.int32)
    assert oracle.check_rules(d["bits"], qw, qz, sc, in_f, g_idx) == 0


@pytest.mark.parametrize("case,rule", [
    (dict(bits=5), 1),
    (dict(bits=1), 1),
    (dict(in_features=240), 2),                       # not divisible by 32
    (dict(qweight=(33, 32)), 2),
    (dict(qzeros=(8, 5)), 3),
    (dict(scales=(8, 31)), 3),
    (dict(g_idx_len=255), 4),
    (dict(g_idx_bad=8), 4),                           # selects no scale row
    (dict(g_idx_bad=-1), 4),
])
def test_reject_rules(case, rule):
    bits = case.get("bits", 4)
    in_f = case.get("in_features", 256)
    qw = case.get("qweight", (in_f // 32 * 4, 32))
    qz = case.get("qzeros", (8, 4))
    sc = case.get("scales", (8, 32))
    n = case.get("g_idx_len", in_f)
    g = (np.arange(n) // 32).astype(np.int32)
    if "g_idx_bad" in case:
        g[17] = case["g_idx_bad"]
    assert oracle.check_rules(bits, qw, qz, sc, in_f, g) == rule
