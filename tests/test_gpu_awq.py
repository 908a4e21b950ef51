"""GPU parity of the AutoAWQ GEMM ingest: gptq_repack_awq through the C ABI against the oracle.

The runtime layout is compared bit for bit with the oracle's runtime layout of the same codes
and zero fields in GPTQ packing (the zero field carries the AWQ zero itself, read with offset
0); GEMM results element by element, max|y - y_ref| <= 4e-3 max|y_ref|, against the oracle's
AWQ reader, on both kernel families.
"""
import numpy as np
import pytest
import torch

import oracle
from weight_only_quantized_gb300 import gptq, synth

from gpu_util import compare

pytestmark = pytest.mark.gpu

# (K, N, group_size, dtype): tiny, ragged N tile, one group, groups of 32, K not a multiple of 128
CASES = [(256, 256, 128, "fp16"), (512, 288, 128, "fp16"), (1024, 512, -1, "bf16"),
         (256, 320, 32, "fp16"), (320, 96, 64, "bf16")]


def _id(c):
    return f"K{c[0]}N{c[1]}g{c[2]}{c[3]}"


def _repack(ck: synth.AwqCheckpoint) -> gptq.Handle:
    h = gptq.gptq_repack_awq(ck.qweight.cuda(), ck.qzeros.cuda(), ck.scales.cuda(), ck.group_size)
    torch.cuda.synchronize()
    return h


def _run(h, x_cpu, N, path):
    x = x_cpu.cuda()
    y = torch.full((x.shape[0], N), float("nan"), dtype=x.dtype, device="cuda")
    gptq.gptq_gemm_path(h, x, y, path)
    torch.cuda.synchronize()
    return y.cpu()


def _oracle(ck, x, rows=None, cols=None):
    return oracle.awq_linear(ck.qweight, ck.qzeros, ck.scales, ck.group_size, ck.dtype, x, rows, cols)


@pytest.mark.parametrize("case", CASES, ids=_id)
def test_awq_repack_bit_exact(case):
    K, N, gs, dt = case
    ck = synth.make_awq_checkpoint(K, N, gs, dt, seed=K + N)
    h = _repack(ck)
    got = gptq.gptq_copy_runtime(h)
    qwg, qzg = oracle.awq_to_gptq_fields(ck.qweight, ck.qzeros, gs)
    ref = oracle.runtime_layout(qwg, qzg, ck.scales, None, 4, gs)
    for key in ("Kr", "Np", "G"):
        assert got[key] == ref[key], key
    for key in ("perm", "cgid", "s_r", "z_r", "wr"):
        assert np.array_equal(got[key], ref[key]), key
    info = gptq.gptq_get_info(h)
    assert info.zero_offset == 0 and info.bits == 4
    assert info.identity == int(np.array_equal(ref["perm"], np.arange(ref["Kr"])) and ref["Kr"] == K)


@pytest.mark.parametrize("case", CASES, ids=_id)
@pytest.mark.parametrize("M", [1, 3, 8, 17, 32])
def test_awq_gemm_parity_small_path(case, M):
    K, N, gs, dt = case
    ck = synth.make_awq_checkpoint(K, N, gs, dt, seed=N + 1)
    h = _repack(ck)
    gptq.gptq_reserve(h, 64)
    x = synth.make_x(M, K, dt, seed=M)
    compare(_run(h, x, N, gptq.PATH_SMALL_M), _oracle(ck, x))


@pytest.mark.parametrize("case", CASES, ids=_id)
@pytest.mark.parametrize("M", [1, 40, 129])
def test_awq_gemm_parity_large_path(case, M):
    K, N, gs, dt = case
    ck = synth.make_awq_checkpoint(K, N, gs, dt, seed=N + 2)
    h = _repack(ck)
    gptq.gptq_reserve(h, 160)
    x = synth.make_x(M, K, dt, seed=M + 7)
    compare(_run(h, x, N, gptq.PATH_LARGE_M), _oracle(ck, x))


@pytest.mark.parametrize("path", [gptq.PATH_SMALL_M, gptq.PATH_LARGE_M])
def test_awq_extreme_zeros(path):
    """Zero 0 with code 15 and zero 15 with code 0: the largest |code - zero| of either sign, and the
    zero fields at both ends of the nibble (no +1 and no wrap)."""
    K, N, gs = 256, 256, 64
    G = K // gs
    codes = np.zeros((K, N), np.uint8)
    zeros = np.zeros((G, N), np.uint8)
    codes[:, 0::2] = 15
    zeros[:, 1::2] = 15
    sc = synth.make_awq_checkpoint(K, N, gs, "fp16", seed=3).scales
    ck = synth.AwqCheckpoint(K, N, gs, "fp16", torch.from_numpy(oracle.awq_pack(codes)),
                             torch.from_numpy(oracle.awq_pack(zeros)), sc)
    h = _repack(ck)
    x = synth.make_x(4, K, "fp16", seed=5)
    compare(_run(h, x, N, path), _oracle(ck, x))


def test_awq_matches_the_gptq_handle_of_the_same_weights():
    """Zeros in 1..15 re-expressed as GPTQ fields (stored minus one): both handles read the same W,
    so the two GEMMs agree to the last bit on every path."""
    K, N, gs = 512, 256, 128
    ck = synth.make_awq_checkpoint(K, N, gs, "bf16", seed=11)
    gen = torch.Generator().manual_seed(12)
    zeros = torch.randint(1, 16, (ck.G, N), generator=gen, dtype=torch.uint8).numpy()
    ck.qzeros = torch.from_numpy(oracle.awq_pack(zeros))
    codes = oracle.awq_unpack(ck.qweight)
    h_awq = _repack(ck)
    qw = torch.from_numpy(oracle.pack_codes(codes, 4)).cuda()
    qz = torch.from_numpy(oracle.pack_zeros(zeros.astype(np.int32), 4)).cuda()
    h_gptq = gptq.gptq_repack(qw, qz, ck.scales.cuda(), None, 4, gs)
    for M, path in ((2, gptq.PATH_SMALL_M), (24, gptq.PATH_SMALL_M), (96, gptq.PATH_LARGE_M)):
        x = synth.make_x(M, K, "bf16", seed=M)
        assert torch.equal(_run(h_awq, x, N, path), _run(h_gptq, x, N, path))


@pytest.mark.parametrize("M", [1, 16, 256])
def test_awq_full_size_decode_layer_sampled(M):
    """A 4096 x 14336 group-128 fp16 AWQ layer (the 8B MLP shape) through gptq_gemm, compared on
    sampled rows and columns with the oracle."""
    K, N = 4096, 14336
    ck = synth.make_awq_checkpoint(K, N, 128, "fp16", seed=21)
    h = _repack(ck)
    gptq.gptq_reserve(h, M)
    x = synth.make_x(M, K, "fp16", seed=22)
    y = _run(h, x, N, gptq.PATH_AUTO)
    rows = np.unique(np.linspace(0, M - 1, min(M, 4)).astype(np.int32))
    cols = np.random.default_rng(0).choice(N, 512, replace=False).astype(np.int32)
    compare(y[rows][:, cols], _oracle(ck, x, rows, cols))


def test_awq_rejects_mismatched_tensors():
    ck = synth.make_awq_checkpoint(256, 256, 128, "fp16", seed=1)
    with pytest.raises(gptq.GptqError):
        gptq.gptq_repack_awq(ck.qweight.cuda(), ck.qzeros[:1].cuda(), ck.scales.cuda(), 128)
    with pytest.raises(gptq.GptqError):
        # N = 24 is not a multiple of 32 (the shapes agree with each other; the library refuses N)
        gptq.gptq_repack_awq(ck.qweight[:, :3].contiguous().cuda(), ck.qzeros[:, :3].contiguous().cuda(),
                             ck.scales[:, :24].contiguous().cuda(), 128)
