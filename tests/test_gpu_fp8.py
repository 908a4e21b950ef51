"""GPU parity of the FP8 block-scaled W8A16 path (gptq_repack_fp8) through the C ABI, against
the oracle's FP8 reader: the runtime layout bit for bit, GEMMs element by element within
max|y - y_ref| <= 4e-3 max|y_ref| on both kernel families."""
import numpy as np
import pytest
import torch

import oracle
from weight_only_quantized_gb300 import gptq, synth

from gpu_util import compare

pytestmark = pytest.mark.gpu

# (K, N, dtype): tiny; ragged N block (288 = 2 blocks + 32); K not a multiple of 128 (padded tail)
CASES = [(256, 256, "bf16"), (256, 256, "fp16"), (384, 288, "bf16"), (320, 96, "fp16"), (640, 512, "bf16")]


def _id(c):
    return f"K{c[0]}N{c[1]}{c[2]}"


def _dt(name):
    return torch.float16 if name == "fp16" else torch.bfloat16


def _repack(ck):
    h = gptq.gptq_repack_fp8(ck.weight.cuda(), ck.scale_inv.cuda(), _dt(ck.dtype))
    torch.cuda.synchronize()
    return h


def _run(h, x_cpu, N, path):
    x = x_cpu.cuda()
    y = torch.full((x.shape[0], N), float("nan"), dtype=x.dtype, device="cuda")
    gptq.gptq_gemm_path(h, x, y, path)
    torch.cuda.synchronize()
    return y.cpu()


@pytest.mark.parametrize("case", CASES, ids=_id)
def test_fp8_layout_bit_exact(case):
    K, N, dt = case
    ck = synth.make_fp8_checkpoint(K, N, dt, seed=K + N)
    h = _repack(ck)
    got = gptq.gptq_copy_runtime(h)
    ref = oracle.runtime_layout_fp8(ck.weight)
    for key in ("Kr", "Np", "G"):
        assert got[key] == ref[key], key
    for key in ("perm", "cgid", "wr"):
        assert np.array_equal(got[key], ref[key]), key
    assert not got["s_r"].any() and not got["z_r"].any()
    info = gptq.gptq_get_info(h)
    assert info.fp8 == 1 and info.bits == 8 and info.group_size == 128


@pytest.mark.parametrize("case", CASES, ids=_id)
@pytest.mark.parametrize("M", [1, 3, 8, 17, 32])
def test_fp8_gemm_parity_small_path(case, M):
    K, N, dt = case
    ck = synth.make_fp8_checkpoint(K, N, dt, seed=N + 1)
    h = _repack(ck)
    x = synth.make_x(M, K, dt, seed=M)
    compare(_run(h, x, N, gptq.PATH_SMALL_M), oracle.fp8_linear(ck.weight, ck.scale_inv, dt, x))


@pytest.mark.parametrize("case", CASES, ids=_id)
@pytest.mark.parametrize("M", [1, 40, 129, 300])
def test_fp8_gemm_parity_large_path(case, M):
    K, N, dt = case
    ck = synth.make_fp8_checkpoint(K, N, dt, seed=N + 2)
    h = _repack(ck)
    gptq.gptq_reserve(h, 300)
    x = synth.make_x(M, K, dt, seed=M + 5)
    compare(_run(h, x, N, gptq.PATH_LARGE_M), oracle.fp8_linear(ck.weight, ck.scale_inv, dt, x))


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_fp8_every_code_and_extreme_factors(dt):
    """Each of the 254 numeric codes in every column (subnormals, +-448, both zeros) and block factors
    spanning 2^-20 .. 2^-6, one per block (outputs stay inside fp16's range)."""
    K, N = 512, 256
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    w = np.zeros((N, K), np.uint8)
    for n in range(N):
        w[n, :254] = np.roll(codes, n)
        w[n, 254:] = codes[(np.arange(K - 254) * 7 + n) % 254]
    s = torch.tensor([[2.0 ** -20, 2.0 ** -6, 2.0 ** -8, 2.0 ** -10], [3.0e-4, 7.0e-3, 2.0 ** -12, 1.2e-2]],
                     dtype=torch.float32)
    ck = synth.Fp8Checkpoint(K, N, dt, torch.from_numpy(w), s)
    h = _repack(ck)
    for M, path in ((4, gptq.PATH_SMALL_M), (64, gptq.PATH_LARGE_M)):
        x = synth.make_x(M, K, dt, seed=M)
        compare(_run(h, x, N, path), oracle.fp8_linear(ck.weight, ck.scale_inv, dt, x))


def test_fp8_one_hot_reads_single_weights():
    """x = e_k gives y[:, n] = round(W[n, k]) exactly: pins the pair order inside a 16-bit half
    (even k in the low byte), the block factor lookup and both conversions."""
    K, N = 256, 256
    for dt in ("bf16", "fp16"):
        ck = synth.make_fp8_checkpoint(K, N, dt, seed=31)
        W = oracle.fp8_dequant(ck.weight, ck.scale_inv)
        h = _repack(ck)
        ks = [0, 1, 2, 3, 126, 127, 128, 255]
        x = torch.zeros(len(ks), K, dtype=_dt(dt))
        for i, k in enumerate(ks):
            x[i, k] = 1.0
        for path in (gptq.PATH_SMALL_M, gptq.PATH_LARGE_M):
            y = _run(h, x, N, path)
            ref = torch.from_numpy(np.stack([W[:, k] for k in ks])).to(_dt(dt))
            assert torch.equal(y, ref), (dt, path)


def test_fp8_bias_and_dispatch():
    K, N = 512, 384
    ck = synth.make_fp8_checkpoint(K, N, "bf16", seed=9)
    h = _repack(ck)
    b = torch.randn(N, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    gptq.gptq_set_bias(h, b.cuda())
    gptq.gptq_reserve(h, 64)
    for M in (1, 24, 64):
        x = synth.make_x(M, K, "bf16", seed=M)
        y = _run(h, x, N, gptq.PATH_AUTO)
        ref = oracle.fp8_linear(ck.weight, ck.scale_inv, "bf16", x) + b.double().numpy()[None, :]
        compare(y, ref)


@pytest.mark.parametrize("M", [1, 16, 256])
def test_fp8_full_size_layer_sampled(M):
    """A 4096 x 14336 bf16 FP8 layer through gptq_gemm, sampled outputs against the oracle."""
    K, N = 4096, 14336
    ck = synth.make_fp8_checkpoint(K, N, "bf16", seed=41)
    h = _repack(ck)
    x = synth.make_x(M, K, "bf16", seed=42)
    y = _run(h, x, N, gptq.PATH_AUTO)
    rows = np.unique(np.linspace(0, M - 1, min(M, 4)).astype(np.int32))
    cols = np.random.default_rng(1).choice(N, 512, replace=False).astype(np.int32)
    compare(y[rows][:, cols], oracle.fp8_linear(ck.weight, ck.scale_inv, "bf16", x, rows, cols))


def test_fp8_rejects_mismatched_scales():
    ck = synth.make_fp8_checkpoint(256, 256, "bf16", seed=1)
    with pytest.raises(gptq.GptqError):
        gptq.gptq_repack_fp8(ck.weight.cuda(), ck.scale_inv[:1].contiguous().cuda(), torch.bfloat16)
