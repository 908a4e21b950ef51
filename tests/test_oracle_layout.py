"""Pins of the oracle's runtime-layout function.

The runtime layout is this library's own kernel-private format, so nothing on the
pages prints its bytes.  It is pinned by (1) invariants of the sorted, padded K
order the chapter-39 loader describes ("sorts the input columns by g_idx once at
load time, so that groups become contiguous"), and (2) a decode-back product:
reading every code out of the layout (field extraction, the inverse of how the
layout function inserts them) and multiplying by x gathered through perm must
give the checkpoint's y.  A wrong group id, a perm in the wrong direction, a
transposed lane or field index all break (2).
"""
import numpy as np
import pytest
import torch

import oracle
from weight_only_quantized_gb300 import synth


def _decode_layout(L, bits, N):
    """codes[j, n] for every sorted row j < Kr and real column n < N, read out of L['wr']."""
    Kr, Np = L["Kr"], L["Np"]
    words = L["wr"].view(np.uint32)
    j = np.arange(Kr)
    B, r = j // 128, j % 128
    c, t, e = r // 32, (r % 32) // 8, r % 8
    p, h = 4 * c + e // 2, e % 2
    planes = [(2, 0, 0), (1, 2, 2)] if bits == 3 else [(bits, 0, 0)]
    codes = np.zeros((Kr, N), np.int64)
    for bp, vbase, shift_into_code in planes:
        F = 16 // bp
        jw, f = p // F, p % F
        q = t * bp + jw
        v = q // 4
        V = vbase + v
        n = np.arange(N)[None, :]
        # inside a group of 32 columns, vector V's columns are rotated by rot(V)
        rot = {4: 2 * V, 8: 2 * (V // 2), 2: 4 * V, 3: np.where(V < 2, 4 * V, 0)}[bits][:, None]
        pos = n // 32 * 32 + (n % 32 + rot) % 32
        word_idx = ((B * bits + V)[:, None] * Np + pos) * 4 + (q % 4)[:, None]
        val = (words[word_idx].astype(np.int64) >> (16 * h + bp * f)[:, None]) & ((1 << bp) - 1)
        codes |= val << shift_into_code
    return codes


CASES = [
    # K, N, bits, group_size, desc_act, dtype
    (256, 256, 4, 128, False, "fp16"),
    (512, 96, 2, 64, True, "bf16"),
    (384, 64, 3, 128, True, "fp16"),
    (256, 288, 8, 32, True, "bf16"),
    (320, 32, 4, -1, False, "fp16"),       # K not a multiple of 128: padded tail
    (512, 64, 4, 96, False, "bf16"),       # groups of 96: each padded to 128
]


@pytest.mark.parametrize("K,N,bits,gs,da,dtype", CASES)
def test_layout_decodes_back_to_checkpoint_product(K, N, bits, gs, da, dtype):
    spec = synth.LayerSpec(K, N, bits, gs, da, dtype=dtype)
    ck = synth.make_checkpoint(spec, seed=K + N + bits)
    L = oracle.runtime_layout(ck.qweight, ck.qzeros, ck.scales, ck.g_idx, bits, gs)
    codes = _decode_layout(L, bits, N).astype(np.float64)
    perm, cgid = L["perm"], L["cgid"]
    g_of_row = cgid[np.arange(L["Kr"]) // 32]
    z = L["z_r"][:, :N].astype(np.float64) + 1.0
    s = torch.from_numpy(L["s_r"][:, :N].view(np.int16)).view(
        torch.float16 if dtype == "fp16" else torch.bfloat16).double().numpy()
    Wr = (codes - z[g_of_row]) * s[g_of_row]                   # [Kr, N] in sorted order
    x = synth.make_x(5, K, dtype, seed=3).double().numpy()
    xg = np.where(perm[None, :] >= 0, x[:, np.maximum(perm, 0)], 0.0)
    y_layout = xg @ Wr
    y_ref = oracle.linear(ck.qweight, ck.qzeros, ck.scales, ck.g_idx, bits, gs, dtype,
                          synth.make_x(5, K, dtype, seed=3))
    assert np.allclose(y_layout, y_ref, rtol=1e-11, atol=1e-11)


@pytest.mark.parametrize("K,N,bits,gs,da,dtype", CASES)
def test_layout_invariants(K, N, bits, gs, da, dtype):
    spec = synth.LayerSpec(K, N, bits, gs, da, dtype=dtype)
    ck = synth.make_checkpoint(spec, seed=1)
    L = oracle.runtime_layout(ck.qweight, ck.qzeros, ck.scales, ck.g_idx, bits, gs)
    Kr, Np, G = L["Kr"], L["Np"], L["G"]
    perm, cgid = L["perm"], L["cgid"]
    assert Kr % 128 == 0 and Kr >= K and Np % 256 == 0 and Np >= N
    real = perm[perm >= 0]
    assert np.array_equal(np.sort(real), np.arange(K))          # each input feature exactly once
    g_idx = synth.sequential_g_idx(K, gs).numpy() if ck.g_idx is None else ck.g_idx.numpy()
    rows = np.nonzero(perm >= 0)[0]
    assert np.array_equal(g_idx[perm[rows]], cgid[rows // 32])  # every row sits in its group's chunks
    assert np.all(np.diff(cgid) >= 0)                           # groups ascend
    for g in range(G):                                          # inside a group, k ascends (stable)
        ks = perm[rows][g_idx[perm[rows]] == g]
        assert np.all(np.diff(ks) > 0)
    assert L["wr"].size == Kr // 128 * bits * Np * 16
    assert np.all(L["s_r"][:, N:] == 0) and np.all(L["z_r"][:, N:] == 0)


def test_unbalanced_groups_pad_each_run_to_32():
    """Any g_idx with values in range is accepted (GPTQ-004); uneven group sizes pad to 32."""
    K, N, G = 256, 64, 4
    rng = np.random.default_rng(0)
    g_idx = rng.integers(0, G, size=K).astype(np.int32)
    g_idx[g_idx == 2] = 1                                       # group 2 left empty
    ck = synth.make_checkpoint(synth.LayerSpec(K, N, 4, 64), seed=2)
    L = oracle.runtime_layout(ck.qweight, ck.qzeros, ck.scales, g_idx, 4, 64)
    counts = np.bincount(g_idx, minlength=G)
    assert L["Kr"] == -(-sum(-(-c // 32) * 32 for c in counts) // 128) * 128
    assert 2 not in set(L["cgid"].tolist())
    codes = _decode_layout(L, 4, N).astype(np.float64)
    g_of_row = L["cgid"][np.arange(L["Kr"]) // 32]
    s = ck.scales.double().numpy()
    Wr = (codes - (L["z_r"][:, :N].astype(np.float64) + 1.0)[g_of_row]) * s[g_of_row]
    W = oracle.dequant(ck.qweight, ck.qzeros, ck.scales, g_idx, 4, 64, "fp16").astype(np.float64)
    rows = np.nonzero(L["perm"] >= 0)[0]
    assert np.array_equal(Wr[rows], W[:, L["perm"][rows]].T)
