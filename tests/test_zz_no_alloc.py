"""gptq_repack_noalloc: the repack for callers that cannot allocate device memory at load time
(all weights carved from one pre-reserved arena, or an allocator owned by another framework).

The test hands it caller-owned buffers through the C ABI and checks that its output equals, bit
for bit, the runtime layout gptq_repack builds for the same checkpoint -- on two calls in a row,
the second with fewer groups than the first, so scratch left over from the first call would show.
This file is named to be collected last.
"""
import numpy as np
import pytest
import torch

from weight_only_quantized_gb300 import gptq, synth

pytestmark = pytest.mark.gpu


def _reference_layout(ck):
    d = dict(qweight=ck.qweight.cuda(), qzeros=ck.qzeros.cuda(), scales=ck.scales.cuda(),
             g_idx=None if ck.g_idx is None else ck.g_idx.cuda())
    h = gptq.gptq_repack(d["qweight"], d["qzeros"], d["scales"], d["g_idx"], ck.spec.bits, ck.spec.group_size)
    out = gptq.gptq_copy_runtime(h)
    h.close()
    return out


def _noalloc_layout(ck):
    s = ck.spec
    G, Np = s.G, -(-s.N // 256) * 256
    kr_cap = -(-(s.K + 31 * G) // 128) * 128
    dev = "cuda"
    wr = torch.empty(kr_cap // 128 * s.bits * Np * 16, dtype=torch.uint8, device=dev)
    perm = torch.empty(kr_cap, dtype=torch.int32, device=dev)
    cgid = torch.empty(kr_cap // 32, dtype=torch.int32, device=dev)
    s_r = torch.empty((G, Np), dtype=torch.int16, device=dev)
    z_r = torch.empty((G, Np), dtype=torch.uint8, device=dev)
    kr = gptq.gptq_repack_noalloc(ck.qweight.cuda(), ck.qzeros.cuda(), ck.scales.cuda(),
                                  None if ck.g_idx is None else ck.g_idx.cuda(), s.bits, s.group_size,
                                  wr, perm, cgid, s_r, z_r)
    torch.cuda.synchronize()
    wr_bytes = kr // 128 * s.bits * Np * 16
    return dict(Kr=kr, wr=wr[:wr_bytes].cpu().numpy(), perm=perm[:kr].cpu().numpy(),
                cgid=cgid[:kr // 32].cpu().numpy(), s_r=s_r.cpu().numpy().view(np.uint16), z_r=z_r.cpu().numpy())


def test_noalloc_repack_matches_gptq_repack_twice():
    first = synth.LayerSpec(1024, 512, 4, 32, True, False, "bf16")      # 32 groups, act-order
    second = synth.LayerSpec(512, 288, 3, 128, True, False, "fp16")     # 4 groups, ragged N
    for spec, seed in ((first, 5), (second, 6)):
        ck = synth.make_checkpoint(spec, seed=seed)
        ref = _reference_layout(ck)
        got = _noalloc_layout(ck)
        assert got["Kr"] == ref["Kr"]
        for key in ("perm", "cgid", "s_r", "z_r", "wr"):
            assert np.array_equal(got[key], ref[key]), (spec, key)


def test_noalloc_rejects_too_many_groups_and_small_buffers():
    # 8192 groups > the fixed scratch's 4096: refused by the library (the outputs are sized right, so
    # the binding's own checks pass)
    spec = synth.LayerSpec(8192 * 4, 64, 4, 4, False, False, "fp16")
    ck = synth.make_checkpoint(spec, seed=1)
    G, Np = spec.G, 256
    kr_cap = -(-(spec.K + 31 * G) // 128) * 128
    perm = torch.empty(kr_cap, dtype=torch.int32, device="cuda")
    cgid = torch.empty(kr_cap // 32, dtype=torch.int32, device="cuda")
    s_r = torch.empty((G, Np), dtype=torch.int16, device="cuda")
    z_r = torch.empty((G, Np), dtype=torch.uint8, device="cuda")
    wr = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(gptq.GptqError) as ei:
        gptq.gptq_repack_noalloc(ck.qweight.cuda(), ck.qzeros.cuda(), ck.scales.cuda(), None, 4, 4,
                                 wr, perm, cgid, s_r, z_r)
    assert ei.value.status == 2 and "4096" in str(ei.value)
    # code and perm buffers smaller than the sorted K: refused after the histogram, nothing written
    spec = synth.LayerSpec(512, 256, 4, 128)
    ck = synth.make_checkpoint(spec, seed=2)
    tiny = torch.empty(16, dtype=torch.int32, device="cuda")
    s_r = torch.empty((spec.G, 256), dtype=torch.int16, device="cuda")
    z_r = torch.empty((spec.G, 256), dtype=torch.uint8, device="cuda")
    with pytest.raises(gptq.GptqError) as ei:
        gptq.gptq_repack_noalloc(ck.qweight.cuda(), ck.qzeros.cuda(), ck.scales.cuda(), None, 4, 128,
                                 tiny.view(torch.uint8), tiny, tiny, s_r, z_r)
    assert ei.value.status == 6
