"""GB300 (sm_103a) GPTQ weight-only linear layer: y = x . dequant(qweight, qzeros, scales, g_idx)^T.

The compute lives in the CUDA library under csrc/ (C ABI: include/gptq.h); gptq.py is
its ctypes binding, synth.py draws seeded synthetic checkpoints, shard.py splits a
checkpoint by output features for one-process-per-GPU replicas.
"""
