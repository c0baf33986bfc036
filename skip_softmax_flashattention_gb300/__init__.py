"""GB300 (sm_103a) skip-softmax (BLASST) FlashAttention forward: prefill and split-KV decode.

The compute runs in the CUDA library built from ``csrc/`` (loaded lazily by
``skip_softmax_flashattention_gb300.blasst``); ``workloads`` draws the seeded
synthetic inputs.
"""
