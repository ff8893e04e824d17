"""GB300-native SparseVILA hot path: salience prefill pruning, query-aware
retrieval and sparse decode attention over a paged bf16 KV cache.

The compute runs in the CUDA library ``libsv`` (hand-written sm_103a kernels
behind a C ABI, declared in ``include/sv.h``); :mod:`.binding` marshals
arguments to it.  :mod:`.synth` draws seeded synthetic inputs.
"""

__all__ = ["binding", "synth", "build"]
