"""Host-side argument handling of the ctypes binding (no GPU, no kernel)."""

import pytest
import torch

from visual_token_sparsity_gb300 import binding as sv


def test_seq_batch_refuses_host_memory():
    """Every tensor handed to the library must be device memory: there is no
    host path to fall back to."""
    with pytest.raises(ValueError, match="CUDA"):
        sv.SeqBatch(torch.zeros(3, 4, dtype=torch.int32), 40, 8)


def test_seq_batch_struct_defaults_to_uniform_lengths():
    """A zero-initialised sv_seq_batch (as C callers write it) has no
    per-sequence arrays."""
    c = sv.sv_seq_batch(None, 3, 4, 40, 8)
    assert (c.batch, c.max_blocks, c.n_vis, c.n_text) == (3, 4, 40, 8)
    assert not c.n_vis_seq and not c.n_text_seq and not c.k_seq
