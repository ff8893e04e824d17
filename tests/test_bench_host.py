"""Host-side logic of bench.py that needs no GPU: the per-sequence-length
workload stays inside its capacities and its byte count reduces to the
uniform one when every sequence has the batch-wide counts."""

import bench
from visual_token_sparsity_gb300 import synth


def test_varlen_counts_within_capacities():
    shape = synth.llava_next_decode(batch=16, keep=0.5, layers=32)
    nv, nt, k = bench.varlen_counts(shape)
    assert len(nv) == len(nt) == len(k) == 16
    for v, t, kk in zip(nv, nt, k):
        assert shape.n_vis // 2 <= v <= shape.n_vis
        assert shape.n_text // 2 <= t <= shape.n_text
        assert 0 <= kk <= min(v, shape.k)
    assert bench.varlen_counts(shape) == (nv, nt, k), "counts must be seeded"


def test_varlen_bytes_reduce_to_uniform():
    shape = synth.llava_next_decode(batch=4, keep=0.5, layers=3)
    B = shape.batch
    rb, ab = bench.decode_bytes(shape)
    assert bench.varlen_bytes(shape, [shape.n_vis] * B, [shape.n_text] * B, [shape.k] * B) == rb + ab
