"""CPU checks of the C ABI: libsv.so builds, loads without a GPU, exports every
function include/sv.h declares (and no other sv_ symbol), and its host-side
argument checks reject bad calls before anything is launched."""

import ctypes
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sv.h")


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sv_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def so():
    if not shutil.which("nvcc") and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    from visual_token_sparsity_gb300 import build
    return build.build()


def test_header_declares_the_boundary_calls():
    names = header_functions()
    for n in ("sv_salience_prefill", "sv_prune_compact", "sv_retrieve_topk", "sv_sparse_decode_attn",
              "sv_evict_qa_tokens", "sv_kv_append", "sv_topk_rows", "sv_read_device_status"):
        assert n in names


def test_library_exports_exactly_the_header(so):
    out = subprocess.run(["nm", "-D", "--defined-only", so], capture_output=True, text=True).stdout
    exported = sorted(set(re.findall(r"\bT (sv_[a-z0-9_]+)$", out, flags=re.M)))
    assert exported == header_functions()
    from visual_token_sparsity_gb300 import binding
    assert sorted(binding.EXPORTED) == header_functions()


def test_library_loads_without_gpu_and_reports_version(so):
    from visual_token_sparsity_gb300 import binding
    lib = binding.load(so)
    assert lib.sv_version().decode().startswith("sv ")
    assert lib.sv_status_string(4).decode() == "workspace too small"


def _fake(addr=0x10000):
    return ctypes.c_void_p(addr)


def test_host_validation_rejects_before_launch(so):
    from visual_token_sparsity_gb300 import binding
    lib = binding.load(so)
    s = ctypes.c_void_p(0)
    # k > n
    assert lib.sv_topk_rows(_fake(), 2, 10, 11, _fake(), _fake(), 256, s) == 1
    assert b"k" in lib.sv_last_error()
    # workspace too small
    assert lib.sv_topk_rows(_fake(), 2, 10, 5, _fake(), _fake(), 16, s) == 4
    # misaligned workspace
    assert lib.sv_topk_rows(_fake(), 2, 10, 5, _fake(), _fake(0x10004), 256, s) == 1
    # salience: unsupported head dim, bad scale, too large N
    assert lib.sv_salience_prefill(_fake(), _fake(), 1, 1, 16, 96, 0.1, _fake(), _fake(), 1 << 20, s) == 2
    assert lib.sv_salience_prefill(_fake(), _fake(), 1, 1, 16, 64, -1.0, _fake(), _fake(), 1 << 20, s) == 1
    assert lib.sv_salience_prefill(_fake(), _fake(), 1, 1, (1 << 24) + 1, 128, 0.1, _fake(), _fake(), 1 << 30, s) == 2
    # retrieval: k > n_vis, H not a multiple of Hkv, head dim 72 unsupported
    layer = binding.sv_kv_layer(_fake(), _fake(), 100, 2, 64)
    seqs = binding.sv_seq_batch(_fake(), 1, 10, 100, 10)
    args = lambda R, H, k: (_fake(), R, H, ctypes.byref(layer), ctypes.byref(seqs), k, _fake(), None,
                            _fake(), 1 << 20, s)
    assert lib.sv_retrieve_topk(*args(1, 4, 101)) == 1
    assert lib.sv_retrieve_topk(*args(1, 3, 10)) == 1
    layer72 = binding.sv_kv_layer(_fake(), _fake(), 100, 2, 72)
    assert lib.sv_retrieve_topk(_fake(), 1, 4, ctypes.byref(layer72), ctypes.byref(seqs), 10, _fake(),
                                None, _fake(), 1 << 20, s) == 2
    # lengths beyond the block table
    seqs_long = binding.sv_seq_batch(_fake(), 1, 10, 150, 20)
    assert lib.sv_retrieve_topk(_fake(), 1, 4, ctypes.byref(layer), ctypes.byref(seqs_long), 10, _fake(),
                                None, _fake(), 1 << 20, s) == 1
    # attention: group size above 16
    layer1 = binding.sv_kv_layer(_fake(), _fake(), 100, 1, 64)
    assert lib.sv_sparse_decode_attn(_fake(), 17, 0.1, ctypes.byref(layer1), ctypes.byref(seqs), None, 0,
                                     _fake(), None, _fake(), 1 << 20, s) == 2
    # fused decode step: missing or misaligned new-token rows, no page for the new token
    fused = lambda seq, kn, vn: lib.sv_decode_append_attn(_fake(), 4, 0.1, ctypes.byref(layer), ctypes.byref(seq),
                                                          kn, vn, None, 0, _fake(), None, _fake(), 1 << 20, s)
    assert fused(seqs, None, _fake()) == 1
    assert b"k_new" in lib.sv_last_error()
    assert fused(seqs, _fake(0x10008), _fake()) == 1
    seqs_full = binding.sv_seq_batch(_fake(), 1, 10, 150, 10)    # 160 tokens fill the 10 pages
    assert fused(seqs_full, _fake(), _fake()) == 1
    assert b"overflows" in lib.sv_last_error()
    # eviction span outside the text
    assert lib.sv_evict_qa_tokens(ctypes.byref(layer), 1, ctypes.byref(seqs), 5, 11, None, _fake(), 256, s) == 1
    assert seqs.n_text == 10


def test_workspace_sizes_are_monotone_in_tokens(so):
    from visual_token_sparsity_gb300 import binding
    lib = binding.load(so)
    for B, H, Hkv, d in ((1, 32, 32, 128), (16, 32, 32, 128), (8, 28, 4, 128), (1, 4, 2, 64)):
        prev = 0
        for n in range(1, 60000, 97):
            w = lib.sv_attn_workspace_bytes(B, H, Hkv, d, n)
            assert w >= prev and w >= 256
            prev = w
    assert lib.sv_retrieve_workspace_bytes(16, 32, 32, 128, 2880, 720) >= 256 + 16 * 32 * 2880 * 4
    assert lib.sv_salience_workspace_bytes(256, 16, 729, 72) >= 256 + 256 * 16 * 729 * 4
    # the streamed schedule also keeps a 16-byte fold record per query
    assert lib.sv_salience_workspace_bytes(1, 16, 16384, 80) >= 256 + 16 * 16384 * (4 + 16)


def test_salience_schedule_switch_and_kernel_counts(so):
    """Resident schedule up to 1024 tokens at d 64 / 72, 768 at d 80, 512 at
    d 128 (3 kernels: salience, exact re-run, head mean); streamed beyond
    (4 kernels: row pass, re-run, column pass, head mean)."""
    from visual_token_sparsity_gb300 import binding
    lib = binding.load(so)
    for d, cap in ((64, 1024), (72, 1024), (80, 768), (128, 512)):
        assert lib.sv_salience_kernel_count(1, d) == 3
        assert lib.sv_salience_kernel_count(cap, d) == 3
        assert lib.sv_salience_kernel_count(cap + 1, d) == 4
        assert lib.sv_salience_kernel_count(50000, d) == 4
    assert lib.sv_salience_kernel_count(100, 96) == 0
    assert lib.sv_salience_kernel_count(0, 64) == 0


def test_ctypes_structs_match_the_header_layout(tmp_path):
    """The binding's ctypes mirrors of sv_kv_layer and sv_seq_batch have the
    C compiler's size and field offsets (a probe compiled against sv.h)."""
    if not shutil.which("gcc"):
        pytest.skip("gcc not available")
    from visual_token_sparsity_gb300 import binding
    probe = tmp_path / "layout.c"
    fields = {"sv_kv_layer": [f for f, _ in binding.sv_kv_layer._fields_],
              "sv_seq_batch": [f for f, _ in binding.sv_seq_batch._fields_]}
    lines = ["#include <stddef.h>", "#include <stdio.h>", '#include "sv.h"', "int main(void) {"]
    for st, fs in fields.items():
        lines.append(f'  printf("{st} size %zu\\n", sizeof({st}));')
        for f in fs:
            lines.append(f'  printf("{st} {f} %zu\\n", offsetof({st}, {f}));')
    lines += ["  return 0;", "}"]
    probe.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), str(probe), "-o", str(exe)],
                   check=True)
    got = {}
    for line in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.splitlines():
        st, f, v = line.split()
        got[(st, f)] = int(v)
    for st, cls in (("sv_kv_layer", binding.sv_kv_layer), ("sv_seq_batch", binding.sv_seq_batch)):
        assert got[(st, "size")] == ctypes.sizeof(cls), st
        for f, _ in cls._fields_:
            assert got[(st, f)] == getattr(cls, f).offset, f"{st}.{f}"


def test_kernel_count_queries(so):
    """Pure host queries: LLaVA-NeXT rows fuse the top-k and the split merge
    (one kernel each); LongVILA's 50176-key rows need a separate top-k, and
    grouped-query attention (G >= 3) always merges its splits in a separate
    kernel, however short the call."""
    from visual_token_sparsity_gb300 import binding
    lib = binding.load(so)
    assert lib.sv_retrieve_kernel_count(1, 32, 2880) == 1     # a few rows: top-k fused
    assert lib.sv_retrieve_kernel_count(16, 32, 2880) == 2    # many rows: separate top-k
    assert lib.sv_retrieve_kernel_count(1, 4, 50176) == 2     # long rows
    assert lib.sv_retrieve_kernel_count(1, 4, 0) == 0
    assert lib.sv_attn_kernel_count(16, 32, 32, 1440 + 128) == 1
    assert lib.sv_attn_kernel_count(8, 28, 4, 12544 + 256) == 2
    assert lib.sv_attn_kernel_count(16, 28, 4, 784 + 256) == 2
    assert lib.sv_attn_kernel_count(1, 28, 4, 40) == 2
    assert lib.sv_attn_kernel_count(1, 4, 2, 144 + 64) == 1    # the round-loop shape (G 2)
    assert lib.sv_attn_kernel_count(1, 28, 5, 100) == 0   # H not a multiple of n_kv_heads
