"""Benchmark of the SparseVILA hot path on GB300.

Default workload: LLaVA-NeXT-7B-shaped decode (Llama-2-7B attention: 32 MHA
heads, head_dim 128, 32 layers; paged bf16 KV with 16-token pages; 2880
visual + 128 text tokens per sequence; batch 16; retrieval keeps 50%).
One step = one decode step over all 32 layers, each layer running query-aware
retrieval (1 query row) followed by sparse decode attention over the selected
visual tokens plus all text tokens.  The step is captured once in a CUDA graph
and replayed.  Inputs are seeded synthetic tensors (no weights or datasets).

The line also carries the prefill salience figure (SigLIP-so400m shape, 256
frames of 729 tokens, 16 heads, d 72) in tokens/s and as a fraction of the
dense bf16 tensor peak.

Usage: python bench.py [--gpus N --steps K --warmup W] [--impl reference]
Multi-GPU (torchrun): every rank runs an independent replica of the workload
(weak scaling, no collective on the data path).
"""

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
# the CPU oracle leg is timed single-threaded (reported as cores = 1)
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "sparse decode step µs & KV-read GB/s vs HBM peak; salience tokens/s vs TC peak"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="sv", choices=["sv", "reference"])
    p.add_argument("--batch", type=int, default=None, help="default: 16 (llava), 8 (longvila), 1 (tiny, rounds)")
    p.add_argument("--keep", type=float, default=0.5)
    p.add_argument("--layers", type=int, default=None, help="default: the model's layer count")
    p.add_argument("--workload", default="llava", choices=["llava", "longvila", "tiny", "rounds"],
                   help="decode shape: LLaVA-NeXT-7B (default, the bench line), LongVILA-7B, the tiny "
                        "single-layer case, or the 5-round question/answer loop on the tiny shapes")
    p.add_argument("--salience-batch", type=int, default=256)
    p.add_argument("--no-salience", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-decode", action="store_true", help="salience measurement only")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-packed", action="store_true", help="skip the pack-once KV comparison")
    p.add_argument("--no-varlen", action="store_true", help="skip the per-sequence-length decode step")
    p.add_argument("--salience-long-n", type=int, default=16384,
                   help="tokens of the long-sequence salience object (0: skip it)")
    p.add_argument("--no-extra", action="store_true",
                   help="skip the LongVILA, other LLaVA-NeXT, tiny-case and round-loop objects of the default line")
    return p.parse_args()


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    hbm, bf16, bf16_sus, src = FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            hbm = float(d.get("hbm_gbs", hbm))
            bf16 = float(d.get("bf16_tflops", bf16))
            bf16_sus = float(d.get("bf16_tflops_sustained", bf16_sus))
            src = "measured"
        except Exception:
            pass
    return {"hbm_gbs": hbm, "bf16_tflops": bf16, "bf16_tflops_sustained": bf16_sus, "source": src}


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)      # let the sampler start before the timed region
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- workload

def measured_traffic(call):
    """DRAM bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum)
    recorded in profiles/traffic.json for this C call, or None when the
    kernel source has changed since the counters were taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        rec = json.load(open(path))[call]
        h = hashlib.sha1()
        for src in rec["sources"]:      # every file the kernel is built from
            h.update(open(os.path.join(ROOT, src), "rb").read())
        if h.hexdigest() != rec["sources_sha1"]:
            return None
        return rec["bytes_per_launch"]
    except Exception:
        return None


def aggregate_replicas(per_rank_ms, bytes_per_rank, world, all_reduce_max=None):
    """Whole-job figure for N independent replicas: each rank processed
    bytes_per_rank; the job time is the slowest rank's.  all_reduce_max
    (a callable list -> list, e.g. a torch.distributed MAX all-reduce) is
    applied to the per-rank times when world > 1.  Returns (ms, GB/s)."""
    ms = list(per_rank_ms)
    if world > 1 and all_reduce_max is not None:
        ms = all_reduce_max(ms)
    return ms, world * bytes_per_rank / (ms[0] * 1e-3) / 1e9


def torch_max_reducer(device):
    import torch.distributed as dist

    def red(vals):
        t = torch.tensor(vals, dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return t.tolist()
    return red


def decode_bytes(shape):
    """Algorithmic HBM bytes of one decode step (all layers, whole batch)."""
    d2 = shape.d * 2
    retrieve = shape.n_vis * shape.Hkv * d2                                # visual keys
    attend = (shape.k + shape.n_text) * shape.Hkv * d2 * 2 + shape.k * shape.Hkv * 4   # K+V + indices
    return shape.layers * shape.batch * retrieve, shape.layers * shape.batch * attend


def varlen_counts(shape):
    """Per-sequence (n_vis, n_text, k) of a threshold-pruned batch: a salience
    threshold keeps a different share of each sequence's visual tokens, so
    visual counts are drawn uniformly from [n_vis / 2, n_vis], text counts
    from [n_text / 2, n_text], and each sequence selects floor(keep * n_vis_b)
    (seeded; the batch-wide counts are the capacities)."""
    rng = np.random.default_rng(shape.seed + 17)
    nv = rng.integers(shape.n_vis // 2, shape.n_vis + 1, size=shape.batch)
    nt = rng.integers(shape.n_text // 2, shape.n_text + 1, size=shape.batch)
    k = np.floor(shape.keep * nv).astype(np.int64)
    return [int(x) for x in nv], [int(x) for x in nt], [int(x) for x in k]


def varlen_bytes(shape, nv, nt, k):
    """Algorithmic HBM bytes of one decode step with per-sequence counts."""
    d2 = shape.d * 2
    per_seq = [v * shape.Hkv * d2 + (kk + t) * shape.Hkv * d2 * 2 + kk * shape.Hkv * 4 for v, t, kk in zip(nv, nt, k)]
    return shape.layers * sum(per_seq)


class DecodeWorkload:
    def __init__(self, shape, dev):
        from visual_token_sparsity_gb300 import binding as sv, synth
        self.sv, self.shape, self.dev = sv, shape, dev
        s = shape
        bt = synth.random_block_table(s.batch, s.max_blocks, s.num_blocks, seed=synth.subseed(s.seed, 0, 99))
        self.bt = bt.to(dev)
        self.seqs = sv.SeqBatch(self.bt, s.n_vis, s.n_text)
        self.layers = []
        for l in range(s.layers):
            lay = synth.draw_decode_layer(s, l, self.bt, device=dev)
            self.layers.append(sv.KvLayer(lay.k_pool, lay.v_pool))
            del lay
        qs = [synth.draw_decode_queries(s, l, device=dev) for l in range(s.layers)]
        self.q_rows = torch.stack([q[0] for q in qs])      # [L][B][1][H][d]
        self.q_dec = torch.stack([q[1] for q in qs])       # [L][B][H][d]
        self.vis = torch.empty(s.layers, s.batch, s.Hkv, s.k, dtype=torch.int32, device=dev)
        self.out = torch.empty(s.layers, s.batch, s.H, s.d, dtype=torch.bfloat16, device=dev)
        self.ws_r = sv.workspace(sv.sv_retrieve_workspace_bytes(s.batch, s.H, s.Hkv, s.d, s.n_vis, s.k), dev)
        self.ws_a = sv.workspace(sv.sv_attn_workspace_bytes(s.batch, s.H, s.Hkv, s.d, s.k + s.n_text), dev)
        self.scale = 1.0 / math.sqrt(s.d)
        torch.cuda.synchronize()

    def retrieve(self, l, q_rows=None):
        s = self.shape
        self.sv.sv_retrieve_topk(self.q_rows[l] if q_rows is None else q_rows, self.layers[l], self.seqs, s.k,
                                 self.vis[l], None, self.ws_r)

    def attend(self, l, q=None, out=None):
        s = self.shape
        self.sv.sv_sparse_decode_attn(self.q_dec[l] if q is None else q, self.scale, self.layers[l], self.seqs,
                                      self.vis[l], s.k, self.out[l] if out is None else out, None, self.ws_a)

    def step(self):
        for l in range(self.shape.layers):
            self.retrieve(l)
            self.attend(l)

    def attn_only_step(self):
        for l in range(self.shape.layers):
            self.attend(l)

    def retrieve_only_step(self):
        for l in range(self.shape.layers):
            self.retrieve(l)

    # pack-once KV: per layer a second paged layer holding, per (sequence, KV
    # head), the selected visual rows then the text rows contiguously
    def make_packed(self):
        sv, s = self.sv, self.shape
        n = s.k + s.n_text
        nblk = (n + 15) // 16
        bt = torch.arange(s.batch * nblk, dtype=torch.int32, device=self.dev).view(s.batch, nblk)
        self.pseqs = sv.SeqBatch(bt, s.k, s.n_text)
        self.players = []
        for l in range(s.layers):
            kp = torch.empty(s.batch * nblk, s.Hkv, 16, s.d, dtype=torch.bfloat16, device=self.dev)
            self.players.append(sv.KvLayer(kp, torch.empty_like(kp)))
        self.ws_p = sv.workspace(256, self.dev)

    def pack_all(self):
        for l in range(self.shape.layers):
            self.sv.sv_pack_kv(self.layers[l], self.seqs, self.vis[l], self.shape.k, self.players[l], self.pseqs,
                               self.ws_p)

    def attn_packed_step(self):
        s = self.shape
        for l in range(s.layers):
            self.sv.sv_sparse_decode_attn(self.q_dec[l], self.scale, self.players[l], self.pseqs, None, 0,
                                          self.out[l], None, self.ws_a)


def time_graph(fn, steps, warmup, stream):
    # the side stream starts after everything already queued on the current
    # stream (inputs drawn, outputs allocated from memory it may still read)
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        for _ in range(max(1, warmup)):
            fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            g.replay()
    torch.cuda.synchronize()
    return g


def replay_timed(g, steps, stream, barrier):
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(steps):
            g.replay()
        end.record(stream)
    torch.cuda.synchronize()
    barrier()
    return start.elapsed_time(end) / steps      # ms per step


def decode_graph_times(wl, steps, warmup, stream, barrier, clocks=None):
    """Device time per step (ms) of three CUDA graphs over all layers:
    retrieval + attention, attention only and retrieval only.  Per-call
    kernel times are the single-call graphs' step time / layers, so launch
    gaps between graphs never count as kernel time."""
    g_step = time_graph(wl.step, steps, max(3, warmup), stream)
    g_attn = time_graph(wl.attn_only_step, steps, 3, stream)
    g_ret = time_graph(wl.retrieve_only_step, steps, 3, stream)
    if clocks is not None:
        with clocks:
            ms = replay_timed(g_step, steps, stream, barrier)
    else:
        ms = replay_timed(g_step, steps, stream, barrier)
    ms_attn = replay_timed(g_attn, steps, stream, barrier)
    ms_ret = replay_timed(g_ret, steps, stream, barrier)
    del g_step, g_attn, g_ret
    return ms, ms_attn, ms_ret


def e2e_throughput(wl, steps, warmup, stream, bytes_step):
    """Same metric through the public C-ABI with host buffers: per step the
    queries come from pinned host memory and the attention outputs go back."""
    s = wl.shape
    hq_rows = torch.empty_like(wl.q_rows, device="cpu").pin_memory()
    hq_dec = torch.empty_like(wl.q_dec, device="cpu").pin_memory()
    hq_rows.copy_(wl.q_rows.cpu())
    hq_dec.copy_(wl.q_dec.cpu())
    hout = torch.empty_like(wl.out, device="cpu").pin_memory()
    dq_rows = torch.empty_like(wl.q_rows)
    dq_dec = torch.empty_like(wl.q_dec)

    def one():
        dq_rows.copy_(hq_rows, non_blocking=True)
        dq_dec.copy_(hq_dec, non_blocking=True)
        for l in range(s.layers):
            wl.retrieve(l, dq_rows[l])
            wl.attend(l, dq_dec[l])
        hout.copy_(wl.out, non_blocking=True)

    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            one()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(steps):
            one()
        torch.cuda.synchronize()
        dt = (time.perf_counter() - t0) / steps
    h2d = hq_rows.numel() * 2 + hq_dec.numel() * 2
    d2h = hout.numel() * 2
    return bytes_step / dt / 1e9, h2d, d2h


def summary_salience_measure(cs, steps, stream):
    """Summary-row salience (CLIP CLS row) over the frames of `cs`: device
    time per call (CUDA graph), and the algorithmic HBM bytes of one call."""
    from visual_token_sparsity_gb300 import binding as sv, synth
    q, k, _ = synth.draw_salience(cs, device="cuda")
    sal = torch.empty(cs.batch, cs.N, device="cuda")
    ws = sv.workspace(sv.sv_salience_summary_workspace_bytes(cs.batch, cs.H, cs.N, cs.d, 1))
    fn = lambda: sv.sv_salience_summary(q, k, 1, 1 / math.sqrt(cs.d), sal, ws)
    g = time_graph(fn, steps, 3, stream)
    ms = replay_timed(g, steps, stream, lambda: None)
    nbytes = cs.batch * cs.H * (cs.N + 1) * cs.d * 2 + cs.batch * cs.N * 4
    return ms * 1e3, nbytes


def salience_measure(batch, steps, warmup, stream, tiny=False, shape=None):
    from visual_token_sparsity_gb300 import binding as sv, synth
    ss = shape or (synth.tiny_salience(batch=batch) if tiny else synth.siglip_salience(batch=batch))
    q, k, _ = synth.draw_salience(ss, device="cuda")
    sal = torch.empty(ss.batch, ss.N, device="cuda")
    ws = sv.workspace(sv.sv_salience_workspace_bytes(ss.batch, ss.H, ss.N, ss.d))
    # rotate across copies so that repeated calls read more than L2 holds
    ncopy = max(1, math.ceil(3 * 129e6 / (2 * q.numel() * 2)))
    qs = [q] + [q.clone() for _ in range(ncopy - 1)]
    ks = [k] + [k.clone() for _ in range(ncopy - 1)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        for i in range(warmup):
            sv.sv_salience_prefill(qs[i % ncopy], ks[i % ncopy], 1 / math.sqrt(ss.d), sal, ws)
        torch.cuda.synchronize()
        start.record(stream)
        for i in range(steps):
            sv.sv_salience_prefill(qs[i % ncopy], ks[i % ncopy], 1 / math.sqrt(ss.d), sal, ws)
        end.record(stream)
    torch.cuda.synchronize()
    ms = start.elapsed_time(end) / steps
    flops = 4.0 * ss.H * ss.N * ss.N * ss.d * ss.batch
    return ss, ms, flops


def prune_measure(batch, steps, stream, pk):
    """Top-k prune + compaction (sv_prune_compact) and threshold prune
    (sv_prune_threshold) of the SigLIP features on real salience: GB/s of the
    algorithmic bytes (salience read, kept rows read and written, indices),
    device time per call from CUDA-graph replay."""
    from visual_token_sparsity_gb300 import binding as sv, synth
    ss = synth.siglip_salience(batch=batch)
    q, k, feat = synth.draw_salience(ss, device="cuda")
    B, N, C = ss.batch, ss.N, ss.C
    sal = torch.empty(B, N, device="cuda")
    ws = sv.workspace(max(sv.sv_salience_workspace_bytes(B, ss.H, N, ss.d), sv.sv_prune_workspace_bytes(B, N, N)))
    sv.sv_salience_prefill(q, k, 1 / math.sqrt(ss.d), sal, ws)
    torch.cuda.synchronize()     # q and k are read until here
    del q, k
    kept = torch.empty(B, ss.k, dtype=torch.int32, device="cuda")
    fout = torch.empty(B, ss.k, C, dtype=torch.bfloat16, device="cuda")
    tidx = torch.empty(B, N, dtype=torch.int32, device="cuda")
    tcnt = torch.empty(B, dtype=torch.int32, device="cuda")
    tout = torch.empty(B, N, C, dtype=torch.bfloat16, device="cuda")
    thr = 1.0 / N     # the mean salience
    # three feature copies, one per call of a graph: consecutive calls read
    # rows of different copies (each call reads and writes more than L2 holds)
    feats = [feat] + [feat.clone() for _ in range(2)]
    calls = {"topk": lambda f: sv.sv_prune_compact(sal, ss.k, f, fout, kept, ws),
             "threshold": lambda f: sv.sv_prune_threshold(sal, thr, f, tout, tidx, tcnt, ws)}
    us = {}
    for name, fn in calls.items():
        g = time_graph(lambda: [fn(f) for f in feats], steps, 3, stream)
        us[name] = replay_timed(g, steps, stream, lambda: None) * 1e3 / len(feats)
        del g
    row = C * 2
    kept_t = int(tcnt.sum().item())
    b_topk = B * N * 4 + B * ss.k * (2 * row + 4)
    b_thr = B * N * 4 + B * N * 4 + B * 4 + kept_t * 2 * row
    out = {"workload": f"{ss.name}: {B} frames x {N} tokens, {C}-wide bf16 features",
           "topk_us": us["topk"], "topk_keep": ss.keep, "topk_gbs": b_topk / (us["topk"] * 1e-6) / 1e9,
           "threshold_us": us["threshold"], "threshold": "mean salience (1/N)",
           "threshold_kept_fraction": kept_t / (B * N),
           "threshold_gbs": b_thr / (us["threshold"] * 1e-6) / 1e9, "peak": pk["hbm_gbs"], "unit": "GB/s",
           "peak_source": pk["source"],
           "bytes": "salience read + kept feature rows read and written + indices"}
    out["topk_frac"] = out["topk_gbs"] / pk["hbm_gbs"]
    out["threshold_frac"] = out["threshold_gbs"] / pk["hbm_gbs"]
    return out


# ---------------------------------------------------------------- CPU oracle

def _one_unit(shape):
    """(layer, sequence) unit shape of a decode workload: one layer, batch 1."""
    from visual_token_sparsity_gb300 import synth
    return synth.DecodeShape(shape.name, H=shape.H, Hkv=shape.Hkv, d=shape.d, n_vis=shape.n_vis,
                             n_text=shape.n_text, layers=1, batch=1, keep=shape.keep, R=shape.R, seed=shape.seed)


def _draw_unit(one, layer):
    from visual_token_sparsity_gb300 import synth
    bt = synth.random_block_table(1, one.max_blocks, one.num_blocks, seed=1, identity=True)
    lay = synth.draw_decode_layer(one, layer, bt)
    qr, qd = synth.draw_decode_queries(one, layer)
    return (lay.k_logical.double().numpy(), lay.v_logical.double().numpy(), qr.double().numpy(),
            qd.double().numpy())


def _oracle_on_unit(one, unit):
    """The oracle's retrieval + sparse attention on one drawn unit; returns seconds."""
    import oracle
    K, V, qr64, qd64 = unit
    t0 = time.perf_counter()
    idx, _ = oracle.retrieve_topk(qr64, K[:, :, :one.n_vis], one.k)
    oracle.sparse_decode_attention(qd64, K, V, idx, one.n_vis, one.n_text)
    return time.perf_counter() - t0


def oracle_sample_seconds(shape, units, seed=0):
    """Run the fp64 oracle on `units` (layer, sequence) pairs of the decode
    workload, starting at layer `seed`; returns (seconds, algorithmic bytes
    covered).  Input drawing is not timed."""
    one = _one_unit(shape)
    rb, ab = decode_bytes(one)
    total = 0.0
    for u in range(units):
        total += _oracle_on_unit(one, _draw_unit(one, seed + u))
    return total, units * (rb + ab)


def _oracle_worker(job):
    """Process-pool task: draw one unit (its own layer) and run the oracle on
    it `reps` times; returns (oracle seconds, bytes)."""
    shape, layer, reps = job
    one = _one_unit(shape)
    unit = _draw_unit(one, layer)
    rb, ab = decode_bytes(one)
    secs = sum(_oracle_on_unit(one, unit) for _ in range(reps))
    return secs, reps * (rb + ab)


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for l in out.splitlines():
            if l.strip().lower().startswith("model name"):
                return l.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


class OraclePool:
    """Spawned worker processes (one per host core, single-threaded numpy)
    that time the oracle on independent (layer, sequence) units.  Spawn, not
    fork: the parent may already hold a CUDA context."""

    def __init__(self, workers=None):
        import multiprocessing as mp
        self.n = workers or host_cores()
        self.pool = mp.get_context("spawn").Pool(self.n)

    def run(self, shape, reps, layer0=0):
        """Every worker runs `reps` oracle passes on its own unit; the job's
        time is the slowest worker's oracle time.  Returns (seconds, bytes)."""
        res = self.pool.map(_oracle_worker, [(shape, layer0 + i, reps) for i in range(self.n)], chunksize=1)
        return max(r[0] for r in res), sum(r[1] for r in res)

    def close(self):
        self.pool.close()
        self.pool.join()


def cpu_baseline(shape, budget_s=8.0, pool=None):
    """The oracle as it stands on the host cores: single-threaded on one unit
    repeated for ~budget_s, then on every core (one unit per worker, same
    number of passes per worker)."""
    one = _one_unit(shape)
    rb, ab = decode_bytes(one)
    unit = _draw_unit(one, 0)
    reps, secs = 0, 0.0
    while secs < budget_s and reps < 2000:
        secs += _oracle_on_unit(one, unit)
        reps += 1
    single = (rb + ab) * reps / secs / 1e9
    out = {"value": single, "unit": "GB/s", "cores": 1, "kind": "oracle", "cpu_model": cpu_model(),
           "host_cores": host_cores(),
           "sample": f"{reps} oracle passes over one (layer, sequence) unit of the same workload "
                     f"(retrieval + sparse attention), fp64 numpy, single thread",
           "single_thread_gbs": single}
    own = pool is None
    try:
        pool = pool or OraclePool()
        per_worker = max(1, int(reps * 0.75))
        t, nb = pool.run(shape, per_worker, layer0=1)
        out.update({"value": nb / t / 1e9, "cores": pool.n, "all_cores_gbs": nb / t / 1e9,
                    "sample": f"all cores: {pool.n} single-threaded workers x {per_worker} oracle passes over "
                              f"their own (layer, sequence) unit (retrieval + sparse attention, fp64 numpy), "
                              f"time = the slowest worker's; single thread: {reps} passes over one unit"})
    except Exception as e:   # the single-thread figure still stands
        out["all_cores_error"] = str(e)[:200]
    finally:
        if own and pool is not None:
            pool.close()
    return out


def rounds_measure(batch, steps, warmup, stream):
    """Latency of the 5-round loop on the tiny shapes: per round, evict the
    previous question/answer, append the 32-token question, retrieve the
    top-25% visual tokens with its 32 query rows, then 256 decode steps of
    (append one token, sparse attention).  Every round starts from the same
    cache state (visual tokens + 32-token prefix), so one CUDA graph of a
    round is replayed; inputs are seeded device buffers."""
    from visual_token_sparsity_gb300 import binding as sv, synth
    s = synth.multiturn(batch=batch)
    dev = torch.device("cuda", 0)
    bt = synth.random_block_table(s.batch, s.max_blocks, s.num_blocks, seed=synth.subseed(s.seed, 0, 98)).to(dev)
    lay = synth.draw_decode_layer(s, 0, bt, device=dev)
    layer = sv.KvLayer(lay.k_pool, lay.v_pool)
    B, Hkv, H, d = s.batch, s.Hkv, s.H, s.d
    ws_r = sv.workspace(sv.sv_retrieve_workspace_bytes(B, H, Hkv, d, s.n_vis, s.k), dev)
    ws_a = sv.workspace(sv.sv_attn_workspace_bytes(B, H, Hkv, d, s.k + 32 + 32 + 256), dev)
    ws_e = sv.workspace(256, dev)
    g = lambda t: synth.subseed(s.seed, 100, t)
    qk = synth.normal_bf16((B, 32, Hkv, d), g(1), device=dev)
    qv = synth.normal_bf16((B, 32, Hkv, d), g(2), device=dev)
    rows = synth.normal_bf16((B, 32, H, d), g(3), device=dev)
    ak = synth.normal_bf16((B, 256, 1, Hkv, d), g(4), device=dev)
    av = synth.normal_bf16((B, 256, 1, Hkv, d), g(5), device=dev)
    aq = synth.normal_bf16((256, B, H, d), g(6), device=dev)
    vis = torch.empty(B, Hkv, s.k, dtype=torch.int32, device=dev)
    outs = torch.empty(256, B, H, d, dtype=torch.bfloat16, device=dev)
    scale = 1.0 / math.sqrt(d)
    ak_steps = [ak[:, t].contiguous() for t in range(256)]
    av_steps = [av[:, t].contiguous() for t in range(256)]

    def one_round():
        seqs = sv.SeqBatch(bt, s.n_vis, 32 + 32 + 256)      # state after a previous round
        sv.sv_evict_qa_tokens([layer], seqs, 32, seqs.n_text, ws_e)
        sv.sv_kv_append(layer, seqs, qk, qv, ws_e)
        seqs.n_text += 32
        sv.sv_retrieve_topk(rows, layer, seqs, s.k, vis, None, ws_r)
        for t in range(256):
            sv.sv_kv_append(layer, seqs, ak_steps[t], av_steps[t], ws_e)
            seqs.n_text += 1
            sv.sv_sparse_decode_attn(aq[t], scale, layer, seqs, vis, s.k, outs[t], None, ws_a)

    # pack-once variant: after the retrieval the selected visual rows and the
    # text are packed into a second paged layer, the answer tokens are appended
    # there and every decode step attends densely over it
    n_pack = s.k + 32 + 32 + 256
    pblk = (n_pack + 15) // 16
    pbt = torch.arange(B * pblk, dtype=torch.int32, device=dev).view(B, pblk)
    pk_pool = torch.empty(B * pblk, Hkv, 16, d, dtype=torch.bfloat16, device=dev)
    player = sv.KvLayer(pk_pool, torch.empty_like(pk_pool))
    outs_p = torch.empty_like(outs)

    def one_round_packed():
        seqs = sv.SeqBatch(bt, s.n_vis, 32 + 32 + 256)
        sv.sv_evict_qa_tokens([layer], seqs, 32, seqs.n_text, ws_e)
        sv.sv_kv_append(layer, seqs, qk, qv, ws_e)
        seqs.n_text += 32
        sv.sv_retrieve_topk(rows, layer, seqs, s.k, vis, None, ws_r)
        pseqs = sv.SeqBatch(pbt, s.k, seqs.n_text)
        sv.sv_pack_kv(layer, seqs, vis, s.k, player, pseqs, ws_e)
        for t in range(256):
            sv.sv_kv_append(player, pseqs, ak_steps[t], av_steps[t], ws_e)
            pseqs.n_text += 1
            sv.sv_sparse_decode_attn(aq[t], scale, player, pseqs, None, 0, outs_p[t], None, ws_a)

    # fused variant: each decode step is one sv_decode_append_attn launch
    akf = [ak[:, t, 0].contiguous() for t in range(256)]
    avf = [av[:, t, 0].contiguous() for t in range(256)]
    outs_f = torch.empty_like(outs)

    def one_round_fused():
        seqs = sv.SeqBatch(bt, s.n_vis, 32 + 32 + 256)
        sv.sv_evict_qa_tokens([layer], seqs, 32, seqs.n_text, ws_e)
        sv.sv_kv_append(layer, seqs, qk, qv, ws_e)
        seqs.n_text += 32
        sv.sv_retrieve_topk(rows, layer, seqs, s.k, vis, None, ws_r)
        for t in range(256):
            sv.sv_decode_append_attn(aq[t], scale, layer, seqs, akf[t], avf[t], vis, s.k, outs_f[t], None, ws_a)
            seqs.n_text += 1

    graph = time_graph(one_round, steps, max(3, warmup), stream)
    ms = replay_timed(graph, steps, stream, lambda: None)
    graph_p = time_graph(one_round_packed, steps, max(3, warmup), stream)
    ms_p = replay_timed(graph_p, steps, stream, lambda: None)
    graph_f = time_graph(one_round_fused, steps, max(3, warmup), stream)
    ms_f = replay_timed(graph_f, steps, stream, lambda: None)
    del graph, graph_p, graph_f
    return {"workload": "round loop: evict, append 32-token question, retrieve top-25% with 32 rows, "
                        "256 x (append + sparse attention); 4 q / 2 KV heads, d 64, 576 visual + 32-token "
                        f"prefix, batch {s.batch}",
            "round_us": ms * 1e3, "per_decode_step_us": ms * 1e3 / 256,
            "rounds_per_s": 1e3 / ms, "gpu_launches_per_round": 1 + 1 + 256 * 2,
            "fused": {"round_us": ms_f * 1e3, "per_decode_step_us": ms_f * 1e3 / 256,
                      "gpu_launches_per_round": 1 + 1 + 256,
                      "note": "same round with each decode step's append and attention in one launch "
                              "(sv_decode_append_attn)"},
            "packed": {"round_us": ms_p * 1e3, "per_decode_step_us": ms_p * 1e3 / 256,
                       "note": "same round with the selection packed once (sv_pack_kv) and dense "
                               "attention over the packed pages"}}


def rounds_main(a):
    """The round loop as its own bench line (--workload rounds)."""
    torch.cuda.set_device(0)
    import __graft_entry__
    __graft_entry__.build()
    stream = torch.cuda.Stream()
    r = rounds_measure(a.batch, a.steps, a.warmup, stream)
    print(json.dumps({"metric": "multi-turn round latency (tiny shapes)", "value": r["round_us"],
                      "unit": "us/round", "n_gpus": 1, "steps": a.steps, "warmup": a.warmup,
                      "higher_is_better": False, "per_decode_step_us": r["per_decode_step_us"], "dtype": "bf16",
                      "data": "synthetic", "gpu_launches": a.steps * r["gpu_launches_per_round"],
                      "packed": r["packed"], "config": {"workload": r["workload"], "batch": a.batch}}))


def exp_bound(ss, ms, clocks):
    """Exp-limited bound of the salience kernel: 2*H*N^2 exps per frame (one
    per logit in each pass) at 32 ex2 results per clock per SM (measured on
    GB300), at the SM clock sampled under load (else the maximum clock)."""
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    mhz = None
    if clocks:
        mhz = clocks.get("sm_mhz") or clocks.get("sm_max_mhz")
    mhz = mhz or 2070.0
    exps = 2.0 * ss.H * ss.N * ss.N * ss.batch
    bound_ms = exps / (32.0 * props.multi_processor_count * mhz * 1e6) * 1e3
    return {"exp_bound_ms": bound_ms, "exp_frac": bound_ms / ms, "exp_bound_clock_mhz": mhz,
            "exp_count": exps}


def tiny_measure(dev, steps, stream):
    """The tiny single-layer case: one decode step (retrieval with 1 query row,
    keep 25%, then sparse attention) and the prefill salience + top-25% prune
    and compaction on the 576-token encoder shape, each as a CUDA graph."""
    from visual_token_sparsity_gb300 import binding as sv, synth
    wl = DecodeWorkload(synth.tiny_decode(), dev)
    ms, ms_attn, ms_ret = decode_graph_times(wl, steps, 3, stream, lambda: None)
    ss = synth.tiny_salience()
    q, k, feat = synth.draw_salience(ss, device=dev)
    sal = torch.empty(ss.batch, ss.N, device=dev)
    ws = sv.workspace(sv.sv_salience_workspace_bytes(ss.batch, ss.H, ss.N, ss.d), dev)
    kept = torch.empty(ss.batch, ss.k, dtype=torch.int32, device=dev)
    fout = torch.empty(ss.batch, ss.k, ss.C, dtype=torch.bfloat16, device=dev)
    sal_fn = lambda: sv.sv_salience_prefill(q, k, 1 / math.sqrt(ss.d), sal, ws)
    pre_fn = lambda: (sal_fn(), sv.sv_prune_compact(sal, ss.k, feat, fout, kept, ws))
    g_sal = time_graph(sal_fn, steps, 3, stream)
    ms_sal = replay_timed(g_sal, steps, stream, lambda: None)
    g_pre = time_graph(pre_fn, steps, 3, stream)
    ms_pre = replay_timed(g_pre, steps, stream, lambda: None)
    del g_sal, g_pre, wl
    return {"workload": "tiny: decode 4 q / 2 KV heads, d 64, 576 visual + 32 text, 1 query row, keep 25% "
                        "(k=144), batch 1; prefill 576 tokens, 4 heads, d 64, keep 25%, 256-wide features",
            "decode_step_us": ms * 1e3, "retrieve_us": ms_ret * 1e3, "attention_us": ms_attn * 1e3,
            "salience_us": ms_sal * 1e3, "prefill_salience_prune_us": ms_pre * 1e3,
            "note": "latency-bound (one small layer): microseconds only, graph replay"}


# ---------------------------------------------------------------- main

def main():
    a = parse()
    if a.batch is None:
        a.batch = {"llava": 16, "longvila": 8}.get(a.workload, 1)
    rank, world, local = dist_env()
    from visual_token_sparsity_gb300 import synth
    if a.workload == "llava":
        shape = synth.llava_next_decode(batch=a.batch, keep=a.keep, layers=a.layers or 32)
    elif a.workload == "longvila":
        shape = synth.longvila_decode(batch=a.batch, layers=a.layers or 28)
    elif a.workload == "tiny":
        shape = synth.tiny_decode(batch=a.batch)
    else:
        return rounds_main(a)
    config = {"workload": f"{shape.name}: {shape.layers} layers, batch {shape.batch}, {shape.H} query heads / "
                          f"{shape.Hkv} KV heads, d {shape.d}, "
                          f"{shape.n_vis} visual + {shape.n_text} text tokens, page 16, retrieval keep {shape.keep} "
                          f"(k={shape.k}), 1 query row",
              "global_batch": shape.batch * world, "layers": shape.layers, "keep": shape.keep,
              "parallelism": f"replicas x{world}",
              "l2": "inputs larger than L2 (KV cache %.1f GB per replica)" % (
                  shape.layers * 2 * shape.num_blocks * shape.Hkv * 16 * shape.d * 2 / 1e9)}

    if a.impl == "reference":
        if rank != 0:
            return
        # the oracle on every host core: each step, every worker runs the
        # oracle once on its own (layer, sequence) unit; the step's time is
        # the slowest worker's
        pool = OraclePool()
        try:
            for i in range(a.warmup):
                pool.run(shape, 1, layer0=i * pool.n)
            t, nb = 0.0, 0
            for i in range(a.steps):
                dt, b = pool.run(shape, 1, layer0=(a.warmup + i) * pool.n)
                t += dt
                nb += b
        finally:
            pool.close()
        v = nb / t / 1e9
        print(json.dumps({"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": a.gpus,
                          "steps": a.steps, "warmup": a.warmup, "ms_per_step": t / a.steps * 1e3,
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                          "data": "synthetic", "config": config,
                          "cpu_baseline": {"value": v, "unit": "GB/s", "cores": pool.n, "kind": "oracle",
                                           "cpu_model": cpu_model(),
                                           "sample": f"each step: {pool.n} single-threaded workers each run the "
                                                     "oracle (retrieval + sparse attention, fp64 numpy) on their "
                                                     "own (layer, sequence) unit of the workload"},
                          "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))
        return

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
        torch.cuda.set_device(local)
        barrier = lambda: dist.barrier(device_ids=[local])
    else:
        torch.cuda.set_device(0)
        barrier = lambda: None
    dev = torch.device("cuda", torch.cuda.current_device())

    import __graft_entry__
    __graft_entry__.build()
    pk = peaks()

    stream = torch.cuda.Stream()
    line = {"metric": METRIC, "value": None, "unit": "GB/s", "n_gpus": world, "steps": a.steps,
            "warmup": a.warmup, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic (seeded N(0,1) K/V with 2% x4 outliers, random page tables)",
            "config": config}
    if not a.no_decode:
        decode_measure(a, shape, dev, stream, barrier, world, pk, line)
    extra_steps = min(50, max(3, a.steps // 2))
    if not a.no_decode and not a.no_extra and a.workload == "llava":
        # the other decode workloads as objects of the same line
        lv = {}
        for b in (8, 1):
            lv[f"b{b}"] = decode_object(synth.longvila_decode(batch=b), dev, extra_steps, 3, stream, pk)
        # a short video on the same model: 16 frames (3136 visual tokens), batch 16
        lv["b16_f16"] = decode_object(synth.longvila_decode(batch=16, frames=16), dev, extra_steps, 3, stream, pk)
        line["longvila"] = lv
        # the other LLaVA-NeXT-7B cases: 25% keep at batch 16, batches 4 and 1
        ln = {"b16_keep0.25": decode_object(synth.llava_next_decode(batch=16, keep=0.25), dev, extra_steps, 3,
                                            stream, pk)}
        for b in (4, 1):
            ln[f"b{b}_keep0.5"] = decode_object(synth.llava_next_decode(batch=b, keep=0.5), dev, extra_steps, 3,
                                                stream, pk)
        line["llava_next"] = ln
        line["tiny"] = tiny_measure(dev, extra_steps, stream)
        line["rounds"] = rounds_measure(1, max(3, extra_steps // 4), 3, stream)
    if not a.no_salience:
        tiny = a.workload == "tiny"
        ss, sms, flops = salience_measure(1 if tiny else a.salience_batch, extra_steps, 3, stream, tiny=tiny)
        tf = flops / (sms * 1e-3) / 1e12
        line["salience"] = {"workload": f"{ss.name}: {ss.batch} frames x {ss.N} tokens, {ss.H} heads, d {ss.d}",
                            "ms": sms, "tokens_per_s": ss.batch * ss.N / (sms * 1e-3),
                            "tflops": tf, "bound": "tensor", "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                            "frac": tf / pk["bf16_tflops"], "peak_source": pk["source"],
                            "flop_count": "4*H*N^2*d per frame (both QK^T passes, d unpadded)",
                            **exp_bound(ss, sms, line.get("clocks"))}
    if not a.no_salience and a.workload != "tiny" and a.salience_long_n > 0:
        # long visual sequence: both operands streamed through 128 x 256 tiles
        from visual_token_sparsity_gb300 import binding as sv
        ls = synth.qwen2vl_salience(N=a.salience_long_n)
        ls_, lms, lflops = salience_measure(1, max(3, extra_steps // 4), 3, stream, shape=ls)
        ltf = lflops / (lms * 1e-3) / 1e12
        line["salience_long"] = {
            "workload": f"{ls.name}: {ls.batch} x {ls.N} tokens, {ls.H} heads, d {ls.d}",
            "ms": lms, "tokens_per_s": ls.batch * ls.N / (lms * 1e-3), "tflops": ltf, "bound": "tensor",
            "peak": pk["bf16_tflops"], "unit": "TFLOP/s", "frac": ltf / pk["bf16_tflops"],
            "peak_source": pk["source"], "kernels_per_call": sv.sv_salience_kernel_count(ls.N, ls.d),
            "flop_count": "4*H*N^2*d (both QK^T passes, d unpadded)", **exp_bound(ls, lms, line.get("clocks"))}
        torch.cuda.empty_cache()
    if not a.no_salience and a.workload != "tiny":
        line["prune"] = prune_measure(a.salience_batch, extra_steps, stream, pk)
        torch.cuda.empty_cache()
        cs = synth.clip_summary_salience(batch=a.salience_batch)
        us, nbytes = summary_salience_measure(cs, extra_steps, stream)
        gbs = nbytes / (us * 1e-6) / 1e9
        line["salience_summary"] = {
            "workload": f"{cs.name}: {cs.batch} frames x {cs.N} tokens, {cs.H} heads, d {cs.d}, 1 summary row",
            "us": us, "gbs": gbs, "bound": "hbm", "peak": pk["hbm_gbs"], "unit": "GB/s",
            "frac": gbs / pk["hbm_gbs"], "peak_source": pk["source"],
            "bytes": "K once + the summary rows of Q + the fp32 salience"}
    if rank == 0:
        if world == 1 and not a.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(shape)
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def launches_per_layer(shape):
    """Kernels one layer of the decode step launches (retrieval + attention)."""
    from visual_token_sparsity_gb300 import binding as sv
    return (sv.sv_retrieve_kernel_count(shape.batch, shape.Hkv, shape.n_vis) +
            sv.sv_attn_kernel_count(shape.batch, shape.H, shape.Hkv, shape.k + shape.n_text))


def roofline_of(shape, ms_attn, ms_ret, pk, with_traffic=True):
    """Roofline record of the dominant C call of a decode step.  The time per
    launch is the single-call graph's step time / layers (graph replay over
    all layers, inputs larger than L2); algorithmic bytes per launch follow
    decode_bytes()."""
    rb, ab = decode_bytes(shape)
    t_ret, t_att = ms_ret / shape.layers, ms_attn / shape.layers
    per_launch_ret, per_launch_att = rb / shape.layers, ab / shape.layers
    if t_att >= t_ret:
        dom = ("sv_sparse_decode_attn (split-K gather attention + combine)", per_launch_att, t_att, "attention")
    else:
        dom = ("sv_retrieve_topk (paged GEMV + radix top-k)", per_launch_ret, t_ret, "retrieve")
    achieved = dom[1] / (dom[2] * 1e-3) / 1e9
    return {"kernel": dom[0], "bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"],
            "unit": "GB/s", "frac": achieved / pk["hbm_gbs"], "peak_source": pk["source"],
            "traffic": (measured_traffic(f"{dom[3]}:{shape.name}:b{shape.batch}:keep{shape.keep}")
                        if with_traffic else None),
            "algorithmic_bytes_per_launch": dom[1],
            "timing": "graph replay of the call over all layers / layers",
            "per_call_us": {"retrieve": t_ret * 1e3, "attention": t_att * 1e3},
            "per_call_gbs": {"retrieve": per_launch_ret / (t_ret * 1e-3) / 1e9,
                             "attention": per_launch_att / (t_att * 1e-3) / 1e9}}


def decode_object(shape, dev, steps, warmup, stream, pk):
    """Step figures of one more decode workload (its own cache, all layers)."""
    rb, ab = decode_bytes(shape)
    wl = DecodeWorkload(shape, dev)
    ms, ms_attn, ms_ret = decode_graph_times(wl, steps, warmup, stream, lambda: None)
    gbs = (rb + ab) / (ms * 1e-3) / 1e9
    out = {"workload": f"{shape.name}: {shape.layers} layers, batch {shape.batch}, {shape.H} q / {shape.Hkv} KV "
                       f"heads, d {shape.d}, {shape.n_vis} visual + {shape.n_text} text, keep {shape.keep} "
                       f"(k={shape.k}), 1 query row",
           "decode_step_us": ms * 1e3, "attn_only_step_us": ms_attn * 1e3, "retrieve_only_step_us": ms_ret * 1e3,
           "gbs": gbs, "frac": gbs / pk["hbm_gbs"], "peak": pk["hbm_gbs"], "peak_source": pk["source"],
           "attn_only_gbs": ab / (ms_attn * 1e-3) / 1e9,
           "gpu_launches_per_step": shape.layers * launches_per_layer(shape),
           "roofline": roofline_of(shape, ms_attn, ms_ret, pk)}
    del wl
    torch.cuda.empty_cache()
    return out


def decode_measure(a, shape, dev, stream, barrier, world, pk, line):
    rb, ab = decode_bytes(shape)
    bytes_step = rb + ab
    wl = DecodeWorkload(shape, dev)
    clk = ClockSampler(torch.cuda.current_device())
    ms, ms_attn, ms_ret = decode_graph_times(wl, a.steps, a.warmup, stream, barrier, clocks=clk)
    (ms, ms_attn, ms_ret), value = aggregate_replicas([ms, ms_attn, ms_ret], bytes_step, world,
                                                      torch_max_reducer(dev) if world > 1 else None)
    line.update({"value": value, "ms_per_step": ms, "decode_step_us": ms * 1e3,
                 "attn_only_step_us": ms_attn * 1e3, "retrieve_only_step_us": ms_ret * 1e3,
                 "clocks": clk.summary(),
                 # per layer: retrieval (+ a separate top-k for long rows) and
                 # attention (+ a merge kernel for many splits), as the library reports
                 "gpu_launches": a.steps * shape.layers * launches_per_layer(shape),
                 "roofline": roofline_of(shape, ms_attn, ms_ret, pk, with_traffic=world == 1),
                 "hbm_frac_step": (bytes_step / (ms * 1e-3) / 1e9) / pk["hbm_gbs"]})

    if not a.no_e2e:
        e2e, h2d, d2h = e2e_throughput(wl, min(50, max(3, a.steps // 2)), 2, stream, bytes_step)
        line["e2e"] = {"value": world * e2e, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
    if not a.no_packed:
        # pack-once KV (round reuse): the selected rows of every layer are
        # packed once per round, then each decode step attends densely
        wl.make_packed()
        g_pack = time_graph(wl.pack_all, a.steps, 3, stream)
        g_dense = time_graph(wl.attn_packed_step, a.steps, 3, stream)
        ms_pack = replay_timed(g_pack, a.steps, stream, barrier)
        ms_dense = replay_timed(g_dense, a.steps, stream, barrier)
        line["packed"] = {
            "attn_only_step_us": ms_dense * 1e3, "gather_attn_only_step_us": ms_attn * 1e3,
            "attention_gbs": ab / (ms_dense * 1e-3) / 1e9, "gather_attention_gbs": ab / (ms_attn * 1e-3) / 1e9,
            "pack_all_layers_us": ms_pack * 1e3,
            "step_us_amortized_256": (ms_dense + ms_pack / 256) * 1e3,
            "note": "attention over the retrieval's selection; pack once per round (all layers), "
                    "then dense attention over the packed pages each decode step"}
        del g_pack, g_dense
    if not a.no_packed:
        # softmax-normalised retrieval for a 32-row question (once per round)
        from visual_token_sparsity_gb300 import binding as sv, synth
        s = shape
        R = 32
        q32 = synth.normal_bf16((s.batch, R, s.H, s.d), synth.subseed(s.seed, 200, 1), device=dev)
        lse32 = torch.zeros(s.batch, R, s.H, device=dev)
        ws_s = sv.workspace(sv.sv_retrieve_softmax_workspace_bytes(s.batch, R, s.H, s.Hkv, s.d, s.n_vis, s.n_text), dev)
        ws_d = sv.workspace(sv.sv_retrieve_workspace_bytes(s.batch, s.H, s.Hkv, s.d, s.n_vis, s.k), dev)
        vis_s = torch.empty(s.batch, s.Hkv, s.k, dtype=torch.int32, device=dev)
        soft = lambda: [sv.sv_retrieve_topk_softmax(q32, wl.scale, wl.layers[l], wl.seqs, s.k, vis_s, None, ws_s)
                        for l in range(s.layers)]
        fused = lambda: [sv.sv_retrieve_topk_softmax(q32, wl.scale, wl.layers[l], wl.seqs, s.k, vis_s, None, ws_s,
                                                     lse=lse32) for l in range(s.layers)]
        dot = lambda: [sv.sv_retrieve_topk(q32, wl.layers[l], wl.seqs, s.k, vis_s, None, ws_d) for l in range(s.layers)]
        res = {}
        for name, fn in (("softmax_us_per_layer", soft), ("softmax_given_lse_us_per_layer", fused),
                         ("dot_us_per_layer", dot)):
            g = time_graph(fn, max(3, a.steps // 4), 3, stream)
            res[name] = replay_timed(g, max(3, a.steps // 4), stream, barrier) * 1e3 / s.layers
            del g
        kv = s.batch * s.Hkv * s.d * 2
        res["question_rows"] = R
        res["softmax_gbs"] = kv * (2 * s.n_vis + s.n_text) / (res["softmax_us_per_layer"] * 1e-6) / 1e9
        res["note"] = ("per layer, once per round: the question's 32 rows score the visual tokens by attention "
                       "mass (two passes over K, or one with the caller's prefill lse) vs the dot product")
        line["retrieval_softmax"] = res
    if not a.no_varlen:
        # per-sequence lengths: the same cache read as a threshold-pruned
        # batch, each sequence with its own visual, text and selected counts
        from visual_token_sparsity_gb300 import binding as sv
        nv, nt, kk = varlen_counts(shape)
        arr = lambda x: torch.tensor(x, dtype=torch.int32, device=dev)
        uniform = wl.seqs
        wl.seqs = sv.SeqBatch(wl.bt, shape.n_vis, shape.n_text, arr(nv), arr(nt), arr(kk))
        g_vl = time_graph(wl.step, a.steps, 3, stream)
        ms_vl = replay_timed(g_vl, a.steps, stream, barrier)
        wl.seqs = uniform
        gbs = varlen_bytes(shape, nv, nt, kk) / (ms_vl * 1e-3) / 1e9
        line["variable_lengths"] = {
            "step_us": ms_vl * 1e3, "gbs": gbs, "frac": gbs / pk["hbm_gbs"], "peak_source": pk["source"],
            "n_vis_range": [min(nv), max(nv)], "n_text_range": [min(nt), max(nt)], "k_range": [min(kk), max(kk)],
            "tokens_vs_uniform": (sum(nv) + sum(nt)) / (shape.batch * (shape.n_vis + shape.n_text)),
            "note": "retrieval + sparse attention per layer with per-sequence counts (sv_seq_batch n_vis_seq / "
                    "n_text_seq / k_seq); GB/s of the per-sequence algorithmic bytes"}
        del g_vl
    del wl
    torch.cuda.empty_cache()


if __name__ == "__main__":
    main()
