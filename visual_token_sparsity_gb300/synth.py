"""Seeded synthetic inputs shaped like the SparseVILA workloads.

This module draws random tensors and lays them out; it holds none of the
method's arithmetic.  Both the CUDA path and the fp64 oracle are fed from the
same tensors drawn here.

Recipe (stand-ins for the LLaVA-NeXT-7B, LongVILA-7B and SigLIP workloads named
on the SparseVILA pages; no dataset or weights are used):

* entries are drawn as fp32 normals from a seeded ``torch.Generator`` and
  rounded to bf16;
* ``round(0.02 * n_vis)`` (half rounded up) visual positions, drawn by a seeded
  permutation and shared by all heads, are salient outliers whose rows are
  multiplied by 4 (keys, and values where the workload says "K,V");
* block tables are a seeded random permutation of the page pool.
"""

from dataclasses import dataclass, field
import math

import torch

BLOCK_TOKENS = 16


def generator(seed, device="cpu"):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal_bf16(shape, seed, std=1.0, device="cpu"):
    """bf16 tensor of N(0, std^2) entries drawn in fp32 from ``seed``."""
    x = torch.randn(*shape, generator=generator(seed, device), device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def n_outliers(n_vis, frac=0.02):
    """Outlier count: frac * n_vis rounded half up (576 -> 12, 729 -> 15)."""
    return int(math.floor(frac * n_vis + 0.5))


def outlier_positions(n_vis, seed, frac=0.02):
    perm = torch.randperm(n_vis, generator=generator(seed))
    return torch.sort(perm[: n_outliers(n_vis, frac)]).values


def scale_token_rows(x, positions, factor, token_dim):
    """Multiply the rows at ``positions`` along ``token_dim`` by ``factor`` (in place)."""
    if positions.numel() == 0:
        return x
    idx = positions.to(x.device)
    sub = x.index_select(token_dim, idx).float() * factor
    x.index_copy_(token_dim, idx, sub.to(x.dtype))
    return x


def blocks_for(n_tokens):
    return (n_tokens + BLOCK_TOKENS - 1) // BLOCK_TOKENS


def random_block_table(batch, max_blocks, num_blocks, seed, identity=False):
    """[batch][max_blocks] int32 table of distinct pool blocks."""
    assert batch * max_blocks <= num_blocks
    if identity:
        ids = torch.arange(batch * max_blocks, dtype=torch.int64)
    else:
        ids = torch.randperm(num_blocks, generator=generator(seed))[: batch * max_blocks]
    return ids.reshape(batch, max_blocks).to(torch.int32)


def scatter_to_pool(x, block_table, num_blocks):
    """Lay a logical [B][Hkv][n][d] tensor out as a paged pool.

    Token t of sequence b goes to row t % 16 of block block_table[b, t // 16];
    the pool is [num_blocks][Hkv][16][d].  Unused rows are zero.
    """
    B, Hkv, n, d = x.shape
    nb = blocks_for(n)
    pad = nb * BLOCK_TOKENS - n
    if pad:
        x = torch.cat([x, x.new_zeros(B, Hkv, pad, d)], dim=2)
    pool = x.new_zeros(num_blocks, Hkv, BLOCK_TOKENS, d)
    blocks = x.reshape(B, Hkv, nb, BLOCK_TOKENS, d).permute(0, 2, 1, 3, 4)  # [B][nb][Hkv][16][d]
    ids = block_table[:, :nb].to(torch.int64).to(x.device)
    pool[ids.reshape(-1)] = blocks.reshape(B * nb, Hkv, BLOCK_TOKENS, d)
    return pool


# --------------------------------------------------------------------------
# Workload shapes


@dataclass
class DecodeShape:
    """Decode-side workload: paged visual+text cache and retrieval/attention."""
    name: str
    H: int
    Hkv: int
    d: int
    n_vis: int
    n_text: int
    layers: int
    batch: int
    keep: float
    R: int = 1
    v_outliers: bool = True
    seed: int = 0
    extra_blocks: int = 0

    @property
    def k(self):
        return int(math.floor(self.keep * self.n_vis))

    @property
    def n_tokens(self):
        return self.n_vis + self.n_text

    @property
    def max_blocks(self):
        return blocks_for(self.n_tokens) + self.extra_blocks

    @property
    def num_blocks(self):
        return self.batch * self.max_blocks


@dataclass
class SalienceShape:
    """Prefill-side workload: encoder Q/K, salience, prune and compaction."""
    name: str
    H: int
    N: int
    d: int
    batch: int
    keep: float
    C: int
    std: float = 1.0
    seed: int = 0

    @property
    def k(self):
        return int(math.floor(self.keep * self.N))


def tiny_decode(batch=1):
    """4 query heads, 2 KV heads, d 64; 576 visual + 32 text tokens; keep 25%."""
    return DecodeShape("tiny-decode", H=4, Hkv=2, d=64, n_vis=576, n_text=32, layers=1,
                       batch=batch, keep=0.25, R=1, v_outliers=True, seed=0)


def tiny_salience(batch=1):
    """576 encoder tokens, 4 heads, d 64, keep 25%, 256-wide bf16 features."""
    return SalienceShape("tiny-salience", H=4, N=576, d=64, batch=batch, keep=0.25, C=256,
                         std=1.0, seed=0)


def llava_next_decode(batch=16, keep=0.5, layers=32):
    """Llama-2-7B attention (32 MHA heads, d 128), 2880 visual (5x576) + 128 text."""
    return DecodeShape("llava-next-7b-decode", H=32, Hkv=32, d=128, n_vis=2880, n_text=128,
                       layers=layers, batch=batch, keep=keep, R=1, v_outliers=True, seed=1)


def siglip_salience(batch=256, keep=0.25):
    """SigLIP-so400m encoder: 729 tokens, 16 heads, d 72, 1152-wide features."""
    return SalienceShape("siglip-so400m-salience", H=16, N=729, d=72, batch=batch, keep=keep,
                         C=1152, std=1.0 / math.sqrt(72.0), seed=2)


def clip_summary_salience(batch=256, keep=0.25):
    """CLIP ViT-L/14-336 encoder: 577 tokens (CLS + 24 x 24 patches), 16 heads,
    d 64, 1024-wide features; salience from the CLS row (one summary token)."""
    return SalienceShape("clip-vit-l-336-summary-salience", H=16, N=577, d=64, batch=batch, keep=keep,
                         C=1024, std=1.0 / math.sqrt(64.0), seed=6)


def qwen2vl_salience(batch=1, N=16384, keep=0.25):
    """Qwen2-VL vision tower (16 heads, d 80) over a long visual sequence:
    N patch tokens of one high-resolution image or video clip; Q, K drawn
    like the SigLIP frames (std 1/sqrt(d), 2% key outliers x4)."""
    return SalienceShape("qwen2-vl-vision-salience", H=16, N=N, d=80, batch=batch, keep=keep, C=1280,
                         std=1.0 / math.sqrt(80.0), seed=7)


def longvila_decode(batch=1, layers=28, frames=256):
    """Qwen2-7B attention (28 q heads, 4 KV heads, d 128), frames x 196 visual
    (256 frames: 50176) + 256 text."""
    return DecodeShape("longvila-7b-decode", H=28, Hkv=4, d=128, n_vis=196 * frames, n_text=256,
                       layers=layers, batch=batch, keep=0.25, R=1, v_outliers=False, seed=3)


def multiturn(batch=1):
    """Tiny-decode shapes driven through 5 question/answer rounds."""
    s = tiny_decode(batch)
    s.name = "multiturn-round-loop"
    s.seed = 4
    s.R = 32
    # room for the persistent 32-token prefix + 32 question + 256 answer tokens
    s.extra_blocks = blocks_for(576 + 32 + 32 + 256) - blocks_for(576 + 32)
    return s


# --------------------------------------------------------------------------
# Tensor draws


@dataclass
class DecodeLayer:
    """One layer's logical cache and paged pools (bf16)."""
    k_logical: torch.Tensor      # [B][Hkv][n_tokens][d]
    v_logical: torch.Tensor
    k_pool: torch.Tensor         # [num_blocks][Hkv][16][d]
    v_pool: torch.Tensor


def subseed(seed, layer, tensor_id):
    return seed * 1_000_000 + layer * 1_000 + tensor_id


def draw_decode_layer(shape: DecodeShape, layer, block_table, device="cpu"):
    B, Hkv, n, d = shape.batch, shape.Hkv, shape.n_tokens, shape.d
    k = normal_bf16((B, Hkv, n, d), subseed(shape.seed, layer, 1), device=device)
    v = normal_bf16((B, Hkv, n, d), subseed(shape.seed, layer, 2), device=device)
    pos = outlier_positions(shape.n_vis, subseed(shape.seed, layer, 3))
    scale_token_rows(k, pos, 4.0, token_dim=2)
    if shape.v_outliers:
        scale_token_rows(v, pos, 4.0, token_dim=2)
    kp = scatter_to_pool(k, block_table, shape.num_blocks)
    vp = scatter_to_pool(v, block_table, shape.num_blocks)
    return DecodeLayer(k, v, kp, vp)


def draw_decode_queries(shape: DecodeShape, layer, device="cpu", rows=None, step=0):
    """Retrieval rows [B][R][H][d] and the decode query [B][H][d]."""
    R = shape.R if rows is None else rows
    qr = normal_bf16((shape.batch, R, shape.H, shape.d), subseed(shape.seed, layer, 10 + 2 * step),
                     device=device)
    qd = normal_bf16((shape.batch, shape.H, shape.d), subseed(shape.seed, layer, 11 + 2 * step),
                     device=device)
    return qr, qd


def draw_salience(shape: SalienceShape, device="cpu"):
    """Encoder Q, K [B][H][N][d] and token features [B][N][C] (bf16)."""
    B, H, N, d = shape.batch, shape.H, shape.N, shape.d
    q = normal_bf16((B, H, N, d), subseed(shape.seed, 0, 1), std=shape.std, device=device)
    k = normal_bf16((B, H, N, d), subseed(shape.seed, 0, 2), std=shape.std, device=device)
    pos = outlier_positions(N, subseed(shape.seed, 0, 3))
    scale_token_rows(k, pos, 4.0, token_dim=2)
    feat = normal_bf16((B, N, shape.C), subseed(shape.seed, 0, 4), device=device)
    return q, k, feat
