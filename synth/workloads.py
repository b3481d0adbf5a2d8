"""Seeded synthetic workloads with the shapes and value distributions of the
five absorbed-MLA decode configurations.

Everything here is input preparation: random draws (numpy PCG64, float64 →
float32), storage casts done by torch (`.to(torch.bfloat16)`,
`.to(torch.float8_e4m3fn)`), paged-cache placement and block tables.  No
attention, projection, merge or quantisation step of the method lives here.

Layouts (all row-major, contiguous):
  cache        [num_blocks, 64, 576]  kv_c in cols 0..511, k_pe in 512..575
  block_table  [B, max_blocks] int32, -1 in unused entries
  seq_lens     [B] int32
  q            [B, q_len, H, 576]
  q_nope       [B*q_len, H, 128],  q_pe [B*q_len, H, 64]
  w_uk_t       [H, 128, 512]  (nope dim p, latent dim l; l contiguous)
  w_uv         [H, 128, 512]  (value dim v, latent dim l; l contiguous)
  w_kvb        [H*256, 512]   rows h*256+[0,128) = per-head W_UK, rows
                              h*256+[128,256) = per-head W_UV (nn.Linear
                              layout: out_features x in_features)
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

BLOCK = 64          # tokens per cache page
KV_LORA = 512       # latent rank L
ROPE = 64           # rope width R
QK_NOPE = 128       # per-head nope width P
V_HEAD = 128        # per-head value width V
D_QK = KV_LORA + ROPE  # 576, the MQA query / key width

__all__ = [
    "BLOCK", "KV_LORA", "ROPE", "QK_NOPE", "V_HEAD", "D_QK",
    "generator", "as_bf16", "as_e4m3", "paged_layout", "fill_cache",
    "DecodeCase", "PrefillCase", "decode_case", "prefill_case",
    "tiny_decode", "dsv3_decode", "long_request", "fp8_decode", "spec_decode",
    "context_prefill", "even_shards", "shard_cache_interleaved",
    "BF16_NAN_BITS", "E4M3_NAN_BITS",
]

BF16_NAN_BITS = 0x7FC0
E4M3_NAN_BITS = 0x7F


def generator(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def as_bf16(x: np.ndarray) -> torch.Tensor:
    """Store float values as bf16 (torch's round-to-nearest-even cast)."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


def as_e4m3(x: np.ndarray) -> torch.Tensor:
    """Store float values as OCP e4m3 (torch's float8_e4m3fn cast).

    Values are clipped to the finite range first because torch's cast turns
    magnitudes >= 480 into NaN instead of saturating."""
    x = np.clip(np.ascontiguousarray(x, dtype=np.float32), -448.0, 448.0)
    return torch.from_numpy(x).to(torch.float8_e4m3fn)


def _normal(g: np.random.Generator, shape, std: float) -> np.ndarray:
    out = g.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        out *= np.float32(std)
    return out


def paged_layout(g: np.random.Generator, seq_lens, spare_frac: float = 0.05,
                 min_max_blocks: int = 1):
    """Random physical placement of each request's pages.

    Returns (block_table [B, max_blocks] int32 with -1 padding, num_blocks).
    The pool holds exactly the pages needed plus ``spare_frac`` unused
    blocks; physical ids are a random permutation of the pool."""
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    pages = (seq_lens + BLOCK - 1) // BLOCK
    total = int(pages.sum())
    spare = max(1, int(math.ceil(spare_frac * total)))
    num_blocks = total + spare
    max_blocks = max(int(pages.max()) if len(pages) else 0, min_max_blocks)
    perm = g.permutation(num_blocks).astype(np.int32)
    bt = np.full((len(seq_lens), max_blocks), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(pages):
        bt[b, :n] = perm[off:off + n]
        off += int(n)
    return bt, num_blocks


def _poison_rows(block_table, seq_lens, num_blocks):
    """Boolean mask [num_blocks, 64] of cache rows no request owns."""
    owned = np.zeros((num_blocks, BLOCK), dtype=bool)
    for b, n in enumerate(seq_lens):
        n = int(n)
        for p in range((n + BLOCK - 1) // BLOCK):
            rows = min(BLOCK, n - p * BLOCK)
            owned[block_table[b, p], :rows] = True
    return ~owned


def fill_cache(g, block_table, seq_lens, num_blocks, *, std_c=1.0, std_pe=1.0,
               kv_dtype="bf16", poison=False):
    """Draw the paged latent cache.

    kv_c ~ N(0, std_c^2) in cols 0..511, k_pe ~ N(0, std_pe^2) in 512..575.
    For ``kv_dtype == "e4m3"`` the per-tensor scale is amax/448 and the
    stored code is the torch e4m3 cast of value/scale.  With ``poison`` every
    row that no request owns (page tails, spare blocks) is set to NaN bits,
    so a kernel that reads past seq_len shows it.

    Returns (cache tensor [num_blocks, 64, 576], k_scale float)."""
    vals = np.empty((num_blocks, BLOCK, D_QK), dtype=np.float32)
    vals[..., :KV_LORA] = _normal(g, (num_blocks, BLOCK, KV_LORA), std_c)
    vals[..., KV_LORA:] = _normal(g, (num_blocks, BLOCK, ROPE), std_pe)
    if kv_dtype == "bf16":
        cache, k_scale = as_bf16(vals), 1.0
    elif kv_dtype == "e4m3":
        amax = float(np.abs(vals).max())
        k_scale = float(np.float32(amax / 448.0))
        cache = as_e4m3(vals / np.float32(k_scale))
    else:
        raise ValueError(kv_dtype)
    if poison:
        mask = torch.from_numpy(_poison_rows(block_table, seq_lens, num_blocks))
        if kv_dtype == "bf16":
            cache.view(torch.int16)[mask] = BF16_NAN_BITS
        else:
            cache.view(torch.uint8)[mask] = E4M3_NAN_BITS
    return cache, k_scale


def even_shards(length: int, n: int):
    """Contiguous ceil-sized token ranges [s*c, min(L,(s+1)*c)) for s < n."""
    c = -(-length // n) if n else 0
    return [(min(length, s * c), min(length, (s + 1) * c)) for s in range(n)]


@dataclass
class DecodeCase:
    name: str
    B: int
    q_len: int
    H: int
    seq_lens: np.ndarray            # [B] int32
    block_table: np.ndarray         # [B, max_blocks] int32
    num_blocks: int
    cache: torch.Tensor             # [num_blocks, 64, 576] bf16 | float8_e4m3fn
    k_scale: float
    kv_dtype: str
    q: torch.Tensor                 # [B, q_len, H, 576] bf16 | float8_e4m3fn
    q_scale: float
    q_dtype: str
    sm_scale: float
    causal: bool
    q_nope: torch.Tensor            # [B*q_len, H, 128] bf16
    q_pe: torch.Tensor              # [B*q_len, H, 64] bf16
    w_uk_t: torch.Tensor            # [H, 128, 512] bf16
    w_uv: torch.Tensor              # [H, 128, 512] bf16
    shards: list = field(default_factory=list)   # per request: [(start, end)]


def decode_case(name, seed, *, B, H, seq_lens, q_len=1, kv_dtype="bf16",
                q_dtype=None, q_std=1.0, kv_std_c=1.0, kv_std_pe=1.0,
                nope_std=1.0, pe_std=1.0, w_uk_std=0.02, w_uv_std=0.02,
                sm_scale=1.0 / math.sqrt(QK_NOPE + ROPE), causal=True,
                n_shards=0, poison=False, spare_frac=0.05):
    g = generator(seed)
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    bt, nb = paged_layout(g, seq_lens, spare_frac=spare_frac)
    cache, k_scale = fill_cache(g, bt, seq_lens, nb, std_c=kv_std_c,
                                std_pe=kv_std_pe, kv_dtype=kv_dtype, poison=poison)
    q_dtype = q_dtype or kv_dtype
    qv = _normal(g, (B, q_len, H, D_QK), q_std)
    if q_dtype == "bf16":
        q, q_scale = as_bf16(qv), 1.0
    else:
        q_scale = float(np.float32(float(np.abs(qv).max()) / 448.0))
        q = as_e4m3(qv / np.float32(q_scale))
    T = B * q_len
    q_nope = as_bf16(_normal(g, (T, H, QK_NOPE), nope_std))
    q_pe = as_bf16(_normal(g, (T, H, ROPE), pe_std))
    w_uk_t = as_bf16(_normal(g, (H, QK_NOPE, KV_LORA), w_uk_std))
    w_uv = as_bf16(_normal(g, (H, V_HEAD, KV_LORA), w_uv_std))
    shards = [even_shards(int(n), n_shards) for n in seq_lens] if n_shards else []
    return DecodeCase(name, B, q_len, H, seq_lens, bt, nb, cache, k_scale, kv_dtype,
                      q, q_scale, q_dtype, sm_scale, causal, q_nope, q_pe,
                      w_uk_t, w_uv, shards)


def tiny_decode(poison=True):
    """Tiny: B=2, H=16, ctx 37 and 130, 2 shards, N(0,1)/sqrt(dim) values."""
    return decode_case(
        "tiny_b2_h16_ctx37_130", 1001, B=2, H=16, seq_lens=[37, 130],
        q_std=1.0 / math.sqrt(192), kv_std_c=1.0 / math.sqrt(512),
        kv_std_pe=1.0 / math.sqrt(64), nope_std=1.0 / math.sqrt(192),
        pe_std=1.0 / math.sqrt(192), w_uk_std=1.0 / math.sqrt(128),
        w_uv_std=1.0 / math.sqrt(512), n_shards=2, poison=poison)


def dsv3_decode(poison=False, B=32, ctx=4096):
    """DeepSeek-V3 decode shape: B=32, H=128, ctx 4096, cache N(0,1)."""
    return decode_case("dsv3_b32_h128_ctx4096", 1002, B=B, H=128,
                       seq_lens=[ctx] * B, poison=poison)


def long_request(poison=False, ctx=131072):
    """Long single request: ctx 131072, 8 equal shards then a merge."""
    return decode_case("long_b1_h128_ctx131072", 1003, B=1, H=128,
                       seq_lens=[ctx], n_shards=8, poison=poison)


def fp8_decode(poison=False, B=64, lo=1024, hi=16384):
    """FP8 KV: B=64, ctx ~ U[1024,16384], e4m3 cache and query."""
    g = generator(2004)
    lens = g.integers(lo, hi, size=B, endpoint=True)
    return decode_case("fp8_b64_h128_ctxU1k_16k", 1004, B=B, H=128,
                       seq_lens=lens, kv_dtype="e4m3", q_dtype="e4m3",
                       poison=poison)


def lognormal_lengths(g, n, median=2048.0, sigma=1.0, lo=2, hi=32768):
    x = np.rint(np.exp(math.log(median) + sigma * g.standard_normal(n)))
    return np.clip(x, lo, hi).astype(np.int32)


def spec_decode(poison=False, B=128):
    """Speculative decode: B=128, q_len=2 causal, ctx lognormal(ln 2048, 1)."""
    lens = lognormal_lengths(generator(2005), B)
    return decode_case("spec_b128_q2_h128_lognormal", 1005, B=B, H=128,
                       seq_lens=lens, q_len=2, poison=poison)


def shard_cache_interleaved(g, cache: torch.Tensor, block_table, ctx_lens, W: int,
                            interleave: int = 1, spare_frac=0.05):
    """Place a global paged cache onto W simulated DCP shards.

    Token t of request r lives on shard k = (t // I) % W at local index
    j = (t // (I*W)) * I + t % I.  Each shard gets its own randomly permuted
    block pool and block table.  Returns a list of
    (shard_cache, shard_block_table [B, mb] int32, local_lens [B] int32)."""
    I = interleave
    B = len(ctx_lens)
    out = []
    for k in range(W):
        local_tokens = []
        for r in range(B):
            n = int(ctx_lens[r])
            ts = np.arange(n)
            sel = ts[(ts // I) % W == k]
            local_tokens.append(sel)
        lens = np.array([len(s) for s in local_tokens], dtype=np.int32)
        bt, nb = paged_layout(g, lens, spare_frac=spare_frac)
        # index through an integer view: torch cannot index float8 on the CPU
        raw = cache.view(torch.uint8) if cache.element_size() == 1 else cache
        sc = torch.zeros((nb,) + tuple(cache.shape[1:]), dtype=raw.dtype)
        for r in range(B):
            ts = local_tokens[r]
            if len(ts) == 0:
                continue
            j = (ts // (I * W)) * I + ts % I
            assert np.array_equal(j, np.arange(len(ts)))
            src_blk = block_table[r, ts // BLOCK]
            src = raw[torch.from_numpy(src_blk.astype(np.int64)),
                      torch.from_numpy((ts % BLOCK).astype(np.int64))]
            dst_blk = bt[r, j // BLOCK]
            sc[torch.from_numpy(dst_blk.astype(np.int64)),
               torch.from_numpy((j % BLOCK).astype(np.int64))] = src
        out.append((sc.view(cache.dtype) if cache.element_size() == 1 else sc, bt, lens))
    return out


@dataclass
class PrefillCase:
    name: str
    B: int
    H: int
    ctx_lens: np.ndarray       # [B] context tokens per request
    new_lens: np.ndarray       # [B] new (query) tokens per request
    block_table: np.ndarray
    num_blocks: int
    cache: torch.Tensor        # global cache [nb, 64, 576] bf16
    W: int
    interleave: int
    shards: list               # W x (cache, block_table, local_lens)
    w_kvb: torch.Tensor        # [H*256, 512] bf16
    q: torch.Tensor            # [sum(new), H, 192] bf16
    new_kv: torch.Tensor       # [sum(new), 576] bf16 latent rows of new tokens
    sm_scale: float


def prefill_case(name, seed, *, ctx_lens, new_lens, H=128, W=4, interleave=1,
                 w_std=0.02, poison=False):
    g = generator(seed)
    ctx_lens = np.asarray(ctx_lens, dtype=np.int32)
    new_lens = np.asarray(new_lens, dtype=np.int32)
    bt, nb = paged_layout(g, ctx_lens)
    cache, _ = fill_cache(g, bt, ctx_lens, nb, poison=poison)
    shards = shard_cache_interleaved(g, cache, bt, ctx_lens, W, interleave)
    w_kvb = as_bf16(_normal(g, (H * (QK_NOPE + V_HEAD), KV_LORA), w_std))
    tq = int(new_lens.sum())
    q = as_bf16(_normal(g, (tq, H, QK_NOPE + ROPE), 1.0))
    new_kv = as_bf16(_normal(g, (tq, D_QK), 1.0))
    return PrefillCase(name, len(ctx_lens), H, ctx_lens, new_lens, bt, nb, cache,
                       W, interleave, shards, w_kvb, q, new_kv,
                       1.0 / math.sqrt(QK_NOPE + ROPE))


def context_prefill(poison=False, ctx=8192, n_req=4, sq=512, H=128):
    """Chunked-prefill context step: 4 x 8192 context rows on 4 interleaved
    shards, 512 new tokens per request, W_kvb ~ N(0, 0.02)."""
    return prefill_case("prefill_4x8192_w4_sq512", 1055, ctx_lens=[ctx] * n_req,
                        new_lens=[sq] * n_req, H=H, W=4, interleave=1,
                        poison=poison)
