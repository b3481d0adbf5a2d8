/*
 * mla.h — C ABI of the GB300 (sm_103a) absorbed Multi-head Latent Attention
 * decode library.
 *
 * Sources of the operations (page title, section):
 *   [Q-REP]   prhub digest of vLLM PR 45964, "MLA DCP 中通过 query 复制跳过
 *             all-gather 通信"
 *   [FP8]     prhub digest of vLLM PR 44044, "支持 DCP + FP8 KV Cache 在 MLA
 *             解码中协同"
 *   [BLOG]    "DeepSeek MLA 在 DCP 分布式环境中的 Prefill 阶段解析"
 *
 * Conventions shared by every entry point
 *   - Every tensor pointer is a caller-owned DEVICE pointer (unless the
 *     argument says "host"), contiguous and row-major in the layout given.
 *     The library never allocates or frees device memory: scratch space is a
 *     caller workspace whose size a *_workspace_size query returns.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream) and returns an int status.  Arguments are
 *     validated on the host before any launch and without a device sync;
 *     a bad argument returns MLA_ERR_INVALID_ARG and launches nothing.
 *   - Device-side data the host cannot see (block ids, seq_lens) is checked
 *     inside the kernels: a bad value sets a bit in a device error word and
 *     the offending row is skipped (never read out of bounds).  Read and
 *     clear that word with mla_get_device_error().
 *   - Dtype codes: MLA_BF16 (bf16), MLA_E4M3 (OCP fp8 e4m3, "fn" variant:
 *     no inf, max 448), MLA_F32 (IEEE float32).  Scales are per-tensor fp32.
 *   - Sizes: L = 512 latent rank, R = 64 rope width, 576 = L + R, nope and
 *     value head widths 128, cache page size 64 tokens.
 *   - Kernels run on the current CUDA device of the calling thread; every
 *     pointer must belong to it.
 */
#ifndef MLA_GB300_H_
#define MLA_GB300_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *mla_stream_t; /* identical to cudaStream_t */

enum mla_status {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1, /* bad pointer / size / dtype combination        */
  MLA_ERR_UNSUPPORTED = 2, /* valid request the library does not implement */
  MLA_ERR_WORKSPACE = 3,   /* workspace missing or smaller than required    */
  MLA_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed          */
};

enum mla_dtype { MLA_BF16 = 0, MLA_E4M3 = 1, MLA_F32 = 2 };

/* Bits of the device error word (mla_get_device_error). */
enum mla_device_error {
  MLA_DEVERR_BLOCK_ID = 1,    /* block-table entry < 0 or >= num_blocks     */
  MLA_DEVERR_SEQ_LEN = 2,     /* seq_len < 0 or > max_blocks * 64           */
  MLA_DEVERR_RANGE = 4,       /* gather range beyond seq_len / workspace    */
  MLA_DEVERR_TIMEOUT = 8,     /* a bounded wait inside a kernel gave up     */
};

/* Self-test of the failure detection every kernel relies on (no
 * counterpart on the pages): one thread waits, through the same bounded
 * mbarrier wait the kernels use, on a barrier that nothing completes; after
 * limit_cycles SM cycles (1 .. 1e9) it gives up and raises
 * MLA_DEVERR_TIMEOUT in the device error word, the way a kernel whose
 * producer or peer stalls reports it.  Faults nothing, and the context stays
 * usable.  MLA_ERR_INVALID_ARG for a limit out of range. */
int mla_selftest_wait_timeout(long long limit_cycles, mla_stream_t stream);

/* Human-readable text of a status code (static storage, never NULL). */
const char *mla_status_string(int status);

/* Library ABI version, currently 1. */
int mla_version(void);

/* Synchronises `stream`, stores the device error word (bitwise OR of
 * mla_device_error values raised since the last call) into *code (host
 * pointer) and clears it.  Returns MLA_ERR_CUDA if the sync fails. */
int mla_get_device_error(int *code, mla_stream_t stream);

/* ---------------------------------------------------------------------
 * A1/A2  Query absorption and concat(-quant)
 * [Q-REP] §实现拆解 5 (decode BMM of the query against W_UK_T);
 * [BLOG] §MLA Prefill vs Decode (Q absorbed into the latent space by an
 * einsum, one latent head of width L+R); [FP8] §关键源码片段
 * mla_attention.py (nope ‖ pe -> (B, N, L+P); _decode_concat_quant_fp8_op).
 *
 *   ql[t,h,l] = sum_p q_nope[t,h,p] * w_uk_t[h,p,l]       (fp32 accumulate)
 *   q_out[t,h,0:512]   = cast(ql[t,h,:]),  q_out[t,h,512:576] = cast(q_pe)
 *
 * q_nope [T,H,128] bf16, q_pe [T,H,64] bf16, w_uk_t [H,128,512] bf16.
 * out_dtype MLA_BF16: round-to-nearest-even of the fp32 value;
 *           MLA_E4M3: e4m3 code of (fp32 value) / q_scale (IEEE fp32
 *                     division, round to nearest even, saturate to +-448);
 *           MLA_F32 : the fp32 value itself.
 * q_out [T,H,576] of out_dtype.  T == 0 is a no-op.  1 <= H <= 4096.
 * q_scale must be finite and > 0 for MLA_E4M3 (ignored otherwise). */
int mla_absorb_q(const void *q_nope, const void *q_pe, const void *w_uk_t,
                 int T, int H, int out_dtype, float q_scale, void *q_out,
                 mla_stream_t stream);

/* ---------------------------------------------------------------------
 * A3/A4/A5  Paged latent decode (forward_mqa) with split-KV and merge
 * [FP8] §关键源码片段 mla_attention.py (forward_mqa(mqa_q, kv_cache, ...)
 * returns attn_out and lse) and §关键源码片段 flashmla.py (split scheduler
 * metadata from seq_lens and the true query-head count); [BLOG] §MLA
 * Prefill vs Decode.
 *
 * For request b, query token i < q_len, head h < H:
 *   range: lo = kv_starts ? max(0, kv_starts[b]) : 0
 *          hi = min(seq_lens[b], causal ? seq_lens[b] - q_len + i + 1 : inf,
 *                   kv_ends ? kv_ends[b] : inf)
 *   s_j  = sm_scale * q_deq[b,i,h,:] . K_j        (j in [lo, hi))
 *   K_j  = kv_deq[slot(b,j), 0:576],  V_j = kv_deq[slot(b,j), 0:512]
 *   slot(b,j) = block_table[b, j/64] * 64 + j%64
 *   lse[b,i,h] = ln sum_j exp(s_j)   (natural log; -inf for an empty range)
 *   out[b,i,h,:] = sum_j exp(s_j - lse) V_j           (0 for an empty range)
 * q_deq = q (bf16) or q_scale * e4m3(q); kv_deq = kv (bf16) or
 * k_scale * e4m3(kv).  q_dtype must equal kv_dtype.
 *
 * q [B,q_len,H,576]; kv_cache [num_blocks,64,576]; block_table
 * [B,max_blocks] int32 (entries past the used pages are ignored);
 * seq_lens [B] int32; kv_starts / kv_ends [B] int32 or NULL (an explicit
 * key shard, e.g. one DCP rank's slice); out [B,q_len,H,512] of out_dtype
 * (MLA_BF16 or MLA_F32); lse [B,q_len,H] fp32.
 *
 * The split of the key ranges over CTAs is planned on the device
 * (mla_decode_plan) and partial results are merged on the device; no host
 * synchronisation.  split_tiles = 0 lets the planner choose; > 0 forces
 * spans of that many 64-token key tiles (testing / tuning).  workspace must
 * hold mla_decode_workspace_size(B, q_len, H, max_blocks*64, split_tiles)
 * bytes (16-byte aligned).
 * Limits: 1 <= B, 1 <= q_len <= 64, 1 <= H <= 4096, 1 <= max_blocks,
 * 1 <= num_blocks < 2^25. */
int mla_decode_workspace_size(int B, int q_len, int H, int max_seq_len,
                              int split_tiles, size_t *bytes);

int mla_decode_paged(const void *q, int q_dtype, float q_scale,
                     const void *kv_cache, int kv_dtype, float k_scale,
                     const int32_t *block_table, const int32_t *seq_lens,
                     const int32_t *kv_starts, const int32_t *kv_ends, int B,
                     int q_len, int H, int max_blocks, int num_blocks,
                     float sm_scale, int causal, int split_tiles, void *out,
                     int out_dtype, float *lse, void *workspace,
                     size_t ws_bytes, mla_stream_t stream);

/* mla_decode_paged without a caller workspace, for callers that cannot
 * allocate device memory at call time: serving runtimes whose device
 * memory is carved up once before traffic starts, plug-in hosts that forbid
 * allocation on the call path, and C callers with no allocator of their
 * own.  No counterpart on the source pages: it is a packaging
 * variant of A3/A4/A5.
 *
 * The plan and the split partials live in one static device array of
 * MLA_NOALLOC_SCRATCH_BYTES (64 MiB) inside the library.  Every GPU on
 * which the library's decode module is loaded holds it until the process
 * exits; with CUDA's default lazy module loading the 64 MiB is committed
 * the first time the decode code is used on a device (the first decode
 * call of any kind), so make that first call before device memory is
 * carved up, and before any stream capture (it also looks the array's
 * device address up once, with cudaGetSymbolAddress, and caches it per
 * device index).  cudaDeviceReset is not supported once the library has
 * been used: the cached address would belong to the old context.
 *
 * Size limit, in caller terms: the workspace is the plan plus one slot of
 * 256.5 KB (a 128 x 512 fp32 partial and its 128 LSEs) for each of
 * J + G partials, J = B * q_len * ceil(H / 128) jobs and G = the number of
 * CTA pairs (76 on a 152-SM GB300) with the automatic split, or
 * ceil(J * (max_blocks + 4) / split_tiles) with a forced
 * split.  About 255 slots fit, so with the automatic split on a GB300 up
 * to about 179 jobs run: the DeepSeek-V3 decode shape (B = 32, q_len 1,
 * H = 128, J = 32) and B = 64 fp8 decode (J = 64) fit; B = 128 with
 * q_len = 2 (J = 256) is rejected.  Larger requests return
 * MLA_ERR_WORKSPACE, after every argument check of mla_decode_paged (a
 * bad argument still returns MLA_ERR_INVALID_ARG).
 * The library never allocates here: no cudaMalloc, cudaFree or allocating
 * library routine.  Every call shares the one array, so calls that overlap
 * on the GPU (different streams, or devices sharing a context) race and
 * must be serialised by the caller.  Nothing in the array needs to start at
 * zero: the plan is rewritten and every partial is written before it is
 * read on each call.  Arguments and results are those of mla_decode_paged. */
#define MLA_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

int mla_decode_paged_noalloc(const void *q, int q_dtype, float q_scale,
                             const void *kv_cache, int kv_dtype, float k_scale,
                             const int32_t *block_table,
                             const int32_t *seq_lens, const int32_t *kv_starts,
                             const int32_t *kv_ends, int B, int q_len, int H,
                             int max_blocks, int num_blocks, float sm_scale,
                             int causal, int split_tiles, void *out,
                             int out_dtype, float *lse, mla_stream_t stream);

/* A3 on its own: writes the split plan that mla_decode_paged computes.
 * Jobs are (i, b, head group of 128) in that nesting order (query token
 * outermost: with an even number of CTA pairs, the pairs working on the
 * query tokens of a request then read the same key tiles at about the same
 * time, so the later read finds them in L2); with the tile
 * size tk = 64 tokens (both kv dtypes; kv_dtype is kept so the tile may
 * differ by format), job j covers key tiles [lo/tk, ceil(hi/tk)); the jobs
 * are concatenated into one flat space where a non-empty job takes 4 units
 * (the cost of switching a CTA pair to it, in tile-equivalents, no keys)
 * followed by its tiles, `total` units in all, and CTA group p owns units
 * [p*C, (p+1)*C) with C = split_tiles if > 0, else
 * max(4, ceil(total / n_groups)), i.e. the tiles of every job it meets.
 * plan [4 + 4*(J+1)] int32 receives: [0] total, [1] C, [2] J, [3] number
 * of spans, then unit_prefix[J+1] (units per job, prefix-summed),
 * seg_prefix[J+1] (partial results per job, prefix-summed), job_lo[J+1],
 * job_hi[J+1] (last entries 0).
 * n_groups = 0 uses half the device's SM count. */
int mla_decode_plan(const int32_t *seq_lens, const int32_t *kv_starts,
                    const int32_t *kv_ends, int B, int q_len, int H,
                    int max_blocks, int causal, int kv_dtype, int split_tiles,
                    int n_groups, int32_t *plan, size_t plan_bytes,
                    mla_stream_t stream);

/* ---------------------------------------------------------------------
 * Before the path: rotary position embedding and the cache write
 * [Q-REP] §关键源码片段 mla.py (rotary_emb(positions, q[..., qk_nope_head_dim:],
 * k_pe) runs before mla_attn); [BLOG] §Chunked Prefill 与 LSE Merge (the
 * new tokens' KV is already in the cache when attention runs).  The pages
 * name the rotation but not its variant: this is RoFormer's rotary
 * embedding (Su et al. 2021), pair i of a 64-wide vector turned by
 *   theta = positions[t] * rope_base^(-2i/64):
 *   (a, b) -> (a cos theta - b sin theta, a sin theta + b cos theta),
 * pairs (2i, 2i+1) for MLA_ROPE_INTERLEAVED, (i, i+32) for MLA_ROPE_HALF.
 * Angles and their sine / cosine are computed in fp64, the rotation in
 * fp32, rounded to bf16 once.
 * For each new token t < T:
 *   q_pe [T,H,64] bf16 (NULL: no query) is rotated in place;
 *   k_pe [T,64] bf16 is rotated in place;
 *   row slot_mapping[t] (= block * 64 + offset) of kv_cache
 *   [num_blocks,64,576] receives kv_c[t] [512] bf16 ‖ the rotated k_pe[t]:
 *   the bits for kv_dtype MLA_BF16, e4m3(fp32(x) / k_scale) (RNE,
 *   saturating) for MLA_E4M3.
 * A negative slot is padding and writes nothing; a slot >= num_blocks*64
 * sets MLA_DEVERR_BLOCK_ID and writes nothing.  positions, slot_mapping
 * [T] int32.  1 < rope_base < inf.  T == 0 is a no-op. */
enum mla_rope_layout { MLA_ROPE_INTERLEAVED = 0, MLA_ROPE_HALF = 1 };

int mla_rope_cache_write(void *q_pe, void *k_pe, const void *kv_c,
                         const int32_t *positions, const int32_t *slot_mapping,
                         int T, int H, float rope_base, int rope_layout,
                         void *kv_cache, int kv_dtype, float k_scale,
                         int num_blocks, mla_stream_t stream);

/* ---------------------------------------------------------------------
 * A5/A10  LSE-rescaling merge of partial attention states
 * [BLOG] §Chunked Prefill 与 LSE Merge (merge_attn_states: elementwise
 * O(B*N*V) rescaling) and §DCP 在 Prefill 与 Decode 中的不同角色 (decode
 * combines per-rank partial outputs by LSE weighting).
 *
 * Per row (t,h): m = max_s lse_s; w_s = exp(lse_s - m) (0 if lse_s = -inf)
 *   out = sum_s w_s * part_s / sum_s w_s;  out_lse = m + ln sum_s w_s.
 * All parts -inf: out = 0, out_lse = -inf.  S = 2 is the pages'
 * prefix/suffix form.
 * parts_out [S,T,H,D] (MLA_BF16 or MLA_F32); parts_lse [S,T,H] fp32;
 * out [T,H,D] (MLA_BF16 or MLA_F32); out_lse [T,H] fp32 or NULL.
 * 1 <= S <= 256, D % 8 == 0, D <= 1024. */
int mla_merge_states(const void *parts_out, int parts_dtype,
                     const float *parts_lse, int S, int T, int H, int D,
                     void *out, int out_dtype, float *out_lse,
                     mla_stream_t stream);

/* ---------------------------------------------------------------------
 * A6  Value up-projection
 * [BLOG] §MLA Prefill vs Decode (W_UV expands the latent output back to
 * per-head values); [Q-REP] §关键源码片段 mla.py (output viewed as
 * (tokens, num_heads * v_head_dim)).
 *   out[t,h,v] = sum_l o_lat[t,h,l] * w_uv[h,v,l]   (fp32 accumulate, RNE)
 * o_lat [T,H,512] bf16, w_uv [H,128,512] bf16, out [T,H,128] bf16.
 * T == 0 is a no-op.  1 <= H <= 4096. */
int mla_v_up(const void *o_lat, const void *w_uv, int T, int H, void *out,
             mla_stream_t stream);

/* ---------------------------------------------------------------------
 * A7  Paged gather (cp_gather_cache / gather_and_maybe_dequant_cache)
 * [BLOG] §与非 DCP 的流程对比 and §关于 cp_gather_cache 的命名澄清 (a gather
 * with no dequantisation); [FP8] §实现拆解 3-4 (dequantising gather,
 * seq_starts).
 *   out[cu_out[b] + j] = cast(kv_cache[slot(b, s_b + j)])
 *   for j < cu_out[b+1] - cu_out[b], s_b = seq_starts ? seq_starts[b] : 0.
 * out_dtype == kv_dtype: exact bit copy (bf16 or e4m3 rows).
 * kv_dtype MLA_E4M3, out_dtype MLA_BF16: bf16(RNE)(fp32(e4m3) * k_scale).
 * cu_out [B+1] int32 device; total_rows (host) >= cu_out[B] sizes out
 * [total_rows, 576] and the launch; rows past cu_out[B] are not written.
 * A row with s_b + j >= seq_lens[b] sets MLA_DEVERR_RANGE and is zeroed. */
int mla_gather_cache(const void *kv_cache, int kv_dtype, float k_scale,
                     const int32_t *block_table, const int32_t *seq_lens,
                     const int32_t *seq_starts, const int32_t *cu_out, int B,
                     int max_blocks, int num_blocks, int total_rows,
                     int out_dtype, void *out, mla_stream_t stream);

/* A7  Gather from W interleaved DCP shards and restore sequence order
 * (local cp_gather_cache on every rank + all_gather(dim=0) + reorg_kvcache,
 * fused; the shards live on this one GPU).
 * [BLOG] §与非 DCP 的流程对比 steps 1-4 (rank-major all-gathered buffer,
 * reorg by padded local lengths and every rank's local context lengths).
 * Placement: token t of request r lives on shard k = (t / I) % W at local
 * index j = (t / (I*W)) * I + t % I, in that shard's paged cache.
 *   out[cu_out[r] + t] = cast(shard_cache[k][slot_k(r, j)]),  t < ctx_r
 * with ctx_r = cu_out[r+1] - cu_out[r].
 * shard_caches / shard_block_tables / shard_num_blocks are HOST arrays of
 * W entries (device pointers / host ints); each table is [B, shard_max_blocks].
 * If rank_major_out != NULL it also receives the all-gathered rank-major
 * buffer: row k*sum_p + padded_cu[r] + j holds shard k's local row j of
 * request r, rows j in [n_{r,k}, p_r) are zero, p_r = max_k n_{r,k} =
 * (ctx_r / (I*W)) * I + min(ctx_r % (I*W), I), padded_cu [B+1] int32 device
 * is the prefix sum of p_r and rank_major_rows (host) = W * sum_p.
 * 1 <= W <= 16, 1 <= I. */
int mla_gather_cache_reorg(int W, int interleave,
                           const void *const *shard_caches,
                           const int32_t *const *shard_block_tables,
                           const int *shard_num_blocks, int shard_max_blocks,
                           int kv_dtype, float k_scale, const int32_t *cu_out,
                           int B, int total_rows, int out_dtype, void *out,
                           void *rank_major_out, const int32_t *padded_cu,
                           int rank_major_rows, mla_stream_t stream);

/* ---------------------------------------------------------------------
 * A8  kv_b_proj expansion of latent rows into per-head K and V
 * [BLOG] §MLA Prefill vs Decode (kv_c decompressed through W_UK/W_UV into
 * N heads, K head dim 128+64, V head dim 128) and §与非 DCP 的流程对比 step 5.
 *   K[n,h,0:128]   = sum_l kv[n,l] * w_kvb[h*256 + c, l]         (c < 128)
 *   V[n,h,0:128]   = sum_l kv[n,l] * w_kvb[h*256 + 128 + c, l]
 *   K[n,h,128:192] = kv[n,512:576]                            (k_pe, copied)
 * kv_rows [N,576] bf16 (e.g. mla_gather_cache output), w_kvb [H*256,512]
 * bf16 (nn.Linear layout), k_out [N,H,192] bf16, v_out [N,H,128] bf16.
 * N == 0 is a no-op.  1 <= H <= 1024. */
int mla_expand_kv(const void *kv_rows, const void *w_kvb, int N, int H,
                  void *k_out, void *v_out, mla_stream_t stream);

/* ---------------------------------------------------------------------
 * A9  Prefill multi-head attention with LSE (run_prefill_new_tokens /
 * run_prefill_context_chunk)
 * [BLOG] §Chunked Prefill 与 LSE Merge (new tokens: causal, returns the
 * softmax LSE; context chunks: non-causal).
 * Request b owns query rows [cu_q[b], cu_q[b+1]) and key rows
 * [cu_k[b], cu_k[b+1]); with nq, nk those counts, query i sees keys
 *   j < nk                       (causal = 0)
 *   j <= i + nk - nq             (causal = 1, bottom-right aligned)
 *   s_j = sm_scale * q.k_j;  lse = ln sum exp(s_j);  out = softmax . V
 * q [Tq,H,192], k [Nk,H,192], v [Nk,H,128] bf16; out [Tq,H,128] bf16;
 * lse [Tq,H] fp32.  cu_q / cu_k [B+1] int32 device; max_q_len (host) bounds
 * every nq and sizes the launch.  A query that sees no key gets out = 0,
 * lse = -inf. */
int mla_prefill_attn(const void *q, const void *k, const void *v,
                     const int32_t *cu_q, const int32_t *cu_k, int B, int Tq,
                     int Nk, int H, int max_q_len, int causal, float sm_scale,
                     void *out, float *lse, mla_stream_t stream);

/* ---------------------------------------------------------------------
 * Host staging of a step's inputs and results
 * [BLOG] §MLA Prefill vs Decode (each decode step takes the new tokens'
 * queries in and hands the attention output on).  No page defines the
 * transfer itself.
 * Copies `bytes` from src to dst, where exactly one of the two is
 * page-locked, device-mapped HOST memory (cudaHostAlloc / cudaHostRegister,
 * e.g. a pinned torch tensor) and the other is memory of the current
 * device; the SMs load and store over the host link (no copy engine), so
 * the call is a kernel launch like every other entry point (asynchronous on
 * `stream`, capturable in a CUDA graph; it waits for the previous kernel in
 * the stream before reading src).  Both pointers 16-byte aligned, bytes a
 * multiple of 16.  bytes == 0 is a no-op.
 * Pageable host memory, host-to-host, device-to-device or another device's
 * memory: MLA_ERR_INVALID_ARG, nothing launched. */
int mla_stage_copy(void *dst, const void *src, size_t bytes, mla_stream_t stream);

#ifdef __cplusplus
} /* extern "C" */
#endif

#endif /* MLA_GB300_H_ */
