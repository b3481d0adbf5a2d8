// A7: paged gather (plain bit copy or e4m3 -> bf16 dequantisation) and the
// fused gather + interleaved-shard reorg.
//
// Both are HBM-bound copies: every request row is read once and written
// once (1152 B + 1152 B for bf16).  A warp takes eight consecutive output
// rows: lanes 0..7 find the eight source rows at once (the segment search
// and block-table reads are dependent loads, so doing them per row would
// leave the copy waiting on them), then all 32 lanes move the eight rows
// with every 16-byte load in flight before the first store.  Sources:
//   "DeepSeek MLA 在 DCP 分布式环境中的 Prefill 阶段解析", §与非 DCP 的流程对比
//   (local gather, rank-major all-gather, reorg_kvcache) and §关于
//   cp_gather_cache 的命名澄清 (gather without dequantisation);
//   prhub digest of vLLM PR 44044, §实现拆解 3-4 (gather_and_maybe_dequant_cache
//   with seq_starts).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "common.cuh"

namespace mla {
namespace {

constexpr int kWarpsPerBlock = 8;
constexpr int kMaxShards = 16;

enum CopyMode { kCopyBf16 = 0, kCopyE4m3 = 1, kDequant = 2 };

// Largest b in [0, n) with cu[b] <= row (cu non-decreasing, cu[0] <= row).
__device__ __forceinline__ int find_segment(const int32_t *cu, int n, int row) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (__ldg(cu + mid) <= row) lo = mid; else hi = mid - 1;
  }
  return lo;
}

constexpr int kRowsPerWarp = 8;

// Eight e4m3 codes -> eight bf16: exact e4m3 -> f16 -> f32, one fp32
// multiply by k_scale, one RNE rounding to bf16.
__device__ __forceinline__ uint4 dequant8(uint2 v, float k_scale) {
  const uint32_t w[2] = {v.x, v.y};
  uint32_t o[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    __nv_fp8x2_storage_t pair =
        static_cast<__nv_fp8x2_storage_t>((w[k >> 1] >> ((k & 1) * 16)) & 0xFFFFu);
    __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3);
    float2 f = __half22float2(*reinterpret_cast<__half2 *>(&h));
    __nv_bfloat16 lo = __float2bfloat16_rn(__fmul_rn(f.x, k_scale));
    __nv_bfloat16 hi = __float2bfloat16_rn(__fmul_rn(f.y, k_scale));
    o[k] = static_cast<uint32_t>(__bfloat16_as_ushort(lo)) |
           (static_cast<uint32_t>(__bfloat16_as_ushort(hi)) << 16);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Copies (or dequantises) the warp's eight 576-element rows.  Lane i < 8
// holds row i's source (nullptr: the row is zeroed) and destination
// (nullptr: the row is not written).  Lanes take consecutive 16-byte output
// chunks, so every load and store instruction covers whole rows' runs.
template <int MODE>
__device__ __forceinline__ void copy_rows(const uint8_t *src_lane, uint8_t *dst_lane,
                                          float k_scale, int lane) {
  constexpr int C = MODE == kCopyE4m3 ? kDqk / 16 : kDqk * 2 / 16;   // output chunks per row
  constexpr int N = kRowsPerWarp * C / 32;                            // per lane: 9 or 18
  static_assert(kRowsPerWarp * C % 32 == 0, "whole chunks per lane");
  const unsigned long long s64 = reinterpret_cast<unsigned long long>(src_lane);
  const unsigned long long d64 = reinterpret_cast<unsigned long long>(dst_lane);
  uint4 v[N];
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const int idx = lane + 32 * i, row = idx / C, c = idx - row * C;
    const uint8_t *src = reinterpret_cast<const uint8_t *>(__shfl_sync(0xffffffffu, s64, row));
    if (!src) {
      v[i] = make_uint4(0, 0, 0, 0);
    } else if (MODE == kDequant) {
      v[i] = dequant8(__ldcs(reinterpret_cast<const uint2 *>(src) + c), k_scale);
    } else {
      v[i] = __ldcs(reinterpret_cast<const uint4 *>(src) + c);
    }
  }
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const int idx = lane + 32 * i, row = idx / C, c = idx - row * C;
    uint8_t *dst = reinterpret_cast<uint8_t *>(__shfl_sync(0xffffffffu, d64, row));
    if (dst) reinterpret_cast<uint4 *>(dst)[c] = v[i];
  }
}

template <int MODE>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
gather_kernel(const uint8_t *__restrict__ cache, int in_row_bytes,
              const int32_t *__restrict__ block_table,
              const int32_t *__restrict__ seq_lens,
              const int32_t *__restrict__ seq_starts,
              const int32_t *__restrict__ cu_out, int B, int max_blocks,
              int num_blocks, int total_rows, float k_scale, uint8_t *out,
              int out_row_bytes, int *err) {
  const int lane = threadIdx.x & 31;
  const int row0 = (blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5)) * kRowsPerWarp;
  if (row0 >= total_rows) return;   // uniform across the warp
  const uint8_t *src = nullptr;
  uint8_t *dst = nullptr;
  const int row = row0 + lane;
  if (lane < kRowsPerWarp && row < total_rows && row >= __ldg(cu_out) &&
      row < __ldg(cu_out + B)) {
    dst = out + static_cast<int64_t>(row) * out_row_bytes;
    const int b = find_segment(cu_out, B, row);
    const int j = row - __ldg(cu_out + b);
    const int pos = (seq_starts ? __ldg(seq_starts + b) : 0) + j;
    const int len = __ldg(seq_lens + b);
    if (pos < 0 || pos >= len || pos / kPage >= max_blocks) {
      raise_error(err, MLA_DEVERR_RANGE);
    } else {
      const int blk = __ldg(block_table + static_cast<int64_t>(b) * max_blocks + pos / kPage);
      if (blk < 0 || blk >= num_blocks) raise_error(err, MLA_DEVERR_BLOCK_ID);
      else src = cache + (static_cast<int64_t>(blk) * kPage + pos % kPage) * in_row_bytes;
    }
  }
  copy_rows<MODE>(src, dst, k_scale, lane);
}

struct ShardSet {
  const uint8_t *cache[kMaxShards];
  const int32_t *table[kMaxShards];
  int num_blocks[kMaxShards];
};

// Shard / local index of global token t (interleave I over W shards).
__device__ __forceinline__ void shard_of(int t, int W, int I, int &k, int &j) {
  k = (t / I) % W;
  j = (t / (I * W)) * I + t % I;
}

__device__ __forceinline__ const uint8_t *shard_row(const ShardSet &s, int k,
                                                    int r, int j, int smb,
                                                    int row_bytes, int *err) {
  if (j / kPage >= smb) {
    raise_error(err, MLA_DEVERR_RANGE);
    return nullptr;
  }
  const int blk = __ldg(s.table[k] + static_cast<int64_t>(r) * smb + j / kPage);
  if (blk < 0 || blk >= s.num_blocks[k]) {
    raise_error(err, MLA_DEVERR_BLOCK_ID);
    return nullptr;
  }
  return s.cache[k] + (static_cast<int64_t>(blk) * kPage + j % kPage) * row_bytes;
}

// Sequence-order output: out[cu_out[r] + t] = shard k's local row j.
template <int MODE>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
reorg_kernel(ShardSet shards, int W, int I, int smb, int in_row_bytes,
             const int32_t *__restrict__ cu_out, int B, int total_rows,
             float k_scale, uint8_t *out, int out_row_bytes, int *err) {
  const int lane = threadIdx.x & 31;
  const int row0 = (blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5)) * kRowsPerWarp;
  if (row0 >= total_rows) return;   // uniform across the warp
  const uint8_t *src = nullptr;
  uint8_t *dst = nullptr;
  const int row = row0 + lane;
  if (lane < kRowsPerWarp && row < total_rows && row >= __ldg(cu_out) &&
      row < __ldg(cu_out + B)) {
    dst = out + static_cast<int64_t>(row) * out_row_bytes;
    const int r = find_segment(cu_out, B, row);
    const int t = row - __ldg(cu_out + r);
    int k, j;
    shard_of(t, W, I, k, j);
    src = shard_row(shards, k, r, j, smb, in_row_bytes, err);
  }
  copy_rows<MODE>(src, dst, k_scale, lane);
}

// Rank-major all-gather buffer: row k*sum_p + padded_cu[r] + j.
template <int MODE>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
rank_major_kernel(ShardSet shards, int W, int I, int smb, int in_row_bytes,
                  const int32_t *__restrict__ cu_out,
                  const int32_t *__restrict__ padded_cu, int B, int sum_p,
                  float k_scale, uint8_t *out, int out_row_bytes, int *err) {
  const int lane = threadIdx.x & 31;
  const int row0 = (blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5)) * kRowsPerWarp;
  if (row0 >= W * sum_p) return;   // uniform across the warp
  const uint8_t *src = nullptr;
  uint8_t *dst = nullptr;
  const int row = row0 + lane;
  if (lane < kRowsPerWarp && row < W * sum_p) {
    const int k = row / sum_p;
    const int rem = row - k * sum_p;
    dst = out + static_cast<int64_t>(row) * out_row_bytes;
    if (rem < __ldg(padded_cu + B)) {   // else a padding row: zeros
      const int r = find_segment(padded_cu, B, rem);
      const int j = rem - __ldg(padded_cu + r);
      const int ctx = __ldg(cu_out + r + 1) - __ldg(cu_out + r);
      const int cyc = I * W;
      const int rm = ctx % cyc;
      const int n_k = (ctx / cyc) * I + min(max(rm - k * I, 0), I);
      if (j < n_k) src = shard_row(shards, k, r, j, smb, in_row_bytes, err);
    }
  }
  copy_rows<MODE>(src, dst, k_scale, lane);
}

int mode_of(int kv_dtype, int out_dtype) {
  if (kv_dtype == MLA_BF16 && out_dtype == MLA_BF16) return kCopyBf16;
  if (kv_dtype == MLA_E4M3 && out_dtype == MLA_E4M3) return kCopyE4m3;
  if (kv_dtype == MLA_E4M3 && out_dtype == MLA_BF16) return kDequant;
  return -1;
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" int mla_gather_cache(const void *kv_cache, int kv_dtype,
                                float k_scale, const int32_t *block_table,
                                const int32_t *seq_lens,
                                const int32_t *seq_starts,
                                const int32_t *cu_out, int B, int max_blocks,
                                int num_blocks, int total_rows, int out_dtype,
                                void *out, mla_stream_t stream) {
  const int mode = mode_of(kv_dtype, out_dtype);
  if (mode < 0) return MLA_ERR_INVALID_ARG;
  if (B < 1 || max_blocks < 1 || num_blocks < 1 || total_rows < 0)
    return MLA_ERR_INVALID_ARG;
  if (!kv_cache || !block_table || !seq_lens || !cu_out || (total_rows && !out))
    return MLA_ERR_INVALID_ARG;
  if (!aligned16(kv_cache) || !aligned16(out)) return MLA_ERR_INVALID_ARG;
  if (mode == kDequant && !(k_scale > 0.f)) return MLA_ERR_INVALID_ARG;
  if (total_rows == 0) return MLA_OK;
  int *err = device_error_word();
  if (!err) return MLA_ERR_CUDA;
  const int in_bytes = kv_dtype == MLA_BF16 ? kDqk * 2 : kDqk;
  const int out_bytes = out_dtype == MLA_BF16 ? kDqk * 2 : kDqk;
  constexpr int kRowsPerBlock = kWarpsPerBlock * kRowsPerWarp;
  dim3 grid((total_rows + kRowsPerBlock - 1) / kRowsPerBlock);
  auto *src = static_cast<const uint8_t *>(kv_cache);
  auto *dst = static_cast<uint8_t *>(out);
#define MLA_GATHER(M)                                                        \
  gather_kernel<M><<<grid, kWarpsPerBlock * 32, 0, stream>>>(                \
      src, in_bytes, block_table, seq_lens, seq_starts, cu_out, B,           \
      max_blocks, num_blocks, total_rows, k_scale, dst, out_bytes, err)
  if (mode == kCopyBf16) MLA_GATHER(kCopyBf16);
  else if (mode == kCopyE4m3) MLA_GATHER(kCopyE4m3);
  else MLA_GATHER(kDequant);
#undef MLA_GATHER
  return launch_status();
}

extern "C" int mla_gather_cache_reorg(
    int W, int interleave, const void *const *shard_caches,
    const int32_t *const *shard_block_tables, const int *shard_num_blocks,
    int shard_max_blocks, int kv_dtype, float k_scale, const int32_t *cu_out,
    int B, int total_rows, int out_dtype, void *out, void *rank_major_out,
    const int32_t *padded_cu, int rank_major_rows, mla_stream_t stream) {
  const int mode = mode_of(kv_dtype, out_dtype);
  if (mode < 0) return MLA_ERR_INVALID_ARG;
  if (W < 1 || W > kMaxShards || interleave < 1 || B < 1 ||
      shard_max_blocks < 1 || total_rows < 0)
    return MLA_ERR_INVALID_ARG;
  if (!shard_caches || !shard_block_tables || !shard_num_blocks || !cu_out)
    return MLA_ERR_INVALID_ARG;
  if (total_rows && !out) return MLA_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(rank_major_out)) return MLA_ERR_INVALID_ARG;
  if (mode == kDequant && !(k_scale > 0.f)) return MLA_ERR_INVALID_ARG;
  if (rank_major_out && (!padded_cu || rank_major_rows < 0 || rank_major_rows % W))
    return MLA_ERR_INVALID_ARG;
  ShardSet s{};
  for (int k = 0; k < W; ++k) {
    if (!shard_caches[k] || !shard_block_tables[k] || shard_num_blocks[k] < 1 ||
        !aligned16(shard_caches[k]))
      return MLA_ERR_INVALID_ARG;
    s.cache[k] = static_cast<const uint8_t *>(shard_caches[k]);
    s.table[k] = shard_block_tables[k];
    s.num_blocks[k] = shard_num_blocks[k];
  }
  int *err = device_error_word();
  if (!err) return MLA_ERR_CUDA;
  const int in_bytes = kv_dtype == MLA_BF16 ? kDqk * 2 : kDqk;
  const int out_bytes = out_dtype == MLA_BF16 ? kDqk * 2 : kDqk;
  auto *dst = static_cast<uint8_t *>(out);
  constexpr int kRowsPerBlock = kWarpsPerBlock * kRowsPerWarp;
  if (total_rows > 0) {
    dim3 grid((total_rows + kRowsPerBlock - 1) / kRowsPerBlock);
#define MLA_REORG(M)                                                         \
  reorg_kernel<M><<<grid, kWarpsPerBlock * 32, 0, stream>>>(                 \
      s, W, interleave, shard_max_blocks, in_bytes, cu_out, B, total_rows,   \
      k_scale, dst, out_bytes, err)
    if (mode == kCopyBf16) MLA_REORG(kCopyBf16);
    else if (mode == kCopyE4m3) MLA_REORG(kCopyE4m3);
    else MLA_REORG(kDequant);
#undef MLA_REORG
    if (cudaGetLastError() != cudaSuccess) return MLA_ERR_CUDA;
  }
  if (rank_major_out && rank_major_rows > 0) {
    const int sum_p = rank_major_rows / W;
    auto *rm = static_cast<uint8_t *>(rank_major_out);
    dim3 grid((rank_major_rows + kRowsPerBlock - 1) / kRowsPerBlock);
#define MLA_RANKMAJOR(M)                                                     \
  rank_major_kernel<M><<<grid, kWarpsPerBlock * 32, 0, stream>>>(            \
      s, W, interleave, shard_max_blocks, in_bytes, cu_out, padded_cu, B,    \
      sum_p, k_scale, rm, out_bytes, err)
    if (mode == kCopyBf16) MLA_RANKMAJOR(kCopyBf16);
    else if (mode == kCopyE4m3) MLA_RANKMAJOR(kCopyE4m3);
    else MLA_RANKMAJOR(kDequant);
#undef MLA_RANKMAJOR
  }
  return launch_status();
}
