// A8: kv_b_proj expansion of gathered latent rows into per-head K and V.
//
// Source: "DeepSeek MLA 在 DCP 分布式环境中的 Prefill 阶段解析", §MLA Prefill vs
// Decode (prefill decompresses kv_c through W_UK / W_UV into N full heads,
// K head width 128 + 64, V head width 128) and §与非 DCP 的流程对比 step 5
// (kv_b_proj after the gather / reorg).
//
//   [K_nope | V][n, h, 0:256] = kv[n, 0:512] . W_kvb[h*256 : h*256+256, :]^T
//   K[n, h, 128:192]         = kv[n, 512:576]          (k_pe, broadcast)
//
// A dense GEMM (M = rows, N = H*256, K = 512) on tcgen05: a persistent grid
// of one CTA per SM walks 128-row x 256-column (one head) tiles.  TMA feeds
// 64-wide K chunks of both operands through a 4-stage ring; one thread
// issues M=128 N=256 K=16 MMAs into one of two TMEM accumulators, so the
// four epilogue warps drain tile i while the tensor core computes tile i+1.
#include <cuda_bf16.h>

#include "common.cuh"
#include "sm100.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kStages = 4;
constexpr int kThreads = 192;
constexpr int kABytes = 128 * 64 * 2;    // 128 rows x 64 K, 16 KB
constexpr int kBBytes = 256 * 64 * 2;    // 256 cols x 64 K, 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kSmemBytes = kStages * kStageBytes + 256 + 1024;
constexpr int kKChunks = 512 / 64;

struct ExpandArgs {
  int N, H, m_tiles, tiles;
  const __nv_bfloat16 *kv;   // [N, 576]
  __nv_bfloat16 *k_out;      // [N, H, 192]
  __nv_bfloat16 *v_out;      // [N, H, 128]
};

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  return bf16x2_rn(a, b);
}

__global__ void __launch_bounds__(kThreads, 1)
expand_kernel(const __grid_constant__ CUtensorMap tm_a,
              const __grid_constant__ CUtensorMap tm_b, ExpandArgs args,
              int *err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kStages * kStageBytes);
  uint64_t *full = bars, *empty = bars + kStages;
  uint64_t *acc_full = bars + 2 * kStages, *acc_empty = acc_full + 2;
  uint64_t *drain = acc_empty + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  const int warp = warp_id(), lane = lane_id();

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&acc_full[s], 1);
      mbar_init(&acc_empty[s], 128);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // tile order: head-major inside a row block so one A block serves H tiles
  // from L2 while W_kvb (H*256 x 512) stays L2-resident as well.
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_a);
    prefetch_tmap(&tm_b);
    int kc = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < args.tiles; tile += gridDim.x) {
      const int mt = tile / args.H, h = tile % args.H;
      for (int c = 0; c < kKChunks; ++c, ++kc) {
        const int s = kc % kStages;
        if (kc >= kStages && !(ok = mbar_wait(&empty[s], ((kc / kStages) - 1) & 1, abort_flag)))
          break;
        uint8_t *dst = smem + s * kStageBytes;
        mbar_arrive_expect_tx(&full[s], kStageBytes);
        tma_load_2d(dst, &tm_a, &full[s], c * 64, mt * 128);
        tma_load_2d(dst + kABytes, &tm_b, &full[s], c * 64, h * 256);
      }
    }
    if (*abort_flag) {
      volatile int no_abort = 0;
      for (int k = max(0, kc - kStages); k < kc; ++k)
        mbar_wait(&full[k % kStages], (k / kStages) & 1, &no_abort);
    }
  } else if (warp == 1 && lane == 0) {
    const uint32_t idesc = idesc_bf16(128, 256, false, false);
    int kc = 0, n = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < args.tiles; tile += gridDim.x, ++n) {
      const int buf = n & 1;
      if (n >= 2 && !(ok = mbar_wait(&acc_empty[buf], ((n >> 1) - 1) & 1, abort_flag))) break;
      tc_fence_after();
      const uint32_t d = tmem + 256 * buf;
      for (int c = 0; c < kKChunks; ++c, ++kc) {
        const int s = kc % kStages;
        if (!(ok = mbar_wait(&full[s], (kc / kStages) & 1, abort_flag))) break;
        tc_fence_after();
        const uint32_t a = smem_u32(smem + s * kStageBytes);
        const uint32_t b = a + kABytes;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_f16_ss(d, sdesc(a + kk * 32, 16, 1024, kSwizzle128B),
                     sdesc(b + kk * 32, 16, 1024, kSwizzle128B), idesc,
                     (c | kk) != 0);
        mma_commit(&empty[s]);
      }
      if (ok) mma_commit(&acc_full[buf]);
    }
    if (!ok) {
      mma_commit(drain);
      volatile int no_abort = 0;
      mbar_wait(drain, 0, &no_abort);
    }
  } else if (warp >= 2) {
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = tmem + ((quarter * 32u) << 16);
    int n = 0;
    for (int tile = blockIdx.x; tile < args.tiles; tile += gridDim.x, ++n) {
      const int buf = n & 1;
      if (!mbar_wait(&acc_full[buf], (n >> 1) & 1, abort_flag)) break;
      tc_fence_after();
      const int mt = tile / args.H, h = tile % args.H;
      const int row = mt * 128 + r;
      const bool valid = row < args.N;
      __nv_bfloat16 *kdst = args.k_out + (static_cast<int64_t>(row) * args.H + h) * 192;
      __nv_bfloat16 *vdst = args.v_out + (static_cast<int64_t>(row) * args.H + h) * 128;
#pragma unroll 1
      for (int c = 0; c < 256; c += 32) {
        uint32_t v[32];
        tmem_ld_x32(lane_base + 256 * buf + c, v);
        if (!valid) continue;
        uint4 *dst = reinterpret_cast<uint4 *>(c < 128 ? kdst + c : vdst + (c - 128));
#pragma unroll
        for (int k = 0; k < 4; ++k)
          dst[k] = make_uint4(
              pack2(__uint_as_float(v[8 * k]), __uint_as_float(v[8 * k + 1])),
              pack2(__uint_as_float(v[8 * k + 2]), __uint_as_float(v[8 * k + 3])),
              pack2(__uint_as_float(v[8 * k + 4]), __uint_as_float(v[8 * k + 5])),
              pack2(__uint_as_float(v[8 * k + 6]), __uint_as_float(v[8 * k + 7])));
      }
      tc_fence_before();
      mbar_arrive(&acc_empty[buf]);
      if (valid) {
        // k_pe is shared by every head: copy the row's 64 rope values
        const uint4 *src = reinterpret_cast<const uint4 *>(
            args.kv + static_cast<int64_t>(row) * kDqk + kLatent);
        uint4 *dst = reinterpret_cast<uint4 *>(kdst + 128);
#pragma unroll
        for (int k = 0; k < 8; ++k) dst[k] = __ldg(src + k);
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) raise_error(err, MLA_DEVERR_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" int mla_expand_kv(const void *kv_rows, const void *w_kvb, int N,
                             int H, void *k_out, void *v_out,
                             mla_stream_t stream) {
  if (N < 0 || H < 1 || H > 1024) return MLA_ERR_INVALID_ARG;
  if (N == 0) return MLA_OK;
  if (!kv_rows || !w_kvb || !k_out || !v_out) return MLA_ERR_INVALID_ARG;
  if (!aligned16(kv_rows) || !aligned16(w_kvb) || !aligned16(k_out) || !aligned16(v_out))
    return MLA_ERR_INVALID_ARG;
  int *err = device_error_word();
  if (!err) return MLA_ERR_CUDA;
  CUtensorMap ta, tb;
  {
    const uint64_t dims[2] = {kDqk, static_cast<uint64_t>(N)};
    const uint64_t strides[1] = {kDqk * 2};
    const uint32_t box[2] = {64, 128};
    if (!make_tmap(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kv_rows, dims, strides,
                   box, CU_TENSOR_MAP_SWIZZLE_128B))
      return MLA_ERR_CUDA;
  }
  {
    const uint64_t dims[2] = {kLatent, static_cast<uint64_t>(H) * 256};
    const uint64_t strides[1] = {kLatent * 2};
    const uint32_t box[2] = {64, 256};
    if (!make_tmap(&tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w_kvb, dims, strides,
                   box, CU_TENSOR_MAP_SWIZZLE_128B))
      return MLA_ERR_CUDA;
  }
  ExpandArgs a;
  a.N = N;
  a.H = H;
  a.m_tiles = (N + 127) / 128;
  a.tiles = a.m_tiles * H;
  a.kv = static_cast<const __nv_bfloat16 *>(kv_rows);
  a.k_out = static_cast<__nv_bfloat16 *>(k_out);
  a.v_out = static_cast<__nv_bfloat16 *>(v_out);
  const int sms = device_sm_count();
  if (sms < 1) return MLA_ERR_CUDA;
  if (cudaFuncSetAttribute(expand_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kSmemBytes) != cudaSuccess)
    return MLA_ERR_CUDA;
  const int grid = a.tiles < sms ? a.tiles : sms;
  expand_kernel<<<grid, kThreads, kSmemBytes, stream>>>(ta, tb, a, err);
  return launch_status();
}
