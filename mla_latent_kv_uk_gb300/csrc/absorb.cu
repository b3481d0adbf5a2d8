// A1/A2 query absorption (+ concat, + optional e4m3 quantisation) and A6
// value up-projection: per-head GEMMs on the 5th-generation tensor cores.
//
// Both are small per-head contractions whose cost is reading the weights
// (W_UK_T / W_UV: H x 128 x 512 bf16 = 16 MiB at H = 128).  Each CTA owns
// one (head, 128-row M tile, token tile): TMA streams 64-wide K chunks of
// the weight and the activations into 128B-swizzled shared memory, one
// thread issues tcgen05.mma (M = 128, N = token tile, K = 16 per
// instruction) into a TMEM accumulator, and four epilogue warps read the
// accumulator with tcgen05.ld (lane = M row) and write the output rows.
//
//   absorb: ql^T[l, t] = sum_p W_UK_T[h][p, l] * q_nope[t, h, p]
//           A = W_UK_T[h] chunk, MN-major (l contiguous); B = q_nope, K-major
//   v_up:   out^T[v, t] = sum_l W_UV[h][v, l] * o_lat[t, h, l]
//           A = W_UV[h], K-major; B = o_lat, K-major
//
// Sources: prhub digest of vLLM PR 45964, §实现拆解 5 (the W_UK_T BMM of the
// decode branch); "DeepSeek MLA 在 DCP 分布式环境中的 Prefill 阶段解析",
// §MLA Prefill vs Decode (einsum absorption; W_UV expansion); prhub digest
// of vLLM PR 44044, §关键源码片段 mla_attention.py (nope ‖ pe concat, then
// _decode_concat_quant_fp8_op with the query scale).
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "sm100.cuh"

namespace mla {
namespace {

using namespace sm100;

enum Op { kAbsorb = 0, kVup = 1 };

constexpr int kStages = 4;
constexpr int kThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int kChunkK = 64;    // K elements per pipeline stage
constexpr int kABytes = 128 * kChunkK * 2;  // one 128 x 64 bf16 A chunk

struct GemmArgs {
  int T, H, NT;            // tokens, heads, token tile (multiple of 16)
  int out_dtype;           // absorb: MLA_BF16 / MLA_E4M3 / MLA_F32
  float q_scale;
  const __nv_bfloat16 *q_pe;  // absorb only
  void *out;
  int *err;
};

__device__ __forceinline__ void store_q(void *out, int dtype, int64_t idx,
                                        float v, float q_scale) {
  if (dtype == MLA_BF16) {
    static_cast<__nv_bfloat16 *>(out)[idx] = __float2bfloat16_rn(v);
  } else if (dtype == MLA_F32) {
    static_cast<float *>(out)[idx] = v;
  } else {
    // e4m3 of the correctly rounded fp32 quotient: RNE, saturate to 448
    static_cast<__nv_fp8_storage_t *>(out)[idx] =
        __nv_cvt_float_to_fp8(__fdiv_rn(v, q_scale), __NV_SATFINITE, __NV_E4M3);
  }
}

template <int OP>
__global__ void __launch_bounds__(kThreads, 1)
head_gemm_kernel(const __grid_constant__ CUtensorMap tm_a,
                 const __grid_constant__ CUtensorMap tm_b, GemmArgs args) {
  constexpr int KC = OP == kAbsorb ? 128 / kChunkK : 512 / kChunkK;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int NT = args.NT;
  const int b_bytes = NT * kChunkK * 2;
  const int stage_bytes = kABytes + b_bytes;  // multiple of 1024 (NT % 16 == 0 -> 2 KB)
  uint8_t *stages = smem;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + kStages * stage_bytes);
  uint64_t *empty = full + kStages;
  uint64_t *done = empty + kStages;
  uint64_t *drain = done + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = warp_id();
  const int lane = lane_id();
  // grid: absorb (latent chunk, head, token tile); v_up (head, token tile)
  const int mchunk = OP == kAbsorb ? blockIdx.x : 0;
  const int h = OP == kAbsorb ? blockIdx.y : blockIdx.x;
  const int ttile = OP == kAbsorb ? blockIdx.z : blockIdx.y;
  const int t0 = ttile * NT;
  const int ntok = min(NT, args.T - t0);
  const uint32_t tmem_cols = NT <= 32 ? 32 : NT <= 64 ? 64 : NT <= 128 ? 128 : 256;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer
    prefetch_tmap(&tm_a);
    prefetch_tmap(&tm_b);
    int armed_last = -1;
    for (int kc = 0; kc < KC; ++kc) {
      const int s = kc % kStages;
      if (kc >= kStages && !mbar_wait(&empty[s], ((kc / kStages) - 1) & 1, abort_flag))
        break;
      uint8_t *a_dst = stages + s * stage_bytes;
      uint8_t *b_dst = a_dst + kABytes;
      mbar_arrive_expect_tx(&full[s], stage_bytes);
      armed_last = kc;
      if (OP == kAbsorb) {
        // W_UK_T viewed as [H*128 rows (p), 512 cols (l)]; box 64 l x 64 p
        const int row = h * 128 + kc * kChunkK;
        tma_load_2d(a_dst, &tm_a, &full[s], mchunk * 128, row);
        tma_load_2d(a_dst + kABytes / 2, &tm_a, &full[s], mchunk * 128 + 64, row);
      } else {
        // W_UV viewed as [H*128 rows (v), 512 cols (l)]; box 64 l x 128 v
        tma_load_2d(a_dst, &tm_a, &full[s], kc * kChunkK, h * 128);
      }
      // activations [T, H, K]: box {64 (k), 1 (h), NT (t)}
      tma_load_3d(b_dst, &tm_b, &full[s], kc * kChunkK, h, t0);
    }
    if (*abort_flag) {
      // let the copies this thread started land before the CTA exits
      for (int kc = max(0, armed_last - kStages + 1); kc <= armed_last; ++kc) {
        volatile int no_abort = 0;
        mbar_wait(&full[kc % kStages], (kc / kStages) & 1, &no_abort);
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer
    const uint32_t idesc = idesc_bf16(128, NT, OP == kAbsorb, false);
    bool ok = true;
    for (int kc = 0; kc < KC && ok; ++kc) {
      const int s = kc % kStages;
      ok = mbar_wait(&full[s], (kc / kStages) & 1, abort_flag);
      if (!ok) break;
      tc_fence_after();
      const uint32_t a_base = smem_u32(stages + s * stage_bytes);
      const uint32_t b_base = a_base + kABytes;
#pragma unroll
      for (int kk = 0; kk < kChunkK / 16; ++kk) {
        uint64_t adesc, bdesc;
        if (OP == kAbsorb) {
          // MN-major A: rows = K (p), 128 B = 64 l per row; 8-row groups
          // 1024 B apart (SBO); the two 64-l halves 8 KB apart (LBO).
          adesc = sdesc(a_base + kk * 2048, kABytes / 2, 1024, kSwizzle128B);
        } else {
          adesc = sdesc(a_base + kk * 32, 16, 1024, kSwizzle128B);
        }
        bdesc = sdesc(b_base + kk * 32, 16, 1024, kSwizzle128B);
        mma_f16_ss(tmem, adesc, bdesc, idesc, (kc | kk) != 0);
      }
      mma_commit(&empty[s]);
    }
    mma_commit(ok ? done : drain);
    if (!ok) {
      volatile int no_abort = 0;
      mbar_wait(drain, 0, &no_abort);
    }
  } else if (warp >= 2) {
    // ---------------- epilogue: TMEM lane = M row, columns = tokens
    const bool ok = mbar_wait(done, 0, abort_flag);
    tc_fence_after();
    const int quarter = warp & 3;
    const int m = quarter * 32 + lane;  // M row owned by this thread
    if (ok) {
      for (int c0 = 0; c0 < NT; c0 += 32) {
        uint32_t r[32];
        tmem_ld_x32(tmem_addr(tmem, warp, c0), r);
        const int nc = min(32, ntok - c0);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          if (c >= nc) break;
          const int t = t0 + c0 + c;
          const float v = __uint_as_float(r[c]);
          if (OP == kAbsorb) {
            const int64_t idx = (static_cast<int64_t>(t) * args.H + h) * kDqk +
                                mchunk * 128 + m;
            store_q(args.out, args.out_dtype, idx, v, args.q_scale);
          } else {
            const int64_t idx = (static_cast<int64_t>(t) * args.H + h) * kVhead + m;
            static_cast<__nv_bfloat16 *>(args.out)[idx] = __float2bfloat16_rn(v);
          }
        }
      }
      if (OP == kAbsorb && mchunk == 0) {
        // q_pe columns 512..575 of every token in the tile
        const int tid = threadIdx.x - 64;
        for (int idx = tid; idx < ntok * kRope; idx += 128) {
          const int t = t0 + idx / kRope, r = idx % kRope;
          const float v = __bfloat162float(
              args.q_pe[(static_cast<int64_t>(t) * args.H + h) * kRope + r]);
          store_q(args.out, args.out_dtype,
                  (static_cast<int64_t>(t) * args.H + h) * kDqk + kLatent + r, v,
                  args.q_scale);
        }
      }
    }
    tc_fence_before();
  }
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) raise_error(args.err, MLA_DEVERR_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, tmem_cols);
  }
}

int token_tile(int T) {
  int nt = ((T + 15) / 16) * 16;
  return nt > 256 ? 256 : nt;
}

size_t smem_bytes(int NT) {
  return 1024 + static_cast<size_t>(kStages) * (kABytes + NT * kChunkK * 2) + 256;
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" int mla_absorb_q(const void *q_nope, const void *q_pe,
                            const void *w_uk_t, int T, int H, int out_dtype,
                            float q_scale, void *q_out, mla_stream_t stream) {
  if (T < 0 || H < 1 || H > 4096) return MLA_ERR_INVALID_ARG;
  if (out_dtype != MLA_BF16 && out_dtype != MLA_E4M3 && out_dtype != MLA_F32)
    return MLA_ERR_INVALID_ARG;
  if (out_dtype == MLA_E4M3 && !(q_scale > 0.f && q_scale < INFINITY))
    return MLA_ERR_INVALID_ARG;
  if (T == 0) return MLA_OK;
  if (!q_nope || !q_pe || !w_uk_t || !q_out) return MLA_ERR_INVALID_ARG;
  if (!aligned16(q_nope) || !aligned16(w_uk_t)) return MLA_ERR_INVALID_ARG;
  int *err = device_error_word();
  if (!err) return MLA_ERR_CUDA;
  const int NT = token_tile(T);
  CUtensorMap ta, tb;
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(kLatent),
                              static_cast<uint64_t>(H) * kNope};
    const uint64_t strides[1] = {kLatent * 2};
    const uint32_t box[2] = {64, 64};
    if (!make_tmap(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w_uk_t, dims,
                   strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return MLA_ERR_CUDA;
  }
  {
    const uint64_t dims[3] = {static_cast<uint64_t>(kNope),
                              static_cast<uint64_t>(H), static_cast<uint64_t>(T)};
    const uint64_t strides[2] = {kNope * 2, static_cast<uint64_t>(H) * kNope * 2};
    const uint32_t box[3] = {64, 1, static_cast<uint32_t>(NT)};
    if (!make_tmap(&tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q_nope, dims,
                   strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return MLA_ERR_CUDA;
  }
  GemmArgs a{T, H, NT, out_dtype, q_scale,
             static_cast<const __nv_bfloat16 *>(q_pe), q_out, err};
  const size_t smem = smem_bytes(NT);
  auto kern = head_gemm_kernel<kAbsorb>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return MLA_ERR_CUDA;
  dim3 grid(kLatent / 128, H, (T + NT - 1) / NT);
  kern<<<grid, kThreads, smem, stream>>>(ta, tb, a);
  return launch_status();
}

extern "C" int mla_v_up(const void *o_lat, const void *w_uv, int T, int H,
                        void *out, mla_stream_t stream) {
  if (T < 0 || H < 1 || H > 4096) return MLA_ERR_INVALID_ARG;
  if (T == 0) return MLA_OK;
  if (!o_lat || !w_uv || !out) return MLA_ERR_INVALID_ARG;
  if (!aligned16(o_lat) || !aligned16(w_uv)) return MLA_ERR_INVALID_ARG;
  int *err = device_error_word();
  if (!err) return MLA_ERR_CUDA;
  const int NT = token_tile(T);
  CUtensorMap ta, tb;
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(kLatent),
                              static_cast<uint64_t>(H) * kVhead};
    const uint64_t strides[1] = {kLatent * 2};
    const uint32_t box[2] = {64, 128};
    if (!make_tmap(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w_uv, dims,
                   strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return MLA_ERR_CUDA;
  }
  {
    const uint64_t dims[3] = {static_cast<uint64_t>(kLatent),
                              static_cast<uint64_t>(H), static_cast<uint64_t>(T)};
    const uint64_t strides[2] = {kLatent * 2,
                                 static_cast<uint64_t>(H) * kLatent * 2};
    const uint32_t box[3] = {64, 1, static_cast<uint32_t>(NT)};
    if (!make_tmap(&tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, o_lat, dims,
                   strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return MLA_ERR_CUDA;
  }
  GemmArgs a{T, H, NT, MLA_BF16, 1.f, nullptr, out, err};
  const size_t smem = smem_bytes(NT);
  auto kern = head_gemm_kernel<kVup>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return MLA_ERR_CUDA;
  dim3 grid(H, (T + NT - 1) / NT);
  kern<<<grid, kThreads, smem, stream>>>(ta, tb, a);
  return launch_status();
}
