// A1/A2 query absorption (+ concat, + optional e4m3 quantisation) and A6
// value up-projection: per-head GEMMs on the 5th-generation tensor cores.
//
// Both are small per-head contractions whose cost is reading the weights
// (W_UK_T / W_UV: H x 128 x 512 bf16 = 16 MiB at H = 128), so the kernels
// are built to keep a whole per-head weight slice in flight: TMA streams it
// into 128B-swizzled shared memory, one thread issues tcgen05.mma (M = 128,
// N = token tile, K = 16) into TMEM, and four epilogue warps move the
// accumulator through a shared-memory staging tile so that every output
// row leaves as coalesced 16-byte stores.
//
//   absorb: ql^T[l, t] = sum_p W_UK_T[h][p, l] * q_nope[t, h, p]
//           one CTA per (head, 256-wide latent half, <=256-token tile):
//           two M=128 accumulators, A = W_UK_T[h] (MN-major, l contiguous),
//           B = q_nope (K-major); all 64 KB of weights requested up front.
//   v_up:   out^T[v, t] = sum_l W_UV[h][v, l] * o_lat[t, h, l]
//           one CTA per (head, token tile): A = W_UV[h] (K-major), B = o_lat
//           (K-major), K = 512 streamed through a ring up to 8 deep.
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

constexpr int kThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int kBoxBytes64 = 64 * 128;   // 64 rows x 64 bf16 (8 KB)
constexpr int kStageTokens = 32;        // epilogue staging granularity

struct GemmArgs {
  int T, H, NT;            // tokens, heads, token tile (multiple of 16)
  int out_dtype;           // absorb: MLA_BF16 / MLA_E4M3 / MLA_F32
  float q_scale;
  const __nv_bfloat16 *q_pe;  // absorb only
  void *out;
  int *err;
};

__device__ __forceinline__ int esize(int dtype) {
  return dtype == MLA_F32 ? 4 : dtype == MLA_BF16 ? 2 : 1;
}

// Writes v (the fp32 value) in `dtype` at byte address p.
__device__ __forceinline__ void put(uint8_t *p, int dtype, float v, float q_scale) {
  if (dtype == MLA_BF16) {
    *reinterpret_cast<__nv_bfloat16 *>(p) = __float2bfloat16_rn(v);
  } else if (dtype == MLA_F32) {
    *reinterpret_cast<float *>(p) = v;
  } else {
    // e4m3 of the correctly rounded fp32 quotient: RNE, saturate to 448
    *reinterpret_cast<__nv_fp8_storage_t *>(p) =
        __nv_cvt_float_to_fp8(__fdiv_rn(v, q_scale), __NV_SATFINITE, __NV_E4M3);
  }
}

__device__ __forceinline__ void epi_bar() {
  asm volatile("bar.sync 1, 128;" ::: "memory");
}

__host__ __device__ inline uint32_t tmem_cols_for(int n) {
  return n <= 32 ? 32 : n <= 64 ? 64 : n <= 128 ? 128 : 256;
}

// ------------------------------------------------------------------ absorb
// One CTA per (head, 128-wide latent block, token tile): four per head, so
// the 16 MiB of weights spread over all SMs in 32 KB pieces and the work
// left after a CTA's data lands (8 MMAs and one store) is short.
constexpr int kAbsorbLat = 128;                       // latent columns per CTA
constexpr int kAbsorbBlocks = kLatent / kAbsorbLat;   // CTAs per head
constexpr int kAbsorbBoxes = 2 * kAbsorbLat / 64;     // W boxes: 2 K-chunks x l-blocks
// smem: A [2 K-chunks][2 l-blocks] of {64 l x 64 p} boxes (32 KB; once the
//       MMAs are done it stages the output), B [2 K-chunks] of {64 p x NT t}
//       (NT * 128 B each), the q_pe tile {64 x NT t} (last latent block
//       only; room for NT rounded up to 32 rows, as its chunks are stored
//       whole).
// The output leaves through tensor-map stores: per 32-token chunk one box
// of this CTA's 128 latent columns and, for the last block, one of the 64
// rope columns (straight from the q_pe tile when the output is bf16).
__global__ void __launch_bounds__(kThreads, 4)   // four CTAs (and their TMEM) per SM
absorb_kernel(const __grid_constant__ CUtensorMap tm_w,
              const __grid_constant__ CUtensorMap tm_q,
              const __grid_constant__ CUtensorMap tm_qpe,
              const __grid_constant__ CUtensorMap tm_out,
              const __grid_constant__ CUtensorMap tm_out_pe, GemmArgs args) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int NT = args.NT;
  uint8_t *sm_a = smem;                          // 32 KB
  uint8_t *sm_b = smem + kAbsorbBoxes * kBoxBytes64;   // 2 * NT * 128
  uint8_t *sm_pe = sm_b + 2 * NT * 128;          // round_up(NT, 32) * 128
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm_pe + ((NT + 31) / 32) * 32 * 128);
  uint64_t *full = bars, *done = bars + 1, *drain = bars + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 3);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  volatile int *go = abort_flag + 1;             // the epilogue's common decision

  const int warp = warp_id(), lane = lane_id();
  const int mq = blockIdx.x;          // latent block: l in [128 mq, 128 mq + 128)
  const bool rope = mq == kAbsorbBlocks - 1;   // this CTA also writes the rope columns
  const int h = blockIdx.y;
  const int t0 = blockIdx.z * NT;
  const int ntok = min(NT, args.T - t0);
  const uint32_t cols = tmem_cols_for(NT);

  if (threadIdx.x == 0) {
    mbar_init(full, 1);
    mbar_init(done, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // launched with programmatic stream serialization: the prologue above
  // overlaps the previous kernel; every global read comes after this wait
  grid_dep_wait();
  grid_dep_launch();

  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_w);
    prefetch_tmap(&tm_q);
    mbar_arrive_expect_tx(full, kAbsorbBoxes * kBoxBytes64 + 2 * NT * 128 + (rope ? NT * 128 : 0));
    // the weights are read once per step: their lines leave L2 first, so
    // the absorbed query written here is still there for the decode
    const uint64_t w_policy = l2_evict_first_policy();
    for (int kc = 0; kc < 2; ++kc) {
      for (int lb = 0; lb < 2; ++lb)   // W_UK_T as [H*128 rows (p), 512 cols (l)]
        tma_load_2d_hint(sm_a + (kc * 2 + lb) * kBoxBytes64, &tm_w, full,
                         kAbsorbLat * mq + 64 * lb, h * 128 + 64 * kc, w_policy);
      tma_load_3d(sm_b + kc * NT * 128, &tm_q, full, 64 * kc, h, t0);
    }
    if (rope) tma_load_3d(sm_pe, &tm_qpe, full, 0, h, t0);
    if (!mbar_wait(full, 0, abort_flag)) {
      volatile int no_abort = 0;
      mbar_wait(full, 0, &no_abort);
    }
  } else if (warp == 1 && lane == 0) {
    const uint32_t idesc = idesc_bf16(128, NT, true, false);
    const bool ok = mbar_wait(full, 0, abort_flag);
    if (ok) {
      tc_fence_after();
      const uint32_t a = smem_u32(sm_a), b = smem_u32(sm_b);
#pragma unroll
      for (int kc = 0; kc < 2; ++kc)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          // MN-major A: 128 B rows = 64 l of one p; 8-p groups 1024 B apart
          // (SBO); the two 64-l blocks of the M = 128 block one box apart (LBO)
          const uint64_t adesc = sdesc(a + kc * 2 * kBoxBytes64 + kk * 2048, kBoxBytes64, 1024,
                                       kSwizzle128B);
          const uint64_t bdesc = sdesc(b + kc * NT * 128 + kk * 32, 16, 1024, kSwizzle128B);
          mma_f16_ss(tmem, adesc, bdesc, idesc, (kc | kk) != 0);
        }
    }
    mma_commit(ok ? done : drain);
    if (!ok) {
      volatile int no_abort = 0;
      mbar_wait(drain, 0, &no_abort);
    }
  } else if (warp >= 2) {
    const int tid = threadIdx.x - 64;
    const int quarter = warp & 3;
    const int lrow = quarter * 32 + lane;       // latent row within the block
    const int dt = args.out_dtype, es = esize(dt);
    mbar_wait(done, 0, abort_flag);
    // one decision for all four warps (a timed-out wait has set the flag
    // before this barrier), so none is left alone at the barriers below
    epi_bar();
    if (tid == 0) *go = *abort_flag ? 0 : 1;
    epi_bar();
    tc_fence_after();
    if (*go) {
      // the MMAs have read A and B: A's 32 KB hold the staging
      uint8_t *stg = sm_a;                      // [32 t][128 l] in the output dtype
      uint8_t *stg_pe = sm_a + kStageTokens * kAbsorbLat * 4;   // [32 t][64]
      for (int c0 = 0; c0 < ntok; c0 += kStageTokens) {
        if (c0 > 0) {   // the previous chunk's stores have read the staging
          if (tid == 0) bulk_wait_read_all();
          epi_bar();
        }
        {
          uint32_t r[32];
          tmem_ld_x32(tmem_addr(tmem, warp, c0), r);
#pragma unroll
          for (int c = 0; c < 32; ++c)
            put(stg + (c * kAbsorbLat + lrow) * es, dt, __uint_as_float(r[c]), args.q_scale);
        }
        if (rope && dt != MLA_BF16) {
          // rope columns in the output dtype (bf16 leaves from its own tile)
          for (int i = tid; i < kStageTokens * 64; i += 128) {
            const int t = i >> 6, c = i & 63;
            const uint32_t raw = reinterpret_cast<const uint16_t *>(sm_pe + (c0 + t) * 128)[c];
            put(stg_pe + (t * 64 + c) * es, dt, __uint_as_float(raw << 16), args.q_scale);
          }
        }
        fence_proxy_async_smem();
        epi_bar();
        if (tid == 0) {
          tma_store_3d(&tm_out, stg, kAbsorbLat * mq, h, t0 + c0);
          if (rope)
            tma_store_3d(&tm_out_pe, dt == MLA_BF16 ? sm_pe + c0 * 128 : stg_pe, kLatent, h,
                         t0 + c0);
        }
      }
      // the stores have completed before this CTA's shared memory is released
      if (tid == 0) bulk_wait_all();
    }
    tc_fence_before();
  }
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) raise_error(args.err, MLA_DEVERR_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, cols);
  }
}

// -------------------------------------------------------------------- v_up
// smem: ring of stages {A: 64 l x 128 v (16 KB), B: 64 l x NT t}, staging.
__global__ void __launch_bounds__(kThreads, 1)
vup_kernel(const __grid_constant__ CUtensorMap tm_w,
           const __grid_constant__ CUtensorMap tm_o, GemmArgs args, int stages) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int KC = 512 / 64;
  const int NT = args.NT;
  const int a_bytes = 128 * 128, stage_bytes = a_bytes + NT * 128;
  uint8_t *sm_o = smem + stages * stage_bytes;          // 32 tokens x 256 B
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm_o + kStageTokens * 256);
  uint64_t *full = bars, *empty = bars + 8, *done = bars + 16, *drain = bars + 17;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 18);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  volatile int *go = abort_flag + 1;             // the epilogue's common decision
  const int warp = warp_id(), lane = lane_id();
  const int h = blockIdx.x;
  const int t0 = blockIdx.y * NT;
  const int ntok = min(NT, args.T - t0);
  const uint32_t cols = tmem_cols_for(NT);

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // launched with programmatic stream serialization: the prologue above
  // overlaps the previous kernel; every global read comes after this wait
  grid_dep_wait();
  grid_dep_launch();

  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_w);
    prefetch_tmap(&tm_o);
    int armed = -1;
    // the weights are read once: their lines leave L2 before the latent
    // output this kernel reads alongside them
    const uint64_t w_policy = l2_evict_first_policy();
    for (int kc = 0; kc < KC; ++kc) {
      const int s = kc % stages;
      if (kc >= stages && !mbar_wait(&empty[s], ((kc / stages) - 1) & 1, abort_flag)) break;
      uint8_t *dst = smem + s * stage_bytes;
      mbar_arrive_expect_tx(&full[s], stage_bytes);
      tma_load_2d_hint(dst, &tm_w, &full[s], kc * 64, h * 128, w_policy);  // W_UV [H*128 (v), 512 (l)]
      tma_load_3d(dst + a_bytes, &tm_o, &full[s], kc * 64, h, t0);
      armed = kc;
    }
    if (*abort_flag) {
      volatile int no_abort = 0;
      for (int kc = max(0, armed - stages + 1); kc <= armed; ++kc)
        mbar_wait(&full[kc % stages], (kc / stages) & 1, &no_abort);
    }
  } else if (warp == 1 && lane == 0) {
    const uint32_t idesc = idesc_bf16(128, NT, false, false);
    bool ok = true;
    for (int kc = 0; kc < KC; ++kc) {
      const int s = kc % stages;
      if (!(ok = mbar_wait(&full[s], (kc / stages) & 1, abort_flag))) break;
      tc_fence_after();
      const uint32_t a = smem_u32(smem + s * stage_bytes), b = a + a_bytes;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_f16_ss(tmem, sdesc(a + kk * 32, 16, 1024, kSwizzle128B),
                   sdesc(b + kk * 32, 16, 1024, kSwizzle128B), idesc, (kc | kk) != 0);
      mma_commit(&empty[s]);
    }
    mma_commit(ok ? done : drain);
    if (!ok) {
      volatile int no_abort = 0;
      mbar_wait(drain, 0, &no_abort);
    }
  } else if (warp >= 2) {
    const int tid = threadIdx.x - 64;
    const int v = (warp & 3) * 32 + lane;
    mbar_wait(done, 0, abort_flag);
    // one decision for all four warps (a timed-out wait has set the flag
    // before this barrier), so none is left alone at the barriers below
    epi_bar();
    if (tid == 0) *go = *abort_flag ? 0 : 1;
    epi_bar();
    tc_fence_after();
    if (*go) {
      for (int c0 = 0; c0 < ntok; c0 += kStageTokens) {
        uint32_t r[32];
        tmem_ld_x32(tmem_addr(tmem, warp, c0), r);
#pragma unroll
        for (int c = 0; c < 32; ++c)
          reinterpret_cast<__nv_bfloat16 *>(sm_o + c * 256)[v] =
              __float2bfloat16_rn(__uint_as_float(r[c]));
        epi_bar();
        const int nt = min(kStageTokens, ntok - c0);
        for (int i = tid; i < nt * 16; i += 128) {
          const int t = t0 + c0 + i / 16, c = i % 16;
          reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(args.out) +
                                    (static_cast<int64_t>(t) * args.H + h) * kVhead)[c] =
              reinterpret_cast<const uint4 *>(sm_o + (i / 16) * 256)[c];
        }
        epi_bar();
      }
    }
    tc_fence_before();
  }
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) raise_error(args.err, MLA_DEVERR_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, cols);
  }
}

int token_tile(int T) {
  int nt = ((T + 15) / 16) * 16;
  return nt > 256 ? 256 : nt;
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
  if (!aligned16(q_nope) || !aligned16(q_pe) || !aligned16(w_uk_t) || !aligned16(q_out))
    return MLA_ERR_INVALID_ARG;
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
  // q_pe [T, H, 64] rows in, and the output [T, H, 576] in boxes of 32
  // tokens x (256 latent | 64 rope) columns out, no swizzle
  CUtensorMap tpe, to_lat, to_pe;
  {
    const uint64_t dims[3] = {static_cast<uint64_t>(kRope), static_cast<uint64_t>(H),
                              static_cast<uint64_t>(T)};
    const uint64_t strides[2] = {kRope * 2, static_cast<uint64_t>(H) * kRope * 2};
    const uint32_t box[3] = {static_cast<uint32_t>(kRope), 1, static_cast<uint32_t>(NT)};
    if (!make_tmap(&tpe, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q_pe, dims, strides, box,
                   CU_TENSOR_MAP_SWIZZLE_NONE))
      return MLA_ERR_CUDA;
  }
  {
    const uint64_t es = out_dtype == MLA_F32 ? 4 : out_dtype == MLA_BF16 ? 2 : 1;
    const CUtensorMapDataType tdt = out_dtype == MLA_F32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                    : out_dtype == MLA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                            : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    const uint64_t dims[3] = {static_cast<uint64_t>(kDqk), static_cast<uint64_t>(H),
                              static_cast<uint64_t>(T)};
    const uint64_t strides[2] = {kDqk * es, static_cast<uint64_t>(H) * kDqk * es};
    const uint32_t box_lat[3] = {kAbsorbLat, 1, static_cast<uint32_t>(kStageTokens)};
    const uint32_t box_pe[3] = {static_cast<uint32_t>(kRope), 1,
                                static_cast<uint32_t>(kStageTokens)};
    if (!make_tmap(&to_lat, tdt, 3, q_out, dims, strides, box_lat, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_tmap(&to_pe, tdt, 3, q_out, dims, strides, box_pe, CU_TENSOR_MAP_SWIZZLE_NONE))
      return MLA_ERR_CUDA;
  }
  GemmArgs a{T, H, NT, out_dtype, q_scale,
             static_cast<const __nv_bfloat16 *>(q_pe), q_out, err};
  const size_t smem =
      1024 + kAbsorbBoxes * kBoxBytes64 + 2 * NT * 128 + ((NT + 31) / 32) * 32 * 128 + 64;
  if (cudaFuncSetAttribute(absorb_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return MLA_ERR_CUDA;
  dim3 grid(kAbsorbBlocks, H, (T + NT - 1) / NT);
  if (launch_pdl(absorb_kernel, grid, dim3(kThreads), smem, stream, ta, tb, tpe, to_lat, to_pe,
                 a) != cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}

extern "C" int mla_v_up(const void *o_lat, const void *w_uv, int T, int H,
                        void *out, mla_stream_t stream) {
  if (T < 0 || H < 1 || H > 4096) return MLA_ERR_INVALID_ARG;
  if (T == 0) return MLA_OK;
  if (!o_lat || !w_uv || !out) return MLA_ERR_INVALID_ARG;
  if (!aligned16(o_lat) || !aligned16(w_uv) || !aligned16(out)) return MLA_ERR_INVALID_ARG;
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
  const int stage_bytes = 128 * 128 + NT * 128;
  int stages = (200 * 1024) / stage_bytes;
  stages = stages > 8 ? 8 : stages;
  const size_t smem = 1024 + static_cast<size_t>(stages) * stage_bytes + kStageTokens * 256 + 256;
  if (cudaFuncSetAttribute(vup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return MLA_ERR_CUDA;
  dim3 grid(H, (T + NT - 1) / NT);
  if (launch_pdl(vup_kernel, grid, dim3(kThreads), smem, stream, ta, tb, a, stages) != cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}
