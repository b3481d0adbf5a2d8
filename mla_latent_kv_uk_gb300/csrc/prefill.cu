// A9: prefill multi-head attention with LSE (run_prefill_new_tokens is the
// causal case, run_prefill_context_chunk the non-causal one).
//
// Source: "DeepSeek MLA 在 DCP 分布式环境中的 Prefill 阶段解析", §Chunked
// Prefill 与 LSE Merge (new tokens attend causally to themselves and return
// the softmax LSE; context chunks are attended without a mask; the two are
// merged by LSE) and §MLA Prefill vs Decode (prefill uses expanded heads:
// QK width 128 + 64 = 192, V width 128).
//
// One CTA per (256 query rows, head, request): two query tiles A and B of
// 128 rows share every K / V tile.  Per 128-key tile and query tile g:
//   S_g = Q_g K^T   tcgen05 M=128 N=128 K=192 (12 MMAs) into TMEM,
//   P_g = exp2(S_g*scale*log2e - m) as bf16 written back over S_g in TMEM,
//   O_g += P_g V    tcgen05 with A = P_g from TMEM, B = V (MN-major).
// The two tiles ping-pong on the tensor core: while one softmax warpgroup
// turns S_A into P_A, the tensor core runs P.V and the next QK of tile B,
// and the other way round, so neither the softmax nor the tensor core waits
// for the other in steady state; each K / V tile is read into the SM once
// for 256 queries.  TMEM: [S_A | O_A | S_B | O_B], 128 columns each.  A
// 2-stage K ring (48 KB tiles: a stage refills once both QKs of its tile
// are done) and one V stage (32 KB, refilled once both P.Vs are done); the
// tiles four ahead are pulled into L2 by tensor prefetches.  Warp 0 = TMA,
// warp 1 = MMA, warps 2..5 = softmax + epilogue of tile A, warps 6..9 of
// tile B (one query row per thread); lazy O rescaling.
#include <cuda_bf16.h>
#include <math.h>

#include "common.cuh"
#include "sm100.cuh"

namespace mla {
namespace {

using namespace sm100;

// L2 prefetch of one tensor-map box (no shared memory, no completion).
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap *map, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z)
               : "memory");
}

constexpr int kBM = 128, kBN = 128;              // query rows per tile, keys per tile
constexpr int kQT = 2;                           // query tiles per CTA
constexpr int kDq = 192, kDv = 128;
constexpr int kBox = 128 * 128;                  // 128 rows x 64 bf16
constexpr int kQBytes = 3 * kBox;                // 48 KB
constexpr int kKBytes = 3 * kBox;                // 48 KB
constexpr int kVBytes = 2 * kBox;                // 32 KB
constexpr int kKStages = 2;
constexpr int kPrefetchAhead = 4;                // tiles pulled into L2 ahead
constexpr int kOffK = kQT * kQBytes;
constexpr int kOffV = kOffK + kKStages * kKBytes;
constexpr int kOffBars = kOffV + kVBytes;
constexpr int kSmemBytes = kOffBars + 256 + 1024;
constexpr int kThreads = 320;
constexpr float kRescaleLog2 = 8.f;
static_assert(kSmemBytes <= 232448, "shared memory of one CTA");

struct PrefillArgs {
  const int32_t *cu_q, *cu_k;
  int H, causal;
  float scale_log2;
  __nv_bfloat16 *out;
  float *lse;
};

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  return bf16x2_rn(a, b);
}

// Key tiles visible to query tile [row0, row0 + rows) of a request with nq
// queries and nk keys (the causal mask aligns the last query with the last key).
__device__ __forceinline__ int tiles_for(int row0, int rows, int nq, int nk, int causal) {
  if (rows <= 0) return 0;
  int key_end = nk;
  if (causal) key_end = min(nk, row0 + rows - 1 + nk - nq + 1);
  key_end = max(key_end, 0);
  return (key_end + kBN - 1) / kBN;
}

// 10 warps: blocks are given registers in units of four warps, so 12 warps'
// worth (at most 168 registers a thread)
__global__ void __launch_bounds__(kThreads, 1)
prefill_kernel(const __grid_constant__ CUtensorMap tm_q,
               const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, PrefillArgs args,
               int *err) {
  const int qp = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int q0 = __ldg(args.cu_q + b), nq = __ldg(args.cu_q + b + 1) - q0;
  const int k0 = __ldg(args.cu_k + b), nk = __ldg(args.cu_k + b + 1) - k0;
  if (qp * kQT * kBM >= nq) return;  // uniform across the CTA: nothing allocated yet
  int rows_g[kQT], nt_g[kQT];
#pragma unroll
  for (int g = 0; g < kQT; ++g) {
    const int row0 = (qp * kQT + g) * kBM;
    rows_g[g] = max(0, min(kBM, nq - row0));
    nt_g[g] = tiles_for(row0, rows_g[g], nq, nk, args.causal);
  }
  const int ntiles = max(nt_g[0], nt_g[1]);

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *sm_q = smem;                        // [kQT] query tiles
  uint8_t *sm_k = smem + kOffK;                // [kKStages] K tiles
  uint8_t *sm_v = smem + kOffV;                // the V tile
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBars);
  uint64_t *k_full = bars, *k_empty = bars + kKStages;
  uint64_t *v_full = bars + 2 * kKStages, *v_empty = v_full + 1;
  uint64_t *s_full = v_empty + 1;              // [kQT]
  uint64_t *p_full = s_full + kQT;             // [kQT]
  uint64_t *pv_done = p_full + kQT;            // [kQT]
  uint64_t *q_full = pv_done + kQT, *drain = q_full + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  const int warp = warp_id(), lane = lane_id();

  if (threadIdx.x == 0) {
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    mbar_init(v_full, 1);
    mbar_init(v_empty, 1);
    for (int g = 0; g < kQT; ++g) {
      mbar_init(&s_full[g], 1);
      mbar_init(&p_full[g], 128);
      mbar_init(&pv_done[g], 1);
    }
    mbar_init(q_full, 1);
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

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------ TMA producer
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    bool ok = true;
    int kt = 0, vt = 0;
    if (ntiles > 0) {
      mbar_arrive_expect_tx(q_full, (rows_g[1] > 0 ? 2 : 1) * kQBytes);
      for (int g = 0; g < kQT; ++g) {
        if (rows_g[g] == 0) continue;
        for (int d = 0; d < 3; ++d)
          tma_load_3d(sm_q + g * kQBytes + d * kBox, &tm_q, q_full, 64 * d, h,
                      q0 + (qp * kQT + g) * kBM);
      }
    }
    auto load_k = [&](int u) -> bool {
      const int s = u % kKStages;
      if (u >= kKStages && !mbar_wait(&k_empty[s], ((u / kKStages) - 1) & 1, abort_flag))
        return false;
      mbar_arrive_expect_tx(&k_full[s], kKBytes);
      const int row = k0 + u * kBN;
      for (int d = 0; d < 3; ++d)
        tma_load_3d(sm_k + s * kKBytes + d * kBox, &tm_k, &k_full[s], 64 * d, h, row);
      // the tiles further ahead go to L2 now (the rings hold one or two)
      for (int a = (u == 0 ? 1 : kPrefetchAhead); a <= kPrefetchAhead; ++a) {
        if (u + a < ntiles) {
          const int prow = k0 + (u + a) * kBN;
          for (int d = 0; d < 3; ++d) tma_prefetch_3d(&tm_k, 64 * d, h, prow);
          for (int d = 0; d < 2; ++d) tma_prefetch_3d(&tm_v, 64 * d, h, prow);
        }
      }
      return true;
    };
    auto load_v = [&](int u) -> bool {
      if (u >= 1 && !mbar_wait(v_empty, (u - 1) & 1, abort_flag)) return false;
      mbar_arrive_expect_tx(v_full, kVBytes);
      const int row = k0 + u * kBN;
      for (int d = 0; d < 2; ++d) tma_load_3d(sm_v + d * kBox, &tm_v, v_full, 64 * d, h, row);
      return true;
    };
    // K(0), K(1), V(0), then per tile t: K(t+1) (its stage frees when both
    // QKs of tile t-1 are done) before V(t) (free when both P.Vs of t-1 are)
    for (; ok && kt < min(ntiles, kKStages); ++kt) ok = load_k(kt);
    for (; ok && vt < ntiles; ++vt) {
      if (vt >= 1 && kt < ntiles && kt == vt + 1) {
        if (!(ok = load_k(kt))) break;
        ++kt;
      }
      if (!(ok = load_v(vt))) break;
    }
    if (*abort_flag) {
      volatile int no_abort = 0;
      for (int k = max(0, kt - kKStages); k < kt; ++k)
        mbar_wait(&k_full[k % kKStages], (k / kKStages) & 1, &no_abort);
      if (vt > 0) mbar_wait(v_full, (vt - 1) & 1, &no_abort);
      if (ntiles > 0) mbar_wait(q_full, 0, &no_abort);
    }
  } else if (warp == 1 && lane == 0) {
    // ----------------------------------------------------------- MMA
    const uint32_t idesc_qk = idesc_bf16(128, kBN, false, false);
    const uint32_t idesc_pv = idesc_bf16(128, kDv, false, true);
    bool ok = ntiles == 0 || mbar_wait(q_full, 0, abort_flag);
    auto issue_qk = [&](int g, int t) {
      const uint32_t qa = smem_u32(sm_q + g * kQBytes);
      const uint32_t kb = smem_u32(sm_k + (t % kKStages) * kKBytes);
      const uint32_t d = tmem + 256 * g;
#pragma unroll
      for (int k = 0; k < kDq / 16; ++k)
        mma_f16_ss(d, sdesc(qa + (k >> 2) * kBox + (k & 3) * 32, 16, 1024, kSwizzle128B),
                   sdesc(kb + (k >> 2) * kBox + (k & 3) * 32, 16, 1024, kSwizzle128B),
                   idesc_qk, k > 0);
      mma_commit(&s_full[g]);
    };
    auto issue_pv = [&](int g, int t) {
      const uint32_t vb = smem_u32(sm_v);
#pragma unroll
      for (int kk = 0; kk < kBN / 16; ++kk)
        mma_f16_ts(tmem + 256 * g + 128, tmem + 256 * g + 8 * kk,
                   sdesc(vb + kk * 2048, kBox, 1024, kSwizzle128B), idesc_pv,
                   (t > 0 || kk > 0) ? 1u : 0u);
      mma_commit(&pv_done[g]);
    };
    // Tile 0's QKs; then per tile t: P.V_A(t), QK_A(t+1), P.V_B(t),
    // QK_B(t+1).  QK_g(t+1) overwrites S_g after P.V_g(t) has read P_g from
    // the same columns (the tensor core runs one thread's MMAs in order).
    if (ok && ntiles > 0 && (ok = mbar_wait(&k_full[0], 0, abort_flag))) {
      tc_fence_after();
      for (int g = 0; g < kQT; ++g)
        if (nt_g[g] > 0) issue_qk(g, 0);
      mma_commit(&k_empty[0]);
    }
    for (int t = 0; ok && t < ntiles; ++t) {
      if (!(ok = mbar_wait(v_full, t & 1, abort_flag))) break;
      bool k_next = false;   // K(t+1) has landed
      for (int g = 0; g < kQT; ++g) {
        if (t < nt_g[g]) {
          if (!(ok = mbar_wait(&p_full[g], t & 1, abort_flag))) break;
          tc_fence_after();
          issue_pv(g, t);
        }
        if (g == kQT - 1) mma_commit(v_empty);   // both P.Vs of tile t issued
        if (t + 1 < nt_g[g]) {
          if (!k_next) {
            if (!(ok = mbar_wait(&k_full[(t + 1) % kKStages], ((t + 1) / kKStages) & 1,
                                 abort_flag)))
              break;
            tc_fence_after();
            k_next = true;
          }
          issue_qk(g, t + 1);
        }
      }
      if (!ok) break;
      if (k_next) mma_commit(&k_empty[(t + 1) % kKStages]);   // both QKs of tile t+1 issued
    }
    if (!ok) {
      mma_commit(drain);
      volatile int no_abort = 0;
      mbar_wait(drain, 0, &no_abort);
    }
  } else if (warp >= 2) {
    // ------------------------------------------- softmax + epilogue of tile g
    const int g = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = tmem + ((quarter * 32u) << 16);
    const uint32_t col_s = 256 * g, col_o = 256 * g + 128;
    const int i = (qp * kQT + g) * kBM + r;         // query index in request
    const int lim = args.causal ? min(nk, i + nk - nq + 1) : nk;
    const int n = nt_g[g];
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int t = 0; t < n; ++t) {
      if (!(ok = mbar_wait(&s_full[g], t & 1, abort_flag))) break;
      tc_fence_after();
      // raw scores; only a tile that crosses this row's limit is masked
      float x[kBN];
#pragma unroll
      for (int c = 0; c < kBN; c += 32) {
        uint32_t v[32];
        tmem_ld_x32(lane_base + col_s + c, v);
#pragma unroll
        for (int k = 0; k < 32; ++k) x[c + k] = __uint_as_float(v[k]);
      }
      if ((t + 1) * kBN > lim) {
#pragma unroll
        for (int k = 0; k < kBN; ++k) x[k] = t * kBN + k < lim ? x[k] : -INFINITY;
      }
      // tile max on the raw scores (four chains), scaled once: scaling by a
      // positive constant keeps the order and rounds each value alike
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int k = 0; k < kBN; k += 2) mx[(k >> 1) & 3] = fmax3(mx[(k >> 1) & 3], x[k], x[k + 1]);
      const float tmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * args.scale_log2;
      if (t > 0) {
        const float m_new = fmaxf(m, tmax);
        const bool need = m_new > m + kRescaleLog2 || (m == -INFINITY && m_new > -INFINITY);
        if (__any_sync(0xffffffffu, need)) {
          // rescale only after P.V(t-1) landed; the barrier is never more
          // than one phase ahead of this wait (P.V(t) needs this tile's P)
          if (!(ok = mbar_wait(&pv_done[g], (t - 1) & 1, abort_flag))) break;
          tc_fence_after();
          const float alpha = need ? (m == -INFINITY ? 0.f : ex2(m - m_new)) : 1.f;
#pragma unroll 1
          for (int c = 0; c < kDv; c += 32) {
            uint32_t o[32];
            tmem_ld_x32(lane_base + col_o + c, o);
#pragma unroll
            for (int k = 0; k < 32; ++k)
              o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
            tmem_st_x32(lane_base + col_o + c, o);
          }
          l *= alpha;
          if (need) m = m_new;
        }
      } else {
        m = tmax;
      }
      const float ms = m == -INFINITY ? 0.f : m;
      // p = 2^(s * scale - m): paired FMAs, then the hardware ex2; the row
      // sum of the unrounded probabilities (see the decode kernel) in four
      // chains of paired adds
      const float nm = -ms, sc = args.scale_log2;
#pragma unroll
      for (int k = 0; k < kBN; k += 2) fma_f32x2(x[k], x[k + 1], x[k], x[k + 1], sc, sc, nm, nm);
#pragma unroll
      for (int k = 0; k < kBN; ++k) x[k] = ex2(x[k]);
      float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int k = 0; k < kBN; k += 4) {
        add_f32x2(ps[0], ps[1], ps[0], ps[1], x[k], x[k + 1]);
        add_f32x2(ps[2], ps[3], ps[2], ps[3], x[k + 2], x[k + 3]);
      }
      const float psum = (ps[0] + ps[1]) + (ps[2] + ps[3]);
#pragma unroll
      for (int c = 0; c < kBN; c += 64) {
        uint32_t pk[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) pk[k] = pack2(x[c + 2 * k], x[c + 2 * k + 1]);
        tmem_st_x32(lane_base + col_s + c / 2, pk);
      }
      l += psum;
      tc_fence_before();
      mbar_arrive(&p_full[g]);
    }
    if (ok && n > 0) ok = mbar_wait(&pv_done[g], (n - 1) & 1, abort_flag);
    tc_fence_after();
    if (ok && rows_g[g] > 0) {
      const bool row_ok = r < rows_g[g];
      const int64_t orow = static_cast<int64_t>(q0 + i) * args.H + h;
      const bool empty = !(l > 0.f);
      const float inv = empty ? 0.f : 1.f / l;
#pragma unroll 1
      for (int c = 0; c < kDv; c += 32) {
        uint32_t o[32];
        if (n > 0) tmem_ld_x32(lane_base + col_o + c, o);
        if (!row_ok) continue;
        uint4 *dst = reinterpret_cast<uint4 *>(args.out + orow * kDv + c);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          float v[8];
#pragma unroll
          for (int e = 0; e < 8; ++e)
            v[e] = (n > 0 && !empty) ? __uint_as_float(o[8 * k + e]) * inv : 0.f;
          dst[k] = make_uint4(pack2(v[0], v[1]), pack2(v[2], v[3]), pack2(v[4], v[5]),
                              pack2(v[6], v[7]));
        }
      }
      if (row_ok)
        args.lse[orow] = empty ? -INFINITY : (m + log2f(l)) * 0.69314718055994531f;
    }
    tc_fence_before();
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

extern "C" int mla_prefill_attn(const void *q, const void *k, const void *v,
                                const int32_t *cu_q, const int32_t *cu_k,
                                int B, int Tq, int Nk, int H, int max_q_len,
                                int causal, float sm_scale, void *out,
                                float *lse, mla_stream_t stream) {
  if (B < 1 || Tq < 0 || Nk < 0 || H < 1 || H > 65535 || max_q_len < 0 || B > 65535)
    return MLA_ERR_INVALID_ARG;
  if (!(sm_scale > 0.f) || !(sm_scale < INFINITY)) return MLA_ERR_INVALID_ARG;
  if (Tq == 0 || max_q_len == 0) return MLA_OK;
  if (!q || !k || !v || !cu_q || !cu_k || !out || !lse) return MLA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return MLA_ERR_INVALID_ARG;
  int *err = device_error_word();
  if (!err) return MLA_ERR_CUDA;
  CUtensorMap tq, tk, tv;
  const uint32_t box[3] = {64, 1, 128};
  {
    const uint64_t dims[3] = {kDq, static_cast<uint64_t>(H), static_cast<uint64_t>(Tq)};
    const uint64_t strides[2] = {kDq * 2, static_cast<uint64_t>(H) * kDq * 2};
    if (!make_tmap(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q, dims, strides, box,
                   CU_TENSOR_MAP_SWIZZLE_128B))
      return MLA_ERR_CUDA;
  }
  const uint64_t nk_rows = Nk > 0 ? static_cast<uint64_t>(Nk) : 1;
  {
    const uint64_t dims[3] = {kDq, static_cast<uint64_t>(H), nk_rows};
    const uint64_t strides[2] = {kDq * 2, static_cast<uint64_t>(H) * kDq * 2};
    if (!make_tmap(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, k, dims, strides, box,
                   CU_TENSOR_MAP_SWIZZLE_128B))
      return MLA_ERR_CUDA;
  }
  {
    const uint64_t dims[3] = {kDv, static_cast<uint64_t>(H), nk_rows};
    const uint64_t strides[2] = {kDv * 2, static_cast<uint64_t>(H) * kDv * 2};
    if (!make_tmap(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, v, dims, strides, box,
                   CU_TENSOR_MAP_SWIZZLE_128B))
      return MLA_ERR_CUDA;
  }
  PrefillArgs a{cu_q, cu_k, H, causal ? 1 : 0, sm_scale * 1.4426950408889634f,
                static_cast<__nv_bfloat16 *>(out), lse};
  if (cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kSmemBytes) != cudaSuccess)
    return MLA_ERR_CUDA;
  dim3 grid((max_q_len + kQT * kBM - 1) / (kQT * kBM), H, B);
  prefill_kernel<<<grid, kThreads, kSmemBytes, stream>>>(tq, tk, tv, a, err);
  return launch_status();
}
