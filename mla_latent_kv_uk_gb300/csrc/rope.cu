// Before the decode path: rotary position embedding of the query's rope
// slice and of k_pe, and the store of the new tokens' latent rows
// kv_c ‖ rope(k_pe) into the paged cache.
//
// Sources: prhub digest of vLLM PR 45964, §关键源码片段 mla.py (rotary_emb is
// applied to q[..., qk_nope_head_dim:] and k_pe before mla_attn); "DeepSeek
// MLA 在 DCP 分布式环境中的 Prefill 阶段解析", §Chunked Prefill 与 LSE Merge
// (the new tokens' KV is in the cache when attention runs).  The rotation is
// RoFormer's rotary embedding (Su et al. 2021): pair i of a 64-wide vector
// turns by position * base^(-2i/64).
//
// Grid (new tokens, blocks of 32 query heads), 128 threads: each CTA
// computes its token's 32 angles in fp64 (one thread per pair, sincos in
// double) and keeps them as fp32 cos / sin in shared memory, then every
// 16-byte chunk of its 32 query heads is handled by one thread (loads and
// stores of 16 bytes, the rotation in fp32, one bf16 rounding); the first
// head block of a token also rotates k_pe and writes the cache row.  The
// kernel is a stream of the tokens' bytes (q_pe in and out, kv_c and k_pe in,
// one cache row out), bound by memory latency at decode batch sizes, hence
// the spread of each token over several CTAs.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <math.h>

#include <cmath>

#include "common.cuh"
#include "sm100.cuh"

namespace mla {
namespace {

constexpr int kRopeThreads = 128;
constexpr int kHeadsPerCta = 32;
constexpr int kPairs = kRope / 2;   // 32

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf(float lo, float hi) { return sm100::bf16x2_rn(lo, hi); }

// (a, b) turned by the angle whose cosine / sine are c, s, in fp32 with one
// fused rounding per output.
__device__ __forceinline__ void rot(float a, float b, float c, float s, float &ra, float &rb) {
  ra = fmaf(a, c, -(b * s));
  rb = fmaf(a, s, b * c);
}

// 8 consecutive dims starting at dim 8*chunk of one interleaved-layout
// vector: pairs 4*chunk .. 4*chunk + 3.
__device__ __forceinline__ uint4 rot_interleaved(uint4 v, int chunk, const float *cs, const float *sn) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int i = 4 * chunk + k;
    float ra, rb;
    rot(bf_lo(w[k]), bf_hi(w[k]), cs[i], sn[i], ra, rb);
    o[k] = pack_bf(ra, rb);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Rotate-half layout: dims 8*chunk .. 8*chunk+7 (a) with dims
// 32 + 8*chunk .. (b), pairs 8*chunk + k.
__device__ __forceinline__ void rot_half(uint4 &va, uint4 &vb, int chunk, const float *cs,
                                         const float *sn) {
  const uint32_t wa[4] = {va.x, va.y, va.z, va.w}, wb[4] = {vb.x, vb.y, vb.z, vb.w};
  uint32_t oa[4], ob[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int i0 = 8 * chunk + 2 * k, i1 = i0 + 1;
    float a0, b0, a1, b1;
    rot(bf_lo(wa[k]), bf_lo(wb[k]), cs[i0], sn[i0], a0, b0);
    rot(bf_hi(wa[k]), bf_hi(wb[k]), cs[i1], sn[i1], a1, b1);
    oa[k] = pack_bf(a0, a1);
    ob[k] = pack_bf(b0, b1);
  }
  va = make_uint4(oa[0], oa[1], oa[2], oa[3]);
  vb = make_uint4(ob[0], ob[1], ob[2], ob[3]);
}

// Eight bf16 values -> eight e4m3 codes of value / k_scale (RNE, saturating).
__device__ __forceinline__ uint2 to_e4m3(uint4 v, float k_scale) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
        make_float2(bf_lo(w[2 * k]) / k_scale, bf_hi(w[2 * k]) / k_scale), __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
        make_float2(bf_lo(w[2 * k + 1]) / k_scale, bf_hi(w[2 * k + 1]) / k_scale), __NV_SATFINITE,
        __NV_E4M3);
    o[k] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
  }
  return make_uint2(o[0], o[1]);
}

__global__ void __launch_bounds__(kRopeThreads)
rope_cache_kernel(uint4 *__restrict__ q_pe, uint4 *__restrict__ k_pe,
                  const uint4 *__restrict__ kv_c, const int32_t *__restrict__ positions,
                  const int32_t *__restrict__ slot_mapping, int H, double log2_base, int half_layout,
                  uint8_t *__restrict__ kv_cache, int fp8, float k_scale, int64_t num_slots,
                  int *err) {
  __shared__ float cs[kPairs], sn[kPairs];
  __shared__ int64_t slot_s;
  const int t = blockIdx.x, hb = blockIdx.y, tid = threadIdx.x;
  if (tid < kPairs) {
    // theta_i = base^(-2i/64); the angle and its sine / cosine in fp64
    const double ang = static_cast<double>(positions[t]) * exp2(-(2.0 * tid / kRope) * log2_base);
    double s, c;
    sincos(ang, &s, &c);
    cs[tid] = static_cast<float>(c);
    sn[tid] = static_cast<float>(s);
  }
  if (tid == kPairs && hb == 0) {
    int64_t slot = slot_mapping[t];
    if (slot >= num_slots) {
      raise_error(err, MLA_DEVERR_BLOCK_ID);
      slot = -1;
    }
    slot_s = slot;
  }
  __syncthreads();
  // this CTA's query heads: rope rows of 128 B = 8 chunks
  if (q_pe) {
    const int h0 = hb * kHeadsPerCta, nh = min(kHeadsPerCta, H - h0);
    uint4 *qt = q_pe + (static_cast<int64_t>(t) * H + h0) * 8;
    if (!half_layout) {
      for (int i = tid; i < nh * 8; i += kRopeThreads)
        qt[i] = rot_interleaved(qt[i], i & 7, cs, sn);
    } else {
      for (int i = tid; i < nh * 4; i += kRopeThreads) {
        uint4 *row = qt + (i >> 2) * 8;
        const int c = i & 3;
        uint4 va = row[c], vb = row[c + 4];
        rot_half(va, vb, c, cs, sn);
        row[c] = va;
        row[c + 4] = vb;
      }
    }
  }
  if (hb != 0) return;   // k_pe and the cache row: the token's first head block
  const int64_t slot = slot_s;
  uint8_t *dst_row = slot >= 0 ? kv_cache + slot * (fp8 ? kDqk : kDqk * 2) : nullptr;
  // k_pe (in place) and the rope part of the cache row
  uint4 *kt = k_pe + static_cast<int64_t>(t) * 8;
  auto store_rope = [&](int chunk, uint4 v) {
    if (!dst_row) return;
    if (fp8) reinterpret_cast<uint2 *>(dst_row + kLatent)[chunk] = to_e4m3(v, k_scale);
    else reinterpret_cast<uint4 *>(dst_row + kLatent * 2)[chunk] = v;
  };
  if (!half_layout) {
    if (tid < 8) {
      const uint4 v = rot_interleaved(kt[tid], tid, cs, sn);
      kt[tid] = v;
      store_rope(tid, v);
    }
  } else if (tid < 4) {
    uint4 va = kt[tid], vb = kt[tid + 4];
    rot_half(va, vb, tid, cs, sn);
    kt[tid] = va;
    kt[tid + 4] = vb;
    store_rope(tid, va);
    store_rope(tid + 4, vb);
  }
  // kv_c: 64 chunks of 8 bf16
  if (dst_row && tid >= 64) {
    const int c = tid - 64;
    const uint4 v = kv_c[static_cast<int64_t>(t) * 64 + c];
    if (fp8) reinterpret_cast<uint2 *>(dst_row)[c] = to_e4m3(v, k_scale);
    else reinterpret_cast<uint4 *>(dst_row)[c] = v;
  }
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" int mla_rope_cache_write(void *q_pe, void *k_pe, const void *kv_c,
                                    const int32_t *positions, const int32_t *slot_mapping,
                                    int T, int H, float rope_base, int rope_layout,
                                    void *kv_cache, int kv_dtype, float k_scale, int num_blocks,
                                    mla_stream_t stream) {
  if (T < 0 || (q_pe && (H < 1 || H > 4096)) || num_blocks < 1 || num_blocks >= (1 << 25))
    return MLA_ERR_INVALID_ARG;
  if (rope_layout != MLA_ROPE_INTERLEAVED && rope_layout != MLA_ROPE_HALF)
    return MLA_ERR_INVALID_ARG;
  if (!(rope_base > 1.f) || !(rope_base < INFINITY)) return MLA_ERR_INVALID_ARG;
  if (kv_dtype != MLA_BF16 && kv_dtype != MLA_E4M3) return MLA_ERR_INVALID_ARG;
  if (kv_dtype == MLA_E4M3 && (!(k_scale > 0.f) || !(k_scale < INFINITY)))
    return MLA_ERR_INVALID_ARG;
  if (T == 0) return MLA_OK;
  if (!k_pe || !kv_c || !positions || !slot_mapping || !kv_cache) return MLA_ERR_INVALID_ARG;
  if ((q_pe && !aligned16(q_pe)) || !aligned16(k_pe) || !aligned16(kv_c) || !aligned16(kv_cache))
    return MLA_ERR_INVALID_ARG;
  int *err = device_error_word();
  if (!err) return MLA_ERR_CUDA;
  const dim3 grid(T, q_pe ? (H + kHeadsPerCta - 1) / kHeadsPerCta : 1);
  rope_cache_kernel<<<grid, kRopeThreads, 0, stream>>>(
      static_cast<uint4 *>(q_pe), static_cast<uint4 *>(k_pe), static_cast<const uint4 *>(kv_c),
      positions, slot_mapping, H, std::log2(static_cast<double>(rope_base)),
      rope_layout == MLA_ROPE_HALF ? 1 : 0, static_cast<uint8_t *>(kv_cache),
      kv_dtype == MLA_E4M3 ? 1 : 0, k_scale, static_cast<int64_t>(num_blocks) * kPage, err);
  return launch_status();
}
