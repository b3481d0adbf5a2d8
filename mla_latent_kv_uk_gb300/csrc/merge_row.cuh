// One warp merges one row of S partial attention states by their LSEs:
//   m = max_s lse_s,  w_s = exp(lse_s - m)  (w_s = 0 for lse_s = -inf),
//   out = sum_s w_s * part_s / sum_s w_s,  out_lse = m + ln(sum_s w_s).
// All parts -inf gives out = 0 and out_lse = -inf.  Parts with weight 0 are
// skipped, so whatever they hold (even NaN) never reaches the output.
#pragma once

#include <cuda_bf16.h>
#include <math.h>

namespace mla {

__device__ __forceinline__ void load8(const __nv_bfloat16 *p, float *v) {
  uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    v[2 * k] = __uint_as_float(w[k] << 16);
    v[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ void load8(const float *p, float *v) {
  float4 a = __ldg(reinterpret_cast<const float4 *>(p));
  float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__device__ __forceinline__ void store8(__nv_bfloat16 *p, const float *v) {
  uint32_t w[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(v[2 * k]));
    uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(v[2 * k + 1]));
    w[k] = lo | (hi << 16);
  }
  *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ void store8(float *p, const float *v) {
  reinterpret_cast<float4 *>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
  reinterpret_cast<float4 *>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}

// part s of the row lives at part0 + s * part_stride (elements); its LSE at
// lse0[s * lse_stride].  D % 8 == 0, D <= 1024.
template <typename Tin, typename Tout>
__device__ __forceinline__ void merge_row(const Tin *part0, int64_t part_stride,
                                          const float *lse0, int64_t lse_stride,
                                          int S, int D, Tout *out,
                                          float *out_lse, int lane) {
  float m = -INFINITY;
  for (int s = lane; s < S; s += 32) m = fmaxf(m, lse0[s * lse_stride]);
#pragma unroll
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const int chunks = D / 8;
  if (m == -INFINITY) {
    float zero[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int c = lane; c < chunks; c += 32) store8(out + c * 8, zero);
    if (out_lse && lane == 0) *out_lse = -INFINITY;
    return;
  }
  float acc[4][8];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[i][e] = 0.f;
  float z = 0.f;
  for (int s = 0; s < S; ++s) {
    const float l = lse0[s * lse_stride];
    if (l == -INFINITY) continue;
    const float w = expf(l - m);
    z += w;
    const Tin *p = part0 + s * part_stride;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int c = lane + 32 * i;
      if (c < chunks) {
        float v[8];
        load8(p + c * 8, v);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[i][e] = fmaf(w, v[e], acc[i][e]);
      }
    }
  }
  const float inv = 1.f / z;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int c = lane + 32 * i;
    if (c < chunks) {
      float v[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] = acc[i][e] * inv;
      store8(out + c * 8, v);
    }
  }
  if (out_lse && lane == 0) *out_lse = m + logf(z);
}

}  // namespace mla
