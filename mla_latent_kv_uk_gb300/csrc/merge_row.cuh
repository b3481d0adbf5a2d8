// One warp merges one row of S partial attention states by their LSEs:
//   m = max_s lse_s,  w_s = exp(lse_s - m)  (w_s = 0 for lse_s = -inf),
//   out = sum_s w_s * part_s / sum_s w_s,  out_lse = m + ln(sum_s w_s).
// All parts -inf gives out = 0 and out_lse = -inf.  Parts with weight 0 are
// skipped, so whatever they hold (even NaN) never reaches the output.
#pragma once

#include <cuda_bf16.h>
#include <math.h>

#include "sm100.cuh"

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
  for (int k = 0; k < 4; ++k) w[k] = sm100::bf16x2_rn(v[2 * k], v[2 * k + 1]);
  *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ void store8(float *p, const float *v) {
  reinterpret_cast<float4 *>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
  reinterpret_cast<float4 *>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}

// part s of the row lives at part0 + s * part_stride (elements); its LSE at
// lse0[s * lse_stride].  D % 8 == 0, D <= 256 * NC (NC 16-byte chunk slots
// per lane).
//
// Latency layout: up to four parts cost one round of loads (LSEs and rows
// together); beyond that lane s holds the LSE of part s (32 parts per pass),
// the weights come from shuffles, and the row data of up to four parts is
// requested before any of it is used, so a row costs a few L2 round trips
// instead of two per part.
template <typename Tin, typename Tout, int NC = 4>
__device__ __forceinline__ void merge_row(const Tin *part0, int64_t part_stride,
                                          const float *lse0, int64_t lse_stride,
                                          int S, int D, Tout *out,
                                          float *out_lse, int lane) {
  if (S <= 4) {
    // Few parts (the usual split): the LSEs and every part's row go out in
    // one round of loads; a part of weight 0 is loaded but masked by a
    // select, so whatever it holds never reaches the output.
    const int chunks = D / 8;
    const float lk = lane < S ? lse0[lane * lse_stride] : -INFINITY;
    float v[4][NC][8];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const Tin *p = part0 + static_cast<int64_t>(u) * part_stride;
#pragma unroll
      for (int i = 0; i < NC; ++i) {
        const int c = lane + 32 * i;
        if (u < S && c < chunks) load8(p + c * 8, v[u][i]);
      }
    }
    float m = lk;
#pragma unroll
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (m == -INFINITY) {
      float zero[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      for (int c = lane; c < chunks; c += 32) store8(out + c * 8, zero);
      if (out_lse && lane == 0) *out_lse = -INFINITY;
      return;
    }
    const float wk = lk == -INFINITY ? 0.f : expf(lk - m);
    float z = wk;
#pragma unroll
    for (int o = 16; o; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    float w[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) w[u] = __shfl_sync(0xffffffffu, wk, u);
    const float inv = 1.f / z;
#pragma unroll
    for (int i = 0; i < NC; ++i) {
      const int c = lane + 32 * i;
      if (c < chunks) {
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (u < S && w[u] != 0.f) {
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = fmaf(w[u], v[u][i][e], acc[e]);
          }
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] *= inv;
        store8(out + c * 8, acc);
      }
    }
    if (out_lse && lane == 0) *out_lse = m + logf(z);
    return;
  }
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
  float acc[NC][8];
#pragma unroll
  for (int i = 0; i < NC; ++i)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[i][e] = 0.f;
  float z = 0.f;
  for (int s0 = 0; s0 < S; s0 += 32) {
    // this pass's weights: lane k holds part s0 + k's (0 for -inf or absent)
    const int sk = s0 + lane;
    const float lk = sk < S ? lse0[sk * lse_stride] : -INFINITY;
    const float wk = lk == -INFINITY ? 0.f : expf(lk - m);
    float zk = wk;
#pragma unroll
    for (int o = 16; o; o >>= 1) zk += __shfl_xor_sync(0xffffffffu, zk, o);
    z += zk;
    const int n = min(32, S - s0);
    for (int b = 0; b < n; b += 4) {
      float w[4];
      float v[4][NC][8];   // [part][chunk slot][element]
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        w[u] = __shfl_sync(0xffffffffu, wk, (b + u) & 31);
        const bool use = b + u < n && w[u] != 0.f;   // weight-0 parts are never read
        const Tin *p = part0 + static_cast<int64_t>(s0 + b + u) * part_stride;
#pragma unroll
        for (int i = 0; i < NC; ++i) {
          const int c = lane + 32 * i;
          if (use && c < chunks) load8(p + c * 8, v[u][i]);
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (!(b + u < n && w[u] != 0.f)) continue;
#pragma unroll
        for (int i = 0; i < NC; ++i) {
          const int c = lane + 32 * i;
          if (c < chunks) {
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[i][e] = fmaf(w[u], v[u][i][e], acc[i][e]);
          }
        }
      }
    }
  }
  const float inv = 1.f / z;
#pragma unroll
  for (int i = 0; i < NC; ++i) {
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
