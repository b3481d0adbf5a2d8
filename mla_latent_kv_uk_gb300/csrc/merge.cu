// A5/A10: LSE-rescaling merge of S partial attention states
// (merge_attn_states).  Source: "DeepSeek MLA 在 DCP 分布式环境中的 Prefill
// 阶段解析", §Chunked Prefill 与 LSE Merge (elementwise rescaling by the
// partial LSEs, O(B*N*V)) and §DCP 在 Prefill 与 Decode 中的不同角色 (decode
// combines per-rank partials by LSE weighting).
//
// HBM-bound: every partial row is read once with 16-byte loads and the
// merged row written once; one thread per 16-byte chunk for up to eight
// parts, one warp per (t, h) row otherwise.
#include <cuda_bf16.h>

#include "common.cuh"
#include "merge_row.cuh"

namespace mla {
namespace {

constexpr int kWarps = 8;

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(kWarps * 32)
merge_kernel(const Tin *__restrict__ parts, const float *__restrict__ plse,
             int S, int rows, int D, Tout *out, float *out_lse) {
  const int row = blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (row >= rows) return;
  merge_row<Tin, Tout>(parts + static_cast<int64_t>(row) * D,
                       static_cast<int64_t>(rows) * D, plse + row, rows, S, D,
                       out + static_cast<int64_t>(row) * D,
                       out_lse ? out_lse + row : nullptr, threadIdx.x & 31);
}

// Few parts (S <= SMAX: 4, the usual shard or prefix / suffix merge, or 8):
// one thread per 16-byte chunk of the output (8 values), every thread
// reading its row's S LSEs itself, so no shuffles and every SM full of
// independent loads.  A part of weight 0 is never read.
constexpr int kChunkThreads = 256;

template <typename Tin, typename Tout, int SMAX>
__global__ void __launch_bounds__(kChunkThreads)
merge_chunks_kernel(const Tin *__restrict__ parts, const float *__restrict__ plse, int S,
                    int64_t rows, int cpr, Tout *out, float *out_lse) {
  const int64_t g = static_cast<int64_t>(blockIdx.x) * kChunkThreads + threadIdx.x;
  const int64_t row = g / cpr;
  const int c = static_cast<int>(g - row * cpr);
  if (row >= rows) return;
  const int D = cpr * 8;
  float l[SMAX], m = -INFINITY;
#pragma unroll
  for (int s = 0; s < SMAX; ++s) {
    l[s] = s < S ? plse[s * rows + row] : -INFINITY;
    m = fmaxf(m, l[s]);
  }
  Tout *dst = out + row * D + c * 8;
  if (m == -INFINITY) {
    const float zero[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    store8(dst, zero);
    if (out_lse && c == 0) out_lse[row] = -INFINITY;
    return;
  }
  float w[SMAX], z = 0.f;
#pragma unroll
  for (int s = 0; s < SMAX; ++s) {
    w[s] = l[s] == -INFINITY ? 0.f : expf(l[s] - m);
    z += w[s];
  }
  float v[SMAX][8];
#pragma unroll
  for (int s = 0; s < SMAX; ++s)
    if (w[s] != 0.f) load8(parts + (s * rows + row) * D + c * 8, v[s]);
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
  for (int s = 0; s < SMAX; ++s)
    if (w[s] != 0.f) {
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = fmaf(w[s], v[s][e], acc[e]);
    }
  const float inv = 1.f / z;
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] *= inv;
  store8(dst, acc);
  if (out_lse && c == 0) out_lse[row] = m + logf(z);
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" int mla_merge_states(const void *parts_out, int parts_dtype,
                                const float *parts_lse, int S, int T, int H,
                                int D, void *out, int out_dtype,
                                float *out_lse, mla_stream_t stream) {
  if (S < 1 || S > 256 || T < 0 || H < 1 || D < 8 || D > 1024 || D % 8)
    return MLA_ERR_INVALID_ARG;
  if ((parts_dtype != MLA_BF16 && parts_dtype != MLA_F32) ||
      (out_dtype != MLA_BF16 && out_dtype != MLA_F32))
    return MLA_ERR_INVALID_ARG;
  if (T == 0) return MLA_OK;
  if (!parts_out || !parts_lse || !out) return MLA_ERR_INVALID_ARG;
  if (!aligned16(parts_out) || !aligned16(out)) return MLA_ERR_INVALID_ARG;
  const int64_t rows64 = static_cast<int64_t>(T) * H;
  if (rows64 > (1ll << 30)) return MLA_ERR_INVALID_ARG;
  const int rows = static_cast<int>(rows64);
  if (S <= 8) {
    // S <= 4 takes the 4-slot form (fewer registers), 5..8 the 8-slot one
    const int cpr = D / 8;
    const dim3 cgrid(static_cast<unsigned>((rows64 * cpr + kChunkThreads - 1) / kChunkThreads));
#define MLA_MERGE_C(TI, TO)                                                   \
  do {                                                                       \
    if (S <= 4)                                                              \
      merge_chunks_kernel<TI, TO, 4><<<cgrid, kChunkThreads, 0, stream>>>(   \
          static_cast<const TI *>(parts_out), parts_lse, S, rows64, cpr,     \
          static_cast<TO *>(out), out_lse);                                  \
    else                                                                     \
      merge_chunks_kernel<TI, TO, 8><<<cgrid, kChunkThreads, 0, stream>>>(   \
          static_cast<const TI *>(parts_out), parts_lse, S, rows64, cpr,     \
          static_cast<TO *>(out), out_lse);                                  \
  } while (0)
    if (parts_dtype == MLA_BF16 && out_dtype == MLA_BF16) MLA_MERGE_C(__nv_bfloat16, __nv_bfloat16);
    else if (parts_dtype == MLA_BF16) MLA_MERGE_C(__nv_bfloat16, float);
    else if (out_dtype == MLA_BF16) MLA_MERGE_C(float, __nv_bfloat16);
    else MLA_MERGE_C(float, float);
#undef MLA_MERGE_C
    return launch_status();
  }
  dim3 grid((rows + kWarps - 1) / kWarps);
#define MLA_MERGE(TI, TO)                                                     \
  merge_kernel<TI, TO><<<grid, kWarps * 32, 0, stream>>>(                     \
      static_cast<const TI *>(parts_out), parts_lse, S, rows, D,             \
      static_cast<TO *>(out), out_lse)
  if (parts_dtype == MLA_BF16 && out_dtype == MLA_BF16) MLA_MERGE(__nv_bfloat16, __nv_bfloat16);
  else if (parts_dtype == MLA_BF16) MLA_MERGE(__nv_bfloat16, float);
  else if (out_dtype == MLA_BF16) MLA_MERGE(float, __nv_bfloat16);
  else MLA_MERGE(float, float);
#undef MLA_MERGE
  return launch_status();
}
