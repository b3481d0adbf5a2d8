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

// Few parts (S <= SMAX: 2, the prefix / suffix merge; 4, the usual shard
// merge; or 8): one thread per CH consecutive 16-byte chunks of an output
// row (8 values each), every thread reading its row's S LSEs itself, so no
// shuffles.  The parts' chunks are requested together with the LSEs (one
// round trip per thread) and CH chunks per part are in flight at once, so
// each SM keeps enough bytes in flight to stream at HBM speed.  A part of
// weight 0 is loaded but never folded in, so whatever it holds never
// reaches the output.
constexpr int kChunkThreads = 256;

// One 16-byte chunk (8 values) of a part as loaded, unpacked to fp32 only
// where it is folded in, so the chunks in flight cost 4 (bf16) or 8 (fp32)
// registers each.
template <typename T> struct Chunk;
template <> struct Chunk<__nv_bfloat16> {
  uint4 u;
  __device__ __forceinline__ void load(const __nv_bfloat16 *p) {
    u = __ldg(reinterpret_cast<const uint4 *>(p));
  }
  __device__ __forceinline__ float at(int e) const {
    const uint32_t w = e < 4 ? (e < 2 ? u.x : u.y) : (e < 6 ? u.z : u.w);
    return __uint_as_float((e & 1) ? (w & 0xFFFF0000u) : (w << 16));
  }
};
template <> struct Chunk<float> {
  float4 a, b;
  __device__ __forceinline__ void load(const float *p) {
    a = __ldg(reinterpret_cast<const float4 *>(p));
    b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
  }
  __device__ __forceinline__ float at(int e) const {
    const float4 &q = e < 4 ? a : b;
    const int i = e & 3;
    return i == 0 ? q.x : i == 1 ? q.y : i == 2 ? q.z : q.w;
  }
};

// registers of the chunks in flight at most 32 -> four CTAs per SM
template <typename Tin, int SMAX, int CH>
constexpr int kMergeCtas = SMAX * CH * static_cast<int>(sizeof(Tin)) * 2 <= 32 ? 4 : 2;

template <typename Tin, typename Tout, int SMAX, int CH>
__global__ void __launch_bounds__(kChunkThreads, (kMergeCtas<Tin, SMAX, CH>))
merge_chunks_kernel(const Tin *__restrict__ parts, const float *__restrict__ plse, int S,
                    int64_t rows, int cpr, Tout *out, float *out_lse) {
  const int gpr = cpr / CH;   // thread groups per row
  const int64_t g = static_cast<int64_t>(blockIdx.x) * kChunkThreads + threadIdx.x;
  const int64_t row = g / gpr;
  const int c0 = static_cast<int>(g - row * gpr) * CH;
  if (row >= rows) return;
  const int D = cpr * 8;
  float l[SMAX], m = -INFINITY;
  Chunk<Tin> v[SMAX][CH];
#pragma unroll
  for (int s = 0; s < SMAX; ++s) {
    l[s] = -INFINITY;
    if (s < S) {
      l[s] = plse[s * rows + row];
      const Tin *src = parts + (s * rows + row) * D + c0 * 8;
#pragma unroll
      for (int k = 0; k < CH; ++k) v[s][k].load(src + k * 8);
    }
  }
#pragma unroll
  for (int s = 0; s < SMAX; ++s) m = fmaxf(m, l[s]);
  Tout *dst = out + row * D + c0 * 8;
  if (m == -INFINITY) {
    const float zero[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
    for (int k = 0; k < CH; ++k) store8(dst + k * 8, zero);
    if (out_lse && c0 == 0) out_lse[row] = -INFINITY;
    return;
  }
  float w[SMAX], z = 0.f;
#pragma unroll
  for (int s = 0; s < SMAX; ++s) {
    w[s] = l[s] == -INFINITY ? 0.f : expf(l[s] - m);
    z += w[s];
  }
  const float inv = 1.f / z;
#pragma unroll
  for (int k = 0; k < CH; ++k) {
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
    for (int s = 0; s < SMAX; ++s)
      if (w[s] != 0.f) {
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = fmaf(w[s], v[s][k].at(e), acc[e]);
      }
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] *= inv;
    store8(dst + k * 8, acc);
  }
  if (out_lse && c0 == 0) out_lse[row] = m + logf(z);
}

template <typename Tin, typename Tout, int SMAX, int CH>
void launch_chunks(const void *parts, const float *plse, int S, int64_t rows, int cpr,
                   void *out, float *out_lse, cudaStream_t stream) {
  const int64_t groups = rows * (cpr / CH);
  const dim3 grid(static_cast<unsigned>((groups + kChunkThreads - 1) / kChunkThreads));
  merge_chunks_kernel<Tin, Tout, SMAX, CH><<<grid, kChunkThreads, 0, stream>>>(
      static_cast<const Tin *>(parts), plse, S, rows, cpr, static_cast<Tout *>(out), out_lse);
}

// S <= 2: two slots, four chunks a thread; S <= 4: four slots, two chunks;
// S <= 8: eight slots, one chunk (fewer chunks when the row has fewer).
template <typename Tin, typename Tout>
void merge_few(const void *parts, const float *plse, int S, int64_t rows, int cpr, void *out,
               float *out_lse, cudaStream_t stream) {
  if (S <= 2) {
    if (cpr % 4 == 0) launch_chunks<Tin, Tout, 2, 4>(parts, plse, S, rows, cpr, out, out_lse, stream);
    else if (cpr % 2 == 0) launch_chunks<Tin, Tout, 2, 2>(parts, plse, S, rows, cpr, out, out_lse, stream);
    else launch_chunks<Tin, Tout, 2, 1>(parts, plse, S, rows, cpr, out, out_lse, stream);
  } else if (S <= 4) {
    if (cpr % 2 == 0) launch_chunks<Tin, Tout, 4, 2>(parts, plse, S, rows, cpr, out, out_lse, stream);
    else launch_chunks<Tin, Tout, 4, 1>(parts, plse, S, rows, cpr, out, out_lse, stream);
  } else {
    launch_chunks<Tin, Tout, 8, 1>(parts, plse, S, rows, cpr, out, out_lse, stream);
  }
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
    const int cpr = D / 8;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (parts_dtype == MLA_BF16 && out_dtype == MLA_BF16)
      merge_few<__nv_bfloat16, __nv_bfloat16>(parts_out, parts_lse, S, rows64, cpr, out, out_lse, st);
    else if (parts_dtype == MLA_BF16)
      merge_few<__nv_bfloat16, float>(parts_out, parts_lse, S, rows64, cpr, out, out_lse, st);
    else if (out_dtype == MLA_BF16)
      merge_few<float, __nv_bfloat16>(parts_out, parts_lse, S, rows64, cpr, out, out_lse, st);
    else
      merge_few<float, float>(parts_out, parts_lse, S, rows64, cpr, out, out_lse, st);
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
