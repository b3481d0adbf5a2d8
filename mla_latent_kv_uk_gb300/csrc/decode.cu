// A3/A4/A5: split-KV plan, paged latent decode (forward_mqa) and the
// on-device merge of split partials.
//
// Sources: prhub digest of vLLM PR 44044, §关键源码片段 mla_attention.py
// (forward_mqa(mqa_q, kv_cache, attn_metadata) -> attn_out, lse) and
// §关键源码片段 flashmla.py (split scheduler metadata derived on the device
// from seq_lens and the true head count); "DeepSeek MLA 在 DCP 分布式环境中的
// Prefill 阶段解析", §MLA Prefill vs Decode (decode keeps KV as one latent
// head of width 512 + 64; the value is the 512-wide latent part) and
// §Chunked Prefill 与 LSE Merge (LSE-rescaling merge of partial states).
//
// Design (GB300, sm_103a):
//  * All 128 heads of a query token share one latent KV row, so per 64-token
//    tile S = Q K^T is a dense [128 x 64 x 576] contraction and O += P V a
//    [128 x 512 x 64] one: both run on tcgen05 with fp32 TMEM accumulators.
//  * The fp32 output of 128 heads x 512 latent columns is exactly one SM's
//    TMEM, so each work span is processed by a PAIR of CTAs, CTA c owning
//    latent output columns [256c, 256c + 256).
//  * decode_pair_kernel<FP8> (bf16 or e4m3 cache): the pair is a 2-CTA
//    cluster that splits the QK contraction by columns.  Each CTA loads
//    only its latent half and its half of the rope columns of every KV
//    tile, and the partial scores are summed through distributed shared
//    memory (see the kernel's comment).  The e4m3 format uses the same
//    layout with half-size stages (twice as many in the ring), kind::f8f6f4
//    MMAs and e4m3 probabilities.
//  * Warp roles (8 warps, by the CTA's rank): TMA producer, MMA issuer,
//    online softmax of the CTA's own head rows (one row per thread), the
//    sending of the forwarded rows' partial scores, and the return of their
//    probabilities; the softmax and return warps also write the epilogue.
//    Lazy rescaling: O is rescaled only when a row max grows by more than
//    2^8.
//  * Work split (A3): every job (request, query token, 128-head group)
//    contributes the 64-token tiles its key range touches, preceded by
//    kJobCost units that stand for the cost of switching to it; jobs are
//    laid end to end and CTA pair p takes units [p*C, (p+1)*C).  A job cut
//    into several spans writes partials (in the output's type) that a merge
//    kernel combines (one CTA per 16 rows, partials streamed in by bulk
//    copies).
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <math.h>

#include <algorithm>
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "merge_row.cuh"
#include "sm100.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kMinTiles = 4;                 // smallest auto span
// Units of the flat split space a non-empty job takes on top of its tiles:
// switching a CTA pair to a job costs its epilogue and query load (about
// 2.5 us, two to three 64-token tiles), so a span that meets a job start is
// given fewer tiles and spans that cross request boundaries end with the
// others.  Four units timed best on the DeepSeek-V3 decode shape (B = 32,
// 4096 tokens each) against two and three.
constexpr int kJobCost = 4;
constexpr float kRescaleLog2 = 8.f;          // lazy rescale threshold
constexpr uint32_t kColO = 0, kColS = 256;   // TMEM columns (both variants)

// ----------------------------------------------------------------- planner
// Plan layout (int32): [0] total units, [1] C, [2] J, [3] spans, then
// tile_prefix[J+1] (prefix of the units per job: its tiles + kJobCost, 0
// for an empty job), seg_prefix[J+1], job_lo[J+1], job_hi[J+1].
struct PlanView {
  const int32_t *base;
  int J;
  __device__ int total() const { return base[0]; }
  __device__ int chunk() const { return base[1]; }
  __device__ const int32_t *tile_prefix() const { return base + 4; }
  __device__ const int32_t *seg_prefix() const { return base + 4 + (J + 1); }
  __device__ const int32_t *job_lo() const { return base + 4 + 2 * (J + 1); }
  __device__ const int32_t *job_hi() const { return base + 4 + 3 * (J + 1); }
};

size_t plan_ints(int J) { return 4 + 4 * static_cast<size_t>(J + 1); }

constexpr int kPlanThreads = 1024;

// Exclusive prefix sum over n values held in v[0..n) (in place), one CTA.
__device__ int block_exclusive_scan(int32_t *v, int n, int32_t *scratch) {
  const int tid = threadIdx.x;
  const int per = (n + kPlanThreads - 1) / kPlanThreads;
  const int a = min(n, tid * per), z = min(n, a + per);
  int local = 0;
  for (int k = a; k < z; ++k) local += v[k];
  // inclusive scan of `local` across the block
  int x = local;
  const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = scratch[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    scratch[lane] = w;
  }
  __syncthreads();
  int run = x - local + (warp ? scratch[warp - 1] : 0);
  const int total = scratch[31];
  for (int k = a; k < z; ++k) {
    const int t = v[k];
    v[k] = run;
    run += t;
  }
  __syncthreads();
  return total;
}

__global__ void __launch_bounds__(kPlanThreads)
plan_kernel(const int32_t *__restrict__ seq_lens,
            const int32_t *__restrict__ kv_starts,
            const int32_t *__restrict__ kv_ends, int B, int q_len, int HG,
            int max_blocks, int causal, int tile, int forced_chunk,
            int groups, int32_t *plan, int *err) {
  __shared__ int32_t scratch[32];
  // the decode grid may be scheduled now; it waits for this grid to finish
  // before it reads the plan
  sm100::grid_dep_launch();
  // launched with programmatic stream serialization: the lengths and
  // ranges may come from the previous kernel in the stream
  sm100::grid_dep_wait();
  const int J = B * q_len * HG;
  int32_t *tp = plan + 4;
  int32_t *sp = tp + (J + 1);
  int32_t *lo_a = sp + (J + 1);
  int32_t *hi_a = lo_a + (J + 1);
  for (int j = threadIdx.x; j < J; j += blockDim.x) {
    const int bi = j / HG;
    const int i = bi / B, b = bi % B;   // token-major job order
    int len = seq_lens[b];
    if (len < 0 || len > max_blocks * kPage) {
      if (i == 0 && j % HG == 0) raise_error(err, MLA_DEVERR_SEQ_LEN);
      len = min(max(len, 0), max_blocks * kPage);
    }
    int hi = causal ? len - q_len + i + 1 : len;
    hi = min(hi, len);
    int lo = 0;
    if (kv_starts) lo = max(lo, kv_starts[b]);
    if (kv_ends) hi = min(hi, kv_ends[b]);
    hi = max(hi, 0);
    lo = min(max(lo, 0), hi);
    lo_a[j] = lo;
    hi_a[j] = hi;
    tp[j] = hi > lo ? (hi + tile - 1) / tile - lo / tile + kJobCost : 0;
  }
  if (threadIdx.x == 0) { lo_a[J] = 0; hi_a[J] = 0; }
  __syncthreads();
  const int total = block_exclusive_scan(tp, J, scratch);
  if (threadIdx.x == 0) tp[J] = total;
  const int C = forced_chunk > 0 ? forced_chunk
                                 : max(kMinTiles, (total + groups - 1) / groups);
  __syncthreads();
  for (int j = threadIdx.x; j < J; j += blockDim.x) {
    const int z = tp[j + 1];
    const int a = tp[j] + (z > tp[j] ? kJobCost : 0);   // the job's first tile
    sp[j] = z > a ? (z - 1) / C - a / C + 1 : 0;
  }
  __syncthreads();
  const int segs = block_exclusive_scan(sp, J, scratch);
  if (threadIdx.x == 0) {
    sp[J] = segs;
    plan[0] = total;
    plan[1] = C;
    plan[2] = J;
    plan[3] = (total + C - 1) / C;
  }
}

// The same plan from one warp, for up to kWarpPlanJobs jobs: every lane
// takes ceil(J/32) <= 8 consecutive jobs, the prefixes come from warp scans
// (no block-wide barriers on the path from the lengths to the plan).
constexpr int kWarpPlanJobs = 256;

__global__ void __launch_bounds__(32)
plan_warp_kernel(const int32_t *__restrict__ seq_lens,
                 const int32_t *__restrict__ kv_starts,
                 const int32_t *__restrict__ kv_ends, int B, int q_len, int HG,
                 int max_blocks, int causal, int tile, int forced_chunk,
                 int groups, int32_t *plan, int *err) {
  sm100::grid_dep_launch();
  // launched with programmatic stream serialization: the lengths and
  // ranges may come from the previous kernel in the stream
  sm100::grid_dep_wait();
  const int lane = threadIdx.x;
  const int J = B * q_len * HG;
  const int per = (J + 31) / 32;
  const int j0 = lane * per;
  int32_t *tp = plan + 4;
  int32_t *sp = tp + (J + 1);
  int32_t *lo_a = sp + (J + 1);
  int32_t *hi_a = lo_a + (J + 1);
  int t[8], local = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int j = j0 + k;
    t[k] = 0;
    if (k < per && j < J) {
      const int bi = j / HG;
      const int i = bi / B, b = bi % B;   // token-major job order
      int len = seq_lens[b];
      if (len < 0 || len > max_blocks * kPage) {
        if (i == 0 && j % HG == 0) raise_error(err, MLA_DEVERR_SEQ_LEN);
        len = min(max(len, 0), max_blocks * kPage);
      }
      int hi = causal ? len - q_len + i + 1 : len;
      hi = min(hi, len);
      int lo = 0;
      if (kv_starts) lo = max(lo, kv_starts[b]);
      if (kv_ends) hi = min(hi, kv_ends[b]);
      hi = max(hi, 0);
      lo = min(max(lo, 0), hi);
      lo_a[j] = lo;
      hi_a[j] = hi;
      t[k] = hi > lo ? (hi + tile - 1) / tile - lo / tile + kJobCost : 0;
      local += t[k];
    }
  }
  // exclusive scan of the lanes' sums; `tot` gets the warp total
  auto excl_scan = [&](int v, int &tot) {
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    tot = __shfl_sync(0xffffffffu, x, 31);
    return x - v;
  };
  int total;
  int run = excl_scan(local, total);
  int a[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    a[k] = run;
    if (k < per && j0 + k < J) tp[j0 + k] = run;
    run += t[k];
  }
  const int C = forced_chunk > 0 ? forced_chunk : max(kMinTiles, (total + groups - 1) / groups);
  int s[8];
  local = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int z = a[k] + t[k];
    const int first = a[k] + (t[k] > 0 ? kJobCost : 0);   // the job's first tile
    s[k] = (k < per && j0 + k < J && z > first) ? (z - 1) / C - first / C + 1 : 0;
    local += s[k];
  }
  int segs;
  run = excl_scan(local, segs);
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    if (k < per && j0 + k < J) sp[j0 + k] = run;
    run += s[k];
  }
  if (lane == 0) {
    tp[J] = total;
    sp[J] = segs;
    lo_a[J] = 0;
    hi_a[J] = 0;
    plan[0] = total;
    plan[1] = C;
    plan[2] = J;
    plan[3] = (total + C - 1) / C;
  }
}

// Launches the plan on `stream` (one warp for small J), programmatic
// stream serialization after the previous kernel.
cudaError_t launch_plan(const int32_t *seq_lens, const int32_t *kv_starts, const int32_t *kv_ends,
                        int B, int q_len, int HG, int max_blocks, int causal, int tile,
                        int split_tiles, int groups, int32_t *plan, int *err,
                        cudaStream_t stream) {
  if (static_cast<int64_t>(B) * q_len * HG <= kWarpPlanJobs)
    return launch_pdl(plan_warp_kernel, dim3(1), dim3(32), 0, stream, seq_lens, kv_starts,
                      kv_ends, B, q_len, HG, max_blocks, causal, tile, split_tiles, groups,
                      plan, err);
  return launch_pdl(plan_kernel, dim3(1), dim3(kPlanThreads), 0, stream, seq_lens, kv_starts,
                    kv_ends, B, q_len, HG, max_blocks, causal, tile, split_tiles, groups, plan,
                    err);
}

// ---------------------------------------------------------- segment walk
struct Seg {
  int job, row0;        // job index, first q row ((b*q_len + i)*H + hg*128)
  int b, hrows;         // request, valid head rows in this group
  int out_row0;         // first output row ((b*q_len + i)*H + hg*128)
  int lo, hi;           // key range
  int tile0, ntiles;    // first absolute tile, tiles in this segment
  int whole, slot;      // covers the whole job?  partial slot otherwise
  int len;              // seq_len of the request (set by the pair kernel's producer)
  int qkc;              // ring index of the first of its two query stages (pair kernel)
};

struct SegWalk {
  PlanView plan;
  int B, q_len, H, HG, groups, tile;
  int p, span_lo, span_hi, j;
  bool started;

  __device__ void init(const int32_t *pl, int J, int ql, int h, int hg,
                       int g, int group_id, int tile_tokens) {
    plan = PlanView{pl, J};
    q_len = ql; H = h; HG = hg; groups = g; tile = tile_tokens;
    B = J / (ql * hg);
    p = group_id;
    started = false;
  }

  // The next segment of this CTA pair, for a whole warp (every lane gets it): the span's
  // first job is found by a 32-way search (one round of loads for up to 32
  // jobs, instead of a chain of dependent loads), and the job's fields and
  // its request's seq_len are loaded together (s.len is set).
  __device__ bool next_warp(Seg &s, const int32_t *__restrict__ seq_lens) {
    const int lane = threadIdx.x & 31;
    const int total = plan.total(), C = plan.chunk();
    const int32_t *tp = plan.tile_prefix();
    while (true) {
      if (!started) {
        if (p * C >= total) return false;
        span_lo = p * C;
        span_hi = min(total, span_lo + C);
        // last j in [0, J] with tp[j] <= span_lo (tp[0] = 0, non-decreasing)
        int a = 0, z = plan.J;
        while (a < z) {
          const int stride = (z - a + 32) / 32;         // ceil((z - a + 1) / 32)
          const int idx = a + lane * stride;
          const bool le = idx <= z && tp[idx] <= span_lo;
          const uint32_t mask = __ballot_sync(0xffffffffu, le);
          const int hi_lane = 31 - __clz(mask);          // lane 0 always qualifies
          const int na = a + hi_lane * stride;
          z = min(z, na + stride - 1);
          a = na;
          if (stride == 1) break;
        }
        j = a;
        started = true;
      }
      if (j >= plan.J) {
        p += groups;
        started = false;
        continue;
      }
      // jobs are token-major: (query token i, request b, head group)
      const int bi = j / HG, hg = j % HG;
      const int i = bi / B, b = bi % B;
      // independent loads, all in flight together
      const int t0 = tp[j], t1 = tp[j + 1];
      const int lo = plan.job_lo()[j], hi = plan.job_hi()[j];
      const int sp = plan.seg_prefix()[j];
      const int len = __ldg(seq_lens + b);
      if (t0 >= span_hi) {
        p += groups;
        started = false;
        continue;
      }
      if (t1 <= t0) { ++j; continue; }    // empty job
      const int a = t0 + kJobCost;        // the job's first tile (after its switch cost)
      const int u0 = max(span_lo, a), u1 = min(span_hi, t1);
      if (u1 <= u0) { ++j; continue; }    // the span meets only the switch cost
      s.job = j;
      s.b = b;
      s.row0 = (b * q_len + i) * H + hg * 128;
      s.out_row0 = s.row0;
      s.hrows = min(128, H - hg * 128);
      s.lo = lo;
      s.hi = hi;
      s.tile0 = lo / tile + (u0 - a);
      s.ntiles = u1 - u0;
      s.whole = (span_lo <= a) && (t1 <= span_hi);
      s.slot = sp + (span_lo / C - a / C);
      s.len = len;
      ++j;
      return true;
    }
  }
};

struct DecodeArgs {
  const int32_t *plan;
  int J;
  const int32_t *block_table;
  const int32_t *seq_lens;
  const uint8_t *q;           // [B, q_len, H, 576] bf16 or e4m3
  int q_len, H, HG, max_blocks, num_blocks, groups;
  float scale_log2;           // sm_scale * log2(e) (* q_scale * k_scale)
  float out_scale;            // 1 (bf16) or k_scale (e4m3 values)
  void *out;
  int out_dtype;
  float *lse;
  float *ws_o;                // [slots, 128, 512]
  float *ws_lse;              // [slots, 128]
  int *err;
};

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  return bf16x2_rn(a, b);
}

// Four probabilities -> four e4m3 codes in one 32-bit TMEM column (element
// k in byte k).
__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c,
                                                float d) {
  const __nv_fp8x2_storage_t lo =
      __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const __nv_fp8x2_storage_t hi =
      __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// ------------------------------------------------- split-QK pair kernel
// The two CTAs of a 2-CTA cluster share one work span.  CTA c loads only
// latent columns [256c, 256c + 256) of each KV tile plus rope columns
// [32c, 32c + 32) (36 KB instead of 72 KB per bf16 tile) and computes the
// partial scores of its 288 columns (16 latent K steps with the query in
// TMEM, 2 rope K steps with the query rope half in shared memory).  The
// partials are summed across the pair through distributed shared memory:
//   * rows (heads) [64c, 64c + 64) are "own" rows of CTA c: it receives the
//     peer's partial scores of those rows (16 KB bulk copy), runs the online
//     softmax on them, writes the probabilities into its P operand tile and
//     copies those rows, with the rescale factor and running row sum, into
//     the peer's P operand tile;
//   * the other 64 rows it forwards: it ships its partial scores to the peer
//     and gets the probabilities back.
// Each CTA still owns output columns [256c, 256c + 256) for all 128 heads,
// and its value operand is exactly the latent boxes it loaded.  P lives in
// shared memory (P.V reads it as the A operand), so a TMEM score buffer is
// free as soon as both row groups have read it: QK runs up to two tiles
// ahead of the softmax, independently of P.V, and the two message latencies
// overlap other tiles' work instead of adding up per tile.
namespace pair {
constexpr int kTile = 64;
constexpr int kThreads = 256;                   // 8 warps, roles below
constexpr int kStages = 4;
constexpr int kBox = 8192;                      // 64 tokens x 64 bf16, SW128
constexpr int kRopeBox = 4096;                  // 64 tokens x 32 bf16, SW64
constexpr int kStageBytes = 4 * kBox + kRopeBox;   // 36 KB
constexpr int kPBuf = 128 * 128;                // 128 heads x 64 tokens bf16, SW128
constexpr int kQRopeBytes = 128 * 64;           // 128 heads x 32 rope dims, SW64
constexpr int kSMsg = 64 * 64 * 4;              // 64 rows x 64 fp32 scores
constexpr int kAlMsg = 2 * 64 * 4;              // alpha[64], l[64]
constexpr int kOffRing = 0;
constexpr int kOffP = kOffRing + kStages * kStageBytes;       // [2] P operand tiles
constexpr int kOffQ = kOffP + 2 * kPBuf;
constexpr int kOffSSend = kOffQ + kQRopeBytes;
constexpr int kOffSRecv = kOffSSend + kSMsg;
constexpr int kOffAlSend = kOffSRecv + kSMsg;                 // [2]
constexpr int kOffAlRecv = kOffAlSend + 2 * kAlMsg;           // [2]
constexpr int kOffBars = kOffAlRecv + 2 * kAlMsg;
constexpr int kMaxStages = 8;                   // ring stages of the e4m3 format
constexpr int kNumBars = 2 * kMaxStages + 28;
constexpr int kSegSlots = 4;                    // segment descriptors in flight
constexpr int kOffSegQ = kOffBars + kNumBars * 8 + 16;
constexpr int kSmem = kOffSegQ + kSegSlots * 64 + 1024;
constexpr int kQkChunks = 3;                    // QK of a tile in three bursts
constexpr uint32_t kColQ = 384;                 // query latent half (128 / 64 columns)
static_assert(kSmem <= 232448, "shared memory of one CTA");
static_assert(kOffP % 1024 == 0 && kOffQ % 1024 == 0 && kStageBytes % 1024 == 0,
              "swizzled tiles start on 1024-byte boundaries");

// What differs between the bf16 and the e4m3 cache.  Either way a CTA loads
// four latent boxes of 64 columns x 64 tokens and one rope box of 32
// columns (its half), every QK K step covers 32 bytes of a row (16 bf16 or
// 32 e4m3: eight 32-bit TMEM columns of the query), and a P.V K step covers
// 2 KB of the value boxes (16 tokens x 128 B or 32 tokens x 64 B), so the
// shared-memory layout above holds both (e4m3 stages are half as large,
// twice as many fill the ring; its P rows are 64 B).
template <bool FP8>
struct Fmt {
  static constexpr int kEsz = FP8 ? 1 : 2;                 // bytes per element
  static constexpr int kBox = 64 * 64 * kEsz;              // latent box
  static constexpr int kRopeBox = 64 * 32 * kEsz;          // rope box
  static constexpr int kStageBytes = 4 * kBox + kRopeBox;  // 18 / 36 KB
  static constexpr int kStages = (4 * 36864) / kStageBytes;   // 8 / 4: the same ring bytes
  static constexpr int kQRopeBytes = 128 * 32 * kEsz;
  static constexpr uint32_t kSwL = FP8 ? sm100::kSwizzle64B : sm100::kSwizzle128B;
  static constexpr uint32_t kSwR = FP8 ? sm100::kSwizzle32B : sm100::kSwizzle64B;
  static constexpr uint32_t kSboL = 8 * 64 * kEsz;         // 8 rows of a latent box
  static constexpr uint32_t kSboR = 8 * 32 * kEsz;         // 8 rows of a rope box
  static constexpr int kStepsPerBox = 64 * kEsz / 32;      // QK K steps per box row
  static constexpr int kLatSteps = 4 * kStepsPerBox;       // 8 / 16
  static constexpr int kRopeSteps = 32 * kEsz / 32;        // 1 / 2
  static constexpr int kChunkSteps = (kLatSteps + kRopeSteps) / 3;   // 3 / 6
  static constexpr int kPvSteps = FP8 ? 2 : 4;             // 32 / 16 tokens per step
  static constexpr int kPRow = 64 * kEsz;                  // bytes of one P row
  static constexpr uint32_t kSwP = FP8 ? sm100::kSwizzle64B : sm100::kSwizzle128B;
  static constexpr uint32_t kSboP = 8 * kPRow;
  static constexpr uint32_t kPMsg = 64 * kPRow + kAlMsg;   // bytes landing per P message
  static constexpr int kQCols = 64 * kEsz;                 // TMEM columns of the query half
  // the query latent half enters through two ring stages, each holding two
  // boxes of 64 columns x 128 rows in the latent swizzle
  static constexpr int kQRow = 64 * kEsz;                  // bytes of a query box row
  static constexpr int kQBox = 128 * kQRow;                // 16 / 8 KB
  static constexpr int kQStageBytes = 2 * kQBox;
  static_assert(kStages <= kMaxStages && kStages * kStageBytes == 4 * 36864, "ring");
  static_assert(3 * kChunkSteps == kLatSteps + kRopeSteps, "three QK chunks");
  static_assert(kQStageBytes <= kStageBytes && kQBox % 1024 == 0, "query stages");
};
}  // namespace pair

template <bool FP8>
__global__ void __launch_bounds__(pair::kThreads, 1)
decode_pair_kernel(const __grid_constant__ CUtensorMap tm_kv,
                   const __grid_constant__ CUtensorMap tm_kr,
                   const __grid_constant__ CUtensorMap tm_qr,
                   const __grid_constant__ CUtensorMap tm_ql,
                   DecodeArgs args) {
  using namespace pair;
  using F = Fmt<FP8>;
  // the format's geometry under the names the code below uses
  constexpr int kStages = F::kStages, kStageBytes = F::kStageBytes, kBox = F::kBox;
  constexpr int kQRopeBytes = F::kQRopeBytes, kPvSteps = F::kPvSteps;
  constexpr int kChunkSteps = F::kChunkSteps;
  constexpr uint32_t kPMsg = F::kPMsg;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *sm_kv = smem + kOffRing;
  uint8_t *sm_p = smem + kOffP;
  uint8_t *sm_q = smem + kOffQ;
  uint8_t *s_send = smem + kOffSSend;
  uint8_t *s_recv = smem + kOffSRecv;
  uint8_t *al_send = smem + kOffAlSend;
  uint8_t *al_recv = smem + kOffAlRecv;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBars);
  uint64_t *kv_full = bars;                 // [kStages]
  uint64_t *kv_empty = bars + kStages;      // [kStages]
  uint64_t *s_full = bars + 2 * kStages;    // [2] QK done
  uint64_t *s_free = s_full + 2;            // [2] both row groups have read S
  uint64_t *p_full = s_free + 2;            // [2] all 128 rows of P in place
  uint64_t *pv_done = p_full + 2;           // [2]
  uint64_t *xp_full = pv_done + 2;          // [2] the peer's P rows + factors landed
  uint64_t *pb_free = xp_full + 2;          // [2] the peer's P.V of two tiles ago is done
  uint64_t *q_full = pb_free + 2;
  uint64_t *q_tmem = q_full + 1;
  uint64_t *q_free = q_tmem + 1;
  uint64_t *drain = q_free + 1;
  uint64_t *xs_full = drain + 1;            // the peer's partial scores landed
  uint64_t *xs_free = xs_full + 1;          // the peer consumed our last scores
  uint64_t *seg_full = xs_free + 1;         // [kSegSlots] descriptor published
  uint64_t *seg_empty = seg_full + kSegSlots;   // [kSegSlots] every consumer has copied it
  uint64_t *stage_ok = seg_empty + kSegSlots;   // outgoing copies have read the P tiles
  uint64_t *epi_done = stage_ok + 1;            // every warp's epilogue staging has been read
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(epi_done + 1);
  Seg *segq = reinterpret_cast<Seg *>(smem + kOffSegQ);   // [kSegSlots]
  static_assert(sizeof(Seg) <= 64, "segment descriptor slot");
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = warp_id(), lane = lane_id();
  const int half = static_cast<int>(cluster_rank());
  const uint32_t peer = static_cast<uint32_t>(half ^ 1);
  const int group = blockIdx.x >> 1;
  // Roles.  A warp reaches only its TMEM lane quadrant (warp % 4), which
  // holds 32 head rows.  In the two quadrants of this CTA's own rows
  // ([64*half, 64*half + 64)) warps 4..7 run the online softmax and warps
  // 0..3 are the TMA producer and the MMA issuer; in the two quadrants of
  // the forwarded rows warps 0..3 send the partial scores to the peer and
  // warps 4..7 take the probabilities back (two streams, each served by a
  // warp of its own, so neither waits behind the other).
  const int quarter = warp & 3;
  const bool own = (quarter >> 1) == half;
  const bool upper = warp >= 4;
  const bool is_producer = own && !upper && (quarter & 1) == 0;
  const bool is_mma = own && !upper && (quarter & 1) == 1;
  const bool is_sender = !own && !upper;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&s_free[s], 4);     // lane 0 of each own-row and sending warp
      mbar_init(&p_full[s], 128);
      mbar_init(&pv_done[s], 1);
      mbar_init(&xp_full[s], 1);
      mbar_init(&pb_free[s], 1);
    }
    mbar_init(q_full, 1);
    mbar_init(q_tmem, 128);
    mbar_init(q_free, 1);
    mbar_init(drain, 1);
    mbar_init(xs_full, 1);
    mbar_init(xs_free, 2);          // lane 0 of each of the peer's own-row warps
    for (int s = 0; s < kSegSlots; ++s) {
      mbar_init(&seg_full[s], 1);
      mbar_init(&seg_empty[s], 7);  // the MMA thread and lane 0 of six warps
    }
    mbar_init(stage_ok, 4);         // lane 0 of warps 4..7, once per segment
    mbar_init(epi_done, 4);         // likewise
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
  // both CTAs' barriers exist before either sends the other anything
  cluster_sync();
  // the prologue above overlaps the plan kernel; the plan is read below
  grid_dep_wait();
  grid_dep_launch();

  SegWalk walk;
  walk.init(args.plan, args.J, args.q_len, args.H, args.HG, args.groups, group, kTile);
  Seg sg;

  if (is_producer) {
    // -------------------------------------------------- TMA producer
    if (lane == 0) {
      prefetch_tmap(&tm_kv);
      prefetch_tmap(&tm_kr);
      prefetch_tmap(&tm_qr);
      prefetch_tmap(&tm_ql);
    }
    int kc = 0, nseg = 0;
    bool ok = true;
    const uint64_t kv_policy = l2_evict_first_policy();
    // Publishes segment descriptor `ns` (or the end marker, ntiles = -1) in
    // the shared-memory ring read by the MMA thread and the softmax warps,
    // so they never walk the plan in global memory themselves.
    auto publish = [&](int ns, bool end) -> bool {
      const int slot = ns % kSegSlots;
      if (ns >= kSegSlots &&
          !mbar_wait(&seg_empty[slot], ((ns / kSegSlots) - 1) & 1, abort_flag))
        return false;
      if (lane == 0) {
        Seg d = sg;
        if (end) d.ntiles = -1;
        segq[slot] = d;
        mbar_arrive(&seg_full[slot]);
      }
      __syncwarp();
      return true;
    };
    while (ok && walk.next_warp(sg, args.seq_lens)) {
      sg.qkc = kc;   // its query stages take the next two ring slots
      if (!(ok = publish(nseg, false))) break;
      const int32_t *bt = args.block_table + static_cast<int64_t>(sg.b) * args.max_blocks;
      int page_base = -(1 << 30), my_blk = -1;
      auto blk_of = [&](int tile) -> int {  // warp-collective
        const int page = tile * kTile / kPage;
        if (page < page_base || page >= page_base + 32) {
          page_base = page;
          my_blk = page + lane < args.max_blocks ? __ldg(bt + page + lane) : -1;
        }
        return __shfl_sync(0xffffffffu, my_blk, page - page_base);
      };
      // Loads this CTA's part of KV tile `tile` into ring slot kc % kStages.
      auto load_tile = [&](int tile) -> bool {
        const int s = kc % kStages;
        if (kc >= kStages && !mbar_wait(&kv_empty[s], ((kc / kStages) - 1) & 1, abort_flag))
          return false;
        const int blk = blk_of(tile);
        if (lane == 0) {
          int row;
          if (blk < 0 || blk >= args.num_blocks) {
            raise_error(args.err, MLA_DEVERR_BLOCK_ID);
            row = args.num_blocks * kPage;  // out of range: TMA fills zeros
          } else {
            row = blk * kPage + (tile * kTile) % kPage;
          }
          uint8_t *dst = sm_kv + s * kStageBytes;
          mbar_arrive_expect_tx(&kv_full[s], kStageBytes);
          // the cache streams through once: its lines go first, so the query
          // rows and the partials written for the merge stay in L2
          for (int j = 0; j < 4; ++j)
            tma_load_2d_hint(dst + j * kBox, &tm_kv, &kv_full[s], 256 * half + 64 * j, row,
                             kv_policy);
          tma_load_2d_hint(dst + 4 * kBox, &tm_kr, &kv_full[s], kLatent + 32 * half, row,
                           kv_policy);
        }
        ++kc;
        return true;
      };
      // Ring stage kc <- query latent columns [256*half + 128*i, +128) of
      // the segment's 128 rows, as two boxes of 64 columns (the softmax
      // warps move them into TMEM and the MMA thread frees the stage).
      auto load_q_stage = [&](int i) -> bool {
        const int s = kc % kStages;
        if (kc >= kStages && !mbar_wait(&kv_empty[s], ((kc / kStages) - 1) & 1, abort_flag))
          return false;
        if (lane == 0) {
          uint8_t *dst = sm_kv + s * kStageBytes;
          mbar_arrive_expect_tx(&kv_full[s], F::kQStageBytes);
          for (int j = 0; j < 2; ++j)
            tma_load_2d(dst + j * F::kQBox, &tm_ql, &kv_full[s], 256 * half + 64 * (2 * i + j),
                        sg.row0);
        }
        ++kc;
        return true;
      };
      // The first segment's query rope half goes out before anything else
      // (nothing is in flight yet and QK(0) needs it).  Every segment's
      // query latent half comes next, ahead of its KV tiles: a later
      // segment's is read into TMEM as soon as the previous segment's last
      // QK is done.  A later segment then loads its first KV tile and its
      // query rope half: the previous segment's last QK (which frees the
      // rope buffer) completes about when the stage of this first tile
      // frees up.
      const bool first = nseg == 0;
      if (first && lane == 0) {
        mbar_arrive_expect_tx(q_full, kQRopeBytes);
        tma_load_2d(sm_q, &tm_qr, q_full, kLatent + 32 * half, sg.row0);
      }
      if (!(ok = load_q_stage(0) && load_q_stage(1))) break;
      const int pre = min(sg.ntiles, 1);
      for (int t = 0; ok && t < pre; ++t) ok = load_tile(sg.tile0 + t);
      if (!ok) break;
      if (!first) {
        if (!(ok = mbar_wait(q_free, (nseg - 1) & 1, abort_flag))) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(q_full, kQRopeBytes);
          tma_load_2d(sm_q, &tm_qr, q_full, kLatent + 32 * half, sg.row0);
        }
      }
      ++nseg;
      for (int t = pre; ok && t < sg.ntiles; ++t) ok = load_tile(sg.tile0 + t);
    }
    if (ok) publish(nseg, true);
    if (*abort_flag && lane == 0) {
      volatile int no_abort = 0;
      for (int k = max(0, kc - kStages); k < kc; ++k)
        mbar_wait(&kv_full[k % kStages], (k / kStages) & 1, &no_abort);
      if (nseg > 0) mbar_wait(q_full, (nseg - 1) & 1, &no_abort);
    }
  } else if (is_mma) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      const uint32_t idesc_qk = FP8 ? idesc_e4m3(128, kTile, false, false)
                                    : idesc_bf16(128, kTile, false, false);
      const uint32_t idesc_pv = FP8 ? idesc_e4m3(128, 256, false, true)
                                    : idesc_bf16(128, 256, false, true);
      const uint32_t q_base = smem_u32(sm_q);
      int kc = 0, uc = 0, nseg = 0;
      bool ok = true;
      // `chunk_c` is a std::integral_constant so the descriptor offsets are
      // compile-time constants.
      auto issue_qk_chunk_c = [&](int kcx, int ucx, bool last, auto chunk_c) {
        constexpr int chunk = decltype(chunk_c)::value;
        const uint32_t stage = smem_u32(sm_kv + (kcx % kStages) * kStageBytes);
        const uint32_t d = tmem + kColS + kTile * (ucx & 1);
#pragma unroll
        for (int j = 0; j < kChunkSteps; ++j) {
          const int k = chunk * kChunkSteps + j;
          if (k < F::kLatSteps) {   // latent: A = query half in TMEM, B = own latent boxes
            const uint64_t bdesc =
                sdesc(stage + (k / F::kStepsPerBox) * kBox + (k % F::kStepsPerBox) * 32, 16,
                      F::kSboL, F::kSwL);
            if constexpr (FP8) mma_f8_ts(d, tmem + kColQ + 8 * k, bdesc, idesc_qk, k > 0 ? 1u : 0u);
            else mma_f16_ts(d, tmem + kColQ + 8 * k, bdesc, idesc_qk, k > 0 ? 1u : 0u);
          } else {                  // rope: this CTA's 32 rope columns
            const int kk = k - F::kLatSteps;
            const uint64_t bdesc = sdesc(stage + 4 * kBox + kk * 32, 16, F::kSboR, F::kSwR);
            const uint64_t adesc = sdesc(q_base + kk * 32, 16, F::kSboR, F::kSwR);
            if constexpr (FP8) mma_f8_ss(d, adesc, bdesc, idesc_qk, 1u);
            else mma_f16_ss(d, adesc, bdesc, idesc_qk, 1u);
          }
        }
        if (chunk == kQkChunks - 1) {
          mma_commit(&s_full[ucx & 1]);
          // the segment's last QK: its query rope half in shared memory is
          // no longer read, the next segment's may be loaded
          if (last) mma_commit(q_free);
        }
      };
      // All 18 K steps of one tile's QK as one straight-line burst: the
      // tensor pipe holds only a couple of queued MMAs, so any other work of
      // this thread between MMAs (a barrier test costs ~70 cycles) idles it.
      auto issue_qk = [&](int kcx, int ucx, bool last) {
        issue_qk_chunk_c(kcx, ucx, last, std::integral_constant<int, 0>{});
        issue_qk_chunk_c(kcx, ucx, last, std::integral_constant<int, 1>{});
        issue_qk_chunk_c(kcx, ucx, last, std::integral_constant<int, 2>{});
      };
      // QK of global tile u (ring slot kcx) waits until its KV tile has
      // landed and both row groups have read the scores of tile u-2 out of
      // the same buffer.
      auto qk = [&](int kcx, int ucx, bool last) -> bool {
        if (!mbar_wait(&kv_full[kcx % kStages], (kcx / kStages) & 1, abort_flag)) return false;
        if (ucx >= 2 && !mbar_wait(&s_free[ucx & 1], ((ucx - 2) >> 1) & 1, abort_flag))
          return false;
        tc_fence_after();
        issue_qk(kcx, ucx, last);
        return true;
      };
      while (ok) {
        // segment nseg from the producer's queue
        {
          const int slot = nseg % kSegSlots;
          if (!(ok = mbar_wait(&seg_full[slot], (nseg / kSegSlots) & 1, abort_flag))) break;
          sg = segq[slot];
          mbar_arrive(&seg_empty[slot]);
          if (sg.ntiles < 0) break;
        }
        ok = mbar_wait(q_full, nseg & 1, abort_flag) &&
             mbar_wait(q_tmem, nseg & 1, abort_flag);
        if (!ok) break;
        // the segment's two query stages are in TMEM: their ring slots go
        // back to the producer, and its KV tiles follow them in the ring
        mbar_arrive(&kv_empty[sg.qkc % kStages]);
        mbar_arrive(&kv_empty[(sg.qkc + 1) % kStages]);
        kc = sg.qkc + 2;
        ++nseg;
        // Fixed order, blocking waits: QK of the segment's first two tiles,
        // then for each tile t the QK of tile t+2 (the scores two tiles
        // ahead, which the score buffers allow) and the P.V of tile t.  The
        // scores of tile t are read before its probabilities exist, so
        // QK(t+2) is ready before P.V(t) and this order never waits on one
        // while the other could go.
        const int n = sg.ntiles;
        for (int u = 0; ok && u < min(2, n); ++u) ok = qk(kc + u, uc + u, u + 1 == n);
        for (int t = 0; ok && t < n; ++t, ++kc, ++uc) {
          if (t + 2 < n && !(ok = qk(kc + 2, uc + 2, t + 3 == n))) break;
          if (!(ok = mbar_wait(&p_full[uc & 1], (uc >> 1) & 1, abort_flag))) break;
          tc_fence_after();
          const uint32_t stage = smem_u32(sm_kv + (kc % kStages) * kStageBytes);
          const uint32_t pbuf = smem_u32(sm_p + (uc & 1) * kPBuf);
#pragma unroll
          for (int kk = 0; kk < kPvSteps; ++kk) {
            // A = P (K-major, 32 bytes of tokens per step); B = the four own
            // latent boxes, MN-major: N-blocks one box apart (LBO), 8-token
            // groups SBO apart, 2 KB of rows per step
            const uint64_t adesc = sdesc(pbuf + kk * 32, 16, F::kSboP, F::kSwP);
            const uint64_t bdesc = sdesc(stage + kk * 2048, kBox, F::kSboL, F::kSwL);
            if constexpr (FP8)
              mma_f8_ss(tmem + kColO, adesc, bdesc, idesc_pv, (t > 0 || kk > 0) ? 1u : 0u);
            else
              mma_f16_ss(tmem + kColO, adesc, bdesc, idesc_pv, (t > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(&kv_empty[kc % kStages]);
          mma_commit(&pv_done[uc & 1]);
        }
      }
      if (!ok) {
        mma_commit(drain);
        volatile int no_abort = 0;
        mbar_wait(drain, 0, &no_abort);
      }
    }
  } else if (is_sender) {
    // ------------------------------- forwarded rows: partial scores out
    // Every tile's partial scores of this warp's 32 rows, in order, each as
    // soon as QK has produced it and the peer has consumed the previous
    // message: TMEM -> s_send (128B-swizzled rows) -> one 8 KB bulk copy
    // into the same place of the peer's s_recv.  The staging buffer is free
    // once this warp's previous copy has been read out of it.
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = tmem + ((quarter * 32u) << 16);
    const int lr = r & 63;
    const int wl = lr >> 5;
    const uint32_t peer_s_recv = peer_smem(s_recv, peer);
    const uint32_t peer_xs_full = peer_smem(xs_full, peer);
    auto warp_ok = [](bool v) { return __all_sync(0xffffffffu, v); };
    int ns = 0, k = 0;
    bool ok = true;
    while (ok) {
      const int slot = ns % kSegSlots;
      if (!warp_ok(mbar_wait(&seg_full[slot], (ns / kSegSlots) & 1, abort_flag))) break;
      const int ntiles = segq[slot].ntiles;
      __syncwarp();
      if (lane == 0) mbar_arrive(&seg_empty[slot]);
      ++ns;
      if (ntiles < 0) break;
      for (int t = 0; t < ntiles; ++t, ++k) {
        if (!warp_ok(mbar_wait(&s_full[k & 1], (k >> 1) & 1, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sv[kTile];
        tmem_ld_x32(lane_base + kColS + kTile * (k & 1), sv);
        tmem_ld_x32(lane_base + kColS + kTile * (k & 1) + 32, sv + 32);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&s_free[k & 1]);   // this warp's score rows are read
          bulk_wait_read_all();          // its copy of tile k-1 has left s_send
        }
        __syncwarp();
        uint4 *dst = reinterpret_cast<uint4 *>(s_send + lr * 256);
#pragma unroll
        for (int j = 0; j < 16; ++j)
          dst[j ^ (lr & 15)] = make_uint4(sv[4 * j], sv[4 * j + 1], sv[4 * j + 2], sv[4 * j + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (k > 0 && !warp_ok(mbar_wait(xs_free, (k - 1) & 1, abort_flag))) {
          ok = false;
          break;
        }
        if (lane == 0)
          bulk_copy_to_peer(peer_s_recv + wl * (kSMsg / 2), s_send + wl * (kSMsg / 2),
                            kSMsg / 2, peer_xs_full);
      }
    }
  } else {
    // ------------------- softmax (own rows) / probabilities in (forwarded)
    const int r = quarter * 32 + lane;        // head row within the group
    const uint32_t lane_base = tmem + ((quarter * 32u) << 16);
    const int tid = threadIdx.x - 128;        // 0..127
    const int lr = r & 63;                    // row within a message
    const bool leader = lr == 0;              // one thread per 64-thread group
    const int wl = lr >> 5;                   // warp within the group
    const uint32_t peer_xs_free = peer_smem(xs_free, peer);
    int uc = 0;
    bool ok = true;
    // a timed-out wait ends the loop for the whole warp at once, so no
    // warp-collective operation is left waiting for a lane that has gone
    auto warp_ok = [](bool v) { return __all_sync(0xffffffffu, v); };
    // Query latent dims [256*half, 256*half + 256) of row r -> TMEM columns
    // [kColQ, kColQ + F::kQCols): two bf16 or four e4m3 per 32-bit column.
    // The segment's query latent half: this thread's row out of the two
    // ring stages (swizzled 16-byte chunks, conflict-free across a warp),
    // then into TMEM; false on a timeout.
    auto load_q_tmem = [&](const Seg &seg) -> bool {
      constexpr int kCh = F::kQRow / 16;   // 16-byte chunks per box row
      const bool valid = r < seg.hrows;
      uint32_t w[F::kQCols];
#pragma unroll
      for (int st = 0; st < 2; ++st) {
        const int qs = seg.qkc + st;
        if (!warp_ok(mbar_wait(&kv_full[qs % kStages], (qs / kStages) & 1, abort_flag)))
          return false;
        const uint8_t *stage = sm_kv + (qs % kStages) * kStageBytes;
#pragma unroll
        for (int bx = 0; bx < 2; ++bx) {
          const uint4 *row = reinterpret_cast<const uint4 *>(stage + bx * F::kQBox + r * F::kQRow);
#pragma unroll
          for (int c = 0; c < kCh; ++c) {
            uint4 v = row[FP8 ? (c ^ ((r >> 1) & 3)) : (c ^ (r & 7))];
            if (!valid) v = make_uint4(0, 0, 0, 0);
            const int k = 4 * ((2 * st + bx) * kCh + c);
            w[k] = v.x; w[k + 1] = v.y; w[k + 2] = v.z; w[k + 3] = v.w;
          }
        }
      }
#pragma unroll
      for (int c = 0; c < F::kQCols / 32; ++c) tmem_st_x32(lane_base + kColQ + 32 * c, w + 32 * c);
      tc_fence_before();
      mbar_arrive(q_tmem);
      return true;
    };
    // Takes the next segment descriptor from the producer's queue
    // (warp-wide); false at the end marker or on a timeout (then ok = false).
    int ns = 0;
    auto take_seg = [&](Seg &out) -> bool {
      const int slot = ns % kSegSlots;
      if (!warp_ok(mbar_wait(&seg_full[slot], (ns / kSegSlots) & 1, abort_flag))) {
        ok = false;
        return false;
      }
      out = segq[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&seg_empty[slot]);
      ++ns;
      return out.ntiles >= 0;
    };
    bool have = take_seg(sg);
    if (have) ok = load_q_tmem(sg);
    Seg nxt;
    bool have_next = false;
    float l_in = 1.f;   // forwarded rows: the owner's running sum, last message
    while (ok && have) {
      // running max and sum; lq (e4m3) sums the rounded probabilities
      float m = -INFINITY, l = 0.f, lq = 0.f;
      const int len = sg.len;
      for (int t = 0; t < sg.ntiles; ++t, ++uc) {
        const int sb = uc & 1;
        uint8_t *pbuf = sm_p + sb * kPBuf;
        if (own) {
          // ---------------------------------------------- online softmax
          ok = warp_ok(mbar_wait(&s_full[sb], (uc >> 1) & 1, abort_flag));
          if (!ok) break;
          tc_fence_after();
          uint32_t sr[kTile];   // this CTA's partial scores of row r
          tmem_ld_x32(lane_base + kColS + kTile * sb, sr);
          tmem_ld_x32(lane_base + kColS + kTile * sb + 32, sr + 32);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&s_free[sb]);   // this warp's score rows are read
          if (leader) mbar_arrive_expect_tx(xs_full, kSMsg);
          ok = warp_ok(mbar_wait(xs_full, uc & 1, abort_flag));
          if (!ok) break;
          const int pos0 = (sg.tile0 + t) * kTile;
          const bool full_tile = pos0 >= sg.lo && pos0 + kTile <= sg.hi;
          const uint4 *src = reinterpret_cast<const uint4 *>(s_recv + lr * 256);
          // Full scores s = own partial + the peer's (paired adds); the tile
          // max is taken on s and scaled once (exact: scaling by a positive
          // constant keeps the order and rounds each product alike), and
          // the exponent s * scale - m is one paired FMA below.
          float x[kTile];
          float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const uint4 v = src[k ^ (lr & 15)];
            add_f32x2(x[4 * k], x[4 * k + 1], __uint_as_float(sr[4 * k]),
                      __uint_as_float(sr[4 * k + 1]), __uint_as_float(v.x), __uint_as_float(v.y));
            add_f32x2(x[4 * k + 2], x[4 * k + 3], __uint_as_float(sr[4 * k + 2]),
                      __uint_as_float(sr[4 * k + 3]), __uint_as_float(v.z), __uint_as_float(v.w));
          }
          // interior tiles (every position inside [lo, hi)) skip the mask
          if (!full_tile) {
#pragma unroll
            for (int k = 0; k < kTile; ++k) {
              const int pos = pos0 + k;
              x[k] = (pos >= sg.lo && pos < sg.hi) ? x[k] : -INFINITY;
            }
          }
#pragma unroll
          for (int k = 0; k < kTile; k += 2) mx[(k >> 1) & 3] = fmax3(mx[(k >> 1) & 3], x[k], x[k + 1]);
          __syncwarp();
          if (lane == 0) mbar_arrive_remote(peer_xs_free);   // this warp's rows of s_recv are consumed
          const float tmax =
              fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * args.scale_log2;
          float alpha = 1.f;
          if (t > 0) {
            const float m_new = fmaxf(m, tmax);
            const bool need = m_new > m + kRescaleLog2;
            if (__any_sync(0xffffffffu, need)) {
              const int up = uc - 1;
              ok = warp_ok(mbar_wait(&pv_done[up & 1], (up >> 1) & 1, abort_flag));
              if (!ok) break;
              tc_fence_after();
              alpha = need ? ex2(m - m_new) : 1.f;
#pragma unroll 1
              for (int c = 0; c < 256; c += 32) {
                uint32_t o[32];
                tmem_ld_x32(lane_base + kColO + c, o);
#pragma unroll
                for (int k = 0; k < 32; ++k)
                  o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
                tmem_st_x32(lane_base + kColO + c, o);
              }
              l *= alpha;
              lq *= alpha;
              if (need) m = m_new;
            }
          } else {
            m = tmax;
          }
          // p = 2^(s * scale - m): paired FMAs, then the hardware ex2; the
          // row sum accumulates in pairs (four chains).  It serves both the
          // LSE and the normalisation of O (bf16 rounding of P moves the
          // weights by ~2^-9 relative, far inside the output tolerance).
          const float nm = -m, sc = args.scale_log2;
#pragma unroll
          for (int k = 0; k < kTile; k += 2)
            fma_f32x2(x[k], x[k + 1], x[k], x[k + 1], sc, sc, nm, nm);
#pragma unroll
          for (int k = 0; k < kTile; ++k) x[k] = ex2(x[k]);
          float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int k = 0; k < kTile; k += 4) {
            add_f32x2(ps[0], ps[1], ps[0], ps[1], x[k], x[k + 1]);
            add_f32x2(ps[2], ps[3], ps[2], ps[3], x[k + 2], x[k + 3]);
          }
          l += (ps[0] + ps[1]) + (ps[2] + ps[3]);
          // P for the P.V operand: bf16 pairs, or e4m3 quads, whose rounding
          // is coarse enough that O is normalised by the sum of the rounded
          // values (lq) while the LSE keeps the unrounded sum
          constexpr int kPk = FP8 ? kTile / 4 : kTile / 2;
          uint32_t pk[kPk];
          if constexpr (FP8) {
            float qs[2] = {0.f, 0.f};
#pragma unroll
            for (int k = 0; k < kPk; ++k) {
              pk[k] = pack_e4m3x4(x[4 * k], x[4 * k + 1], x[4 * k + 2], x[4 * k + 3]);
              __half2_raw h0 = __nv_cvt_fp8x2_to_halfraw2(
                  static_cast<__nv_fp8x2_storage_t>(pk[k] & 0xFFFFu), __NV_E4M3);
              __half2_raw h1 = __nv_cvt_fp8x2_to_halfraw2(
                  static_cast<__nv_fp8x2_storage_t>(pk[k] >> 16), __NV_E4M3);
              const float2 f0 = __half22float2(*reinterpret_cast<__half2 *>(&h0));
              const float2 f1 = __half22float2(*reinterpret_cast<__half2 *>(&h1));
              qs[k & 1] += (f0.x + f0.y) + (f1.x + f1.y);
            }
            lq += qs[0] + qs[1];
          } else {
#pragma unroll
            for (int k = 0; k < kPk; ++k) pk[k] = pack_bf16(x[2 * k], x[2 * k + 1]);
          }
          // P tile `sb` and the factor slot are free once P.V of tile uc-2
          // is done here (and the copy out of them has landed) and in the
          // peer (which takes our rows into its own P tile)
          if (uc >= 2) {
            const int up = uc - 2;
            ok = warp_ok(mbar_wait(&pv_done[sb], (up >> 1) & 1, abort_flag) &&
                         mbar_wait(&pb_free[sb], (up >> 1) & 1, abort_flag));
            if (!ok) break;
          }
          // row r of the K-major P operand: 8 chunks of 8 bf16 tokens,
          // 128B-swizzled, or 4 chunks of 16 e4m3 tokens, 64B-swizzled (the
          // 16-byte chunk index XOR the address bits above the row pair)
          uint4 *prow = reinterpret_cast<uint4 *>(pbuf + r * F::kPRow);
#pragma unroll
          for (int j = 0; j < kPk / 4; ++j)
            prow[FP8 ? (j ^ ((r >> 1) & 3)) : (j ^ (r & 7))] =
                make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
          // factors of this warp's rows: alpha[32] then the normaliser of O
          // (the running sum l, or lq for e4m3 P) [32]
          float *al = reinterpret_cast<float *>(al_send + sb * kAlMsg + wl * (kAlMsg / 2));
          al[lane] = alpha;
          al[32 + lane] = FP8 ? lq : l;
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            // this warp's 32 rows of P (contiguous) and their factors -> the
            // same places in the peer
            const uint32_t xbar = peer_smem(&xp_full[sb], peer);
            uint8_t *rows = pbuf + (64 * half + 32 * wl) * F::kPRow;
            bulk_copy_to_peer(peer_smem(rows, peer), rows, 32 * F::kPRow, xbar);
            uint8_t *al_dst = al_recv + sb * kAlMsg + wl * (kAlMsg / 2);
            bulk_copy_to_peer(peer_smem(al_dst, peer), al, kAlMsg / 2, xbar);
          }
        } else {
          // ------------------------------------- forwarded rows: P back
          // Our P.V of tile uc-2 is done: the peer may overwrite our P tile
          // `sb` with its rows of tile uc.
          if (leader && uc >= 2) {
            const int up = uc - 2;
            if (mbar_wait(&pv_done[sb], (up >> 1) & 1, abort_flag))
              mbar_arrive_remote(peer_smem(&pb_free[sb], peer));
          }
          if (leader) mbar_arrive_expect_tx(&xp_full[sb], kPMsg);
          ok = warp_ok(mbar_wait(&xp_full[sb], (uc >> 1) & 1, abort_flag));
          if (!ok) break;
          // the peer's P rows are already in our P tile; apply its factors
          const float *al =
              reinterpret_cast<const float *>(al_recv + sb * kAlMsg + wl * (kAlMsg / 2));
          const float alpha = al[lane];
          l_in = al[32 + lane];
          if (t > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
            const int up = uc - 1;
            ok = warp_ok(mbar_wait(&pv_done[up & 1], (up >> 1) & 1, abort_flag));
            if (!ok) break;
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < 256; c += 32) {
              uint32_t o[32];
              tmem_ld_x32(lane_base + kColO + c, o);
#pragma unroll
              for (int k = 0; k < 32; ++k)
                o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
              tmem_st_x32(lane_base + kColO + c, o);
            }
          }
        }
        const int pos0 = (sg.tile0 + t) * kTile;
        if (pos0 + kTile > len) {
          // cache rows past seq_len may hold anything (even NaN bits): zero
          // them in this CTA's value boxes so that P = 0 contributes nothing
          const int first = max(0, len - pos0);
          const int nrows = kTile - first;
          // (every 16-byte chunk of a row: the swizzle only permutes them)
          constexpr int kCh = 4 * F::kEsz;   // 16-byte chunks per box row
          uint8_t *vbase = sm_kv + ((sg.qkc + 2 + t) % kStages) * kStageBytes;
          for (int idx = tid; idx < nrows * 4 * kCh; idx += 128) {
            const int box = idx / (nrows * kCh);
            const int rem = idx - box * nrows * kCh;
            reinterpret_cast<uint4 *>(vbase + box * kBox + (first + rem / kCh) * 16 * kCh)[rem % kCh] =
                make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        tc_fence_before();
        mbar_arrive(&p_full[sb]);
        if (t + 1 == sg.ntiles) {
          // QK of this segment is complete (this thread has waited for the
          // last tile's scores), so the next segment's query can go into
          // TMEM now, overlapping the last P.V and the exchange with the peer
          have_next = take_seg(nxt);
          if (!ok) break;
          if (have_next && !(ok = load_q_tmem(nxt))) break;
        }
      }
      if (!ok) break;
      {
        const int up = uc - 1;  // the last PV of this segment (all earlier ones are done too)
        ok = warp_ok(mbar_wait(&pv_done[up & 1], (up >> 1) & 1, abort_flag));
      }
      if (!ok) break;
      tc_fence_after();
      // The epilogue stages through the P tiles: every bulk copy out of
      // them (this CTA's rows of P to the peer) must have been read first.
      if (lane == 0) {
        bulk_wait_read_all();
        mbar_arrive(stage_ok);
      }
      ok = warp_ok(mbar_wait(stage_ok, (ns - 2) & 1, abort_flag));   // segment ns-2
      if (!ok) break;
      const Seg cur = sg;
      sg = nxt;
      have = have_next;
      // ---- epilogue: O / l for this CTA's 256 latent columns, all rows,
      // with plain stores: each 128-byte piece of a row (32 fp32 or 64 bf16
      // columns) goes through one of two 4 KB staging buffers of this warp
      // in the idle P tiles and leaves as whole 128-byte rows, four rows per
      // store instruction.  Nothing waits on the stores; tensor-map stores
      // from the same buffers would wait for the TMA engine to read each
      // one, behind the next segment's KV loads (~3.5 us per epilogue).
      const float inv = args.out_scale / (own ? (FP8 ? lq : l) : l_in);
      const bool row_ok = r < cur.hrows;
      // partials take the output's type (a bf16 output is rounded to bf16
      // anyway; the merge adds at most half a bf16 step of each part)
      const bool bf16_out = args.out_dtype == MLA_BF16;
      const int esz = bf16_out ? 2 : 4;
      // a partial slot always has 128 rows; whole-job rows past the head
      // count belong to the next query row and are not written
      const int nrows = cur.whole ? cur.hrows : 128;
      uint8_t *dst0 = cur.whole
          ? static_cast<uint8_t *>(args.out) +
                (static_cast<int64_t>(cur.out_row0) * kLatent + 256 * half) * esz
          : reinterpret_cast<uint8_t *>(args.ws_o) +
                (static_cast<int64_t>(cur.slot) * 128 * kLatent + 256 * half) * esz;
      const int64_t rstride = static_cast<int64_t>(kLatent) * esz;
      uint4 *stg = reinterpret_cast<uint4 *>(sm_p + (warp - 4) * 8192);
#pragma unroll 1
      for (int c = 0; c < 256; c += 64) {
        uint32_t o[64];
        tmem_ld_x64(lane_base + kColO + c, o);
        auto f = [&](int k) { return __uint_as_float(o[k]) * inv; };
        // one (bf16) or two (fp32) 128-byte pieces of this row
#pragma unroll
        for (int pc = 0; pc < 2; ++pc) {
          if (bf16_out && pc == 1) break;
          uint4 *buf = stg + pc * 256;
          __syncwarp();   // the previous use of `buf` has been read out
          if (bf16_out) {
#pragma unroll
            for (int k = 0; k < 8; ++k)
              buf[lane * 8 + (k ^ (lane & 7))] =
                  make_uint4(pack_bf16(f(8 * k), f(8 * k + 1)), pack_bf16(f(8 * k + 2), f(8 * k + 3)),
                             pack_bf16(f(8 * k + 4), f(8 * k + 5)),
                             pack_bf16(f(8 * k + 6), f(8 * k + 7)));
          } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const int e = 32 * pc + 4 * k;
              buf[lane * 8 + (k ^ (lane & 7))] =
                  make_uint4(__float_as_uint(f(e)), __float_as_uint(f(e + 1)),
                             __float_as_uint(f(e + 2)), __float_as_uint(f(e + 3)));
            }
          }
          __syncwarp();
          uint8_t *dst = dst0 + static_cast<int64_t>(c + 32 * pc) * esz;
#pragma unroll
          for (int it = 0; it < 8; ++it) {
            const int row = it * 4 + (lane >> 3), ch = lane & 7;   // 4 rows per instruction
            const int R = quarter * 32 + row;
            if (R < nrows)
              reinterpret_cast<uint4 *>(dst + R * rstride)[ch] = buf[row * 8 + (ch ^ (row & 7))];
          }
        }
      }
      __syncwarp();
      // The P tiles are written again in the next segment (own rows, and
      // the peer's rows after our signal), also by other warps of this CTA:
      // every warp's staging has been read out first.
      if (lane == 0) mbar_arrive(epi_done);
      ok = warp_ok(mbar_wait(epi_done, (ns - 2) & 1, abort_flag));
      if (!ok) break;
      const int64_t orow = static_cast<int64_t>(cur.out_row0 + r);
      if (row_ok && own) {
        const float lse = (m + log2f(l)) * 0.69314718055994531f;
        if (cur.whole) args.lse[orow] = lse;
        else args.ws_lse[static_cast<int64_t>(cur.slot) * 128 + r] = lse;
      }
      tc_fence_before();
    }
  }
  // every bulk copy this CTA issued has landed before either CTA leaves
  bulk_wait_all();
  __syncthreads();
  cluster_sync();
  if (threadIdx.x == 0 && *abort_flag) raise_error(args.err, MLA_DEVERR_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Combines the partials of every job cut into several spans; writes zeros
// and -inf for jobs with an empty key range.  One CTA per (job, 16-row
// block): the 16 rows of one partial are contiguous (32 KB), so each part
// is one bulk copy, with its 16 LSEs, into a 3-deep shared-memory ring (two
// CTAs per SM keep ~190 KB of partials in flight).  Thread t owns row t/16
// and the float4 columns (t%16) + 16k, k < 8 (conflict-free shared reads,
// 128-byte output runs), and folds the parts in with an online rescale, so
// any number of parts works.
namespace mrg {
constexpr int kRows = 16;
constexpr int kRingBytes = 96 * 1024;
constexpr int kLseBytes = kRows * 4;
// Parts are stored in the output's type (T): 16 rows x 512 of them per
// part, a ring of as many as fit in kRingBytes (3 fp32 or 6 bf16 parts).
template <typename T>
struct Geo {
  static constexpr int kPartElems = kRows * kLatent;
  static constexpr int kPartBytes = kPartElems * static_cast<int>(sizeof(T));
  static constexpr int kRing = kRingBytes / kPartBytes;
  static constexpr int kOffLse = kRing * kPartBytes;
  static constexpr int kOffBars = kOffLse + kRing * kLseBytes;
  static constexpr int kSmem = kOffBars + kRing * 8 + 16 + 128;
};
}  // namespace mrg

template <typename Tout>
__global__ void __launch_bounds__(256, 2)
decode_merge_kernel(const int32_t *__restrict__ plan, int J, int q_len, int H, int HG,
                    const Tout *__restrict__ ws_o,
                    const float *__restrict__ ws_lse, Tout *out, float *lse, int *err) {
  using namespace mrg;
  using G = mrg::Geo<Tout>;
  constexpr int kRing = G::kRing, kPartBytes = G::kPartBytes, kPartElems = G::kPartElems;
  constexpr int kOffLse = G::kOffLse, kOffBars = G::kOffBars;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  Tout *parts = reinterpret_cast<Tout *>(smem);
  const float *lses = reinterpret_cast<const float *>(smem + kOffLse);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + kOffBars);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(full + kRing);
  sm100::grid_dep_wait();   // partials of the decode grid
  sm100::grid_dep_launch();
  const int j = blockIdx.x / (128 / kRows), rb = blockIdx.x % (128 / kRows);
  if (j >= J) return;
  const int hg = j % HG;
  if (rb * kRows >= H - hg * 128) return;   // the whole block is past the head count
  const int32_t *sp = plan + 4 + (J + 1);
  const int s0 = sp[j], nseg = sp[j + 1] - s0;
  if (nseg == 1) return;  // written directly by the decode kernel
  const int t = threadIdx.x, lr = t >> 4, q0 = t & 15;
  const int r = rb * kRows + lr;
  float acc[32];
#pragma unroll
  for (int k = 0; k < 32; ++k) acc[k] = 0.f;
  float m = -INFINITY, z = 0.f;
  if (nseg > 0) {
    if (t == 0) {
      for (int b = 0; b < kRing; ++b) mbar_init(&full[b], 1);
      *abort_flag = 0;
      fence_barrier_init();
    }
    __syncthreads();
    int issued = 0;
    auto issue = [&](int s) {   // thread 0
      const int b = s % kRing;
      const int64_t slot = s0 + s;
      mbar_arrive_expect_tx(&full[b], kPartBytes + kLseBytes);
      bulk_load(parts + b * kPartElems, ws_o + (slot * 128 + rb * kRows) * kLatent, kPartBytes,
                &full[b]);
      bulk_load(smem + kOffLse + b * kLseBytes, ws_lse + slot * 128 + rb * kRows, kLseBytes,
                &full[b]);
      ++issued;
    };
    if (t == 0)
      for (int s = 0; s < min(nseg, kRing); ++s) issue(s);
    int s = 0;
    for (; s < nseg; ++s) {
      const int b = s % kRing;
      mbar_wait(&full[b], (s / kRing) & 1, abort_flag);
      if (__syncthreads_or(*abort_flag != 0)) break;   // a timeout ends the loop for all
      const float ls = lses[b * kRows + lr];
      if (ls != -INFINITY) {   // an empty part (weight 0) is never folded in
        const float mn = fmaxf(m, ls);
        const float sc = expf(m - mn), w = expf(ls - mn);
        z = z * sc + w;
        m = mn;
        const Tout *row = parts + b * kPartElems + lr * kLatent;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          float4 v;
          if constexpr (std::is_same<Tout, float>::value) {
            v = reinterpret_cast<const float4 *>(row)[q0 + 16 * k];
          } else {
            const uint2 w = reinterpret_cast<const uint2 *>(row)[q0 + 16 * k];
            v = make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u),
                            __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u));
          }
          acc[4 * k] = fmaf(w, v.x, acc[4 * k] * sc);
          acc[4 * k + 1] = fmaf(w, v.y, acc[4 * k + 1] * sc);
          acc[4 * k + 2] = fmaf(w, v.z, acc[4 * k + 2] * sc);
          acc[4 * k + 3] = fmaf(w, v.w, acc[4 * k + 3] * sc);
        }
      }
      __syncthreads();   // every thread has read buffer b
      if (t == 0 && s + kRing < nseg) issue(s + kRing);
    }
    if (s < nseg) {
      // timed out: the copies still in flight land before the CTA leaves
      if (t == 0) {
        volatile int no_abort = 0;
        for (int u = s; u < issued; ++u) mbar_wait(&full[u % kRing], (u / kRing) & 1, &no_abort);
        raise_error(err, MLA_DEVERR_TIMEOUT);
      }
      return;
    }
  }
  if (hg * 128 + r >= H) return;
  // jobs are token-major: (query token i, request b, head group)
  const int bq = J / (q_len * HG), i = (j / HG) / bq, b = (j / HG) % bq;
  const int64_t orow = static_cast<int64_t>(b * q_len + i) * H + hg * 128 + r;
  const float inv = m == -INFINITY ? 0.f : 1.f / z;
  Tout *dst = out + orow * kLatent;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int c = 4 * (q0 + 16 * k);
    const float a0 = acc[4 * k] * inv, a1 = acc[4 * k + 1] * inv, a2 = acc[4 * k + 2] * inv,
                a3 = acc[4 * k + 3] * inv;
    if constexpr (std::is_same<Tout, float>::value) {
      *reinterpret_cast<float4 *>(dst + c) = make_float4(a0, a1, a2, a3);
    } else {
      *reinterpret_cast<uint2 *>(dst + c) = make_uint2(bf16x2_rn(a0, a1), bf16x2_rn(a2, a3));
    }
  }
  if (q0 == 0) lse[orow] = m == -INFINITY ? -INFINITY : m + logf(z);
}

struct WsLayout {
  size_t plan_off, o_off, lse_off, total;
  int64_t slots;
};

WsLayout ws_layout(int B, int q_len, int H, int max_seq_len, int split_tiles,
                   int groups) {
  const int HG = (H + 127) / 128;
  const int64_t J = static_cast<int64_t>(B) * q_len * HG;
  // a job's key range [lo, hi) with 0 <= lo <= hi <= max_seq_len touches
  // ceil(hi / tile) - floor(lo / tile) <= ceil(max_seq_len / tile) tiles
  // (64 tokens for both formats), plus its switch cost in units
  const int64_t tiles_per_job = (static_cast<int64_t>(max_seq_len) + 63) / 64 + kJobCost;
  const int64_t total_max = J * tiles_per_job;
  const int64_t spans = split_tiles > 0 ? (total_max + split_tiles - 1) / split_tiles
                                        : static_cast<int64_t>(groups);
  WsLayout w;
  w.slots = J + spans;
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  w.plan_off = 0;
  w.o_off = up(plan_ints(static_cast<int>(J)) * sizeof(int32_t));
  w.lse_off = up(w.o_off + static_cast<size_t>(w.slots) * 128 * kLatent * sizeof(float));
  w.total = up(w.lse_off + static_cast<size_t>(w.slots) * 128 * sizeof(float));
  return w;
}

// Launch configuration of the bf16 pair kernel: 2-CTA clusters, with
// programmatic stream serialization after the plan kernel.
struct PairLaunch {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  PairLaunch(int clusters, cudaStream_t stream) {
    cfg.gridDim = dim3(2 * clusters);
    cfg.blockDim = dim3(pair::kThreads);
    cfg.dynamicSmemBytes = pair::kSmem;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
  }
};

// Work groups (CTA pairs) per launch: one per two SMs, capped by how many
// 2-CTA clusters of the pair kernel can be resident at once (a cluster
// needs both SMs in one GPC), so the whole grid runs in a single wave.
// Cached per device.
int groups_for_device() {
  constexpr int kMaxDevices = 64;
  static int cache[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  const int sms = device_sm_count();
  int g = sms >= 2 ? sms / 2 : 1;
  if (dev < 0 || dev >= kMaxDevices) return g;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] > 0) return cache[dev];
  int clusters = 0;
  // (the two formats' kernels have the same launch shape and shared memory)
  if (cudaFuncSetAttribute(decode_pair_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           pair::kSmem) == cudaSuccess) {
    PairLaunch pl(g, nullptr);
    if (cudaOccupancyMaxActiveClusters(&clusters, decode_pair_kernel<false>, &pl.cfg) != cudaSuccess)
      clusters = 0;
  }
  cudaGetLastError();   // a failed query leaves no sticky error behind
  if (clusters > 0) g = std::min(g, clusters);
  cache[dev] = g;
  return g;
}

bool decode_shape_ok(int B, int q_len, int H) {
  if (B < 1 || q_len < 1 || q_len > 64 || H < 1 || H > 4096) return false;
  const int64_t J = static_cast<int64_t>(B) * q_len * ((H + 127) / 128);
  return J <= (1 << 22);
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" int mla_decode_workspace_size(int B, int q_len, int H,
                                         int max_seq_len, int split_tiles,
                                         size_t *bytes) {
  if (!bytes || !decode_shape_ok(B, q_len, H) || max_seq_len < 0 || split_tiles < 0)
    return MLA_ERR_INVALID_ARG;
  const int g = groups_for_device();
  *bytes = ws_layout(B, q_len, H, max_seq_len, split_tiles, g).total;
  return MLA_OK;
}

extern "C" int mla_decode_plan(const int32_t *seq_lens, const int32_t *kv_starts,
                               const int32_t *kv_ends, int B, int q_len, int H,
                               int max_blocks, int causal, int kv_dtype,
                               int split_tiles, int n_groups, int32_t *plan,
                               size_t plan_bytes, mla_stream_t stream) {
  if (!decode_shape_ok(B, q_len, H) || max_blocks < 1 || split_tiles < 0 ||
      n_groups < 0 || !seq_lens || !plan)
    return MLA_ERR_INVALID_ARG;
  if (kv_dtype != MLA_BF16 && kv_dtype != MLA_E4M3) return MLA_ERR_INVALID_ARG;
  const int HG = (H + 127) / 128;
  const int J = B * q_len * HG;
  if (plan_bytes < plan_ints(J) * sizeof(int32_t)) return MLA_ERR_WORKSPACE;
  const int g = n_groups > 0 ? n_groups : groups_for_device();
  int *err = device_error_word();
  if (!err) return MLA_ERR_CUDA;
  const int tile = pair::kTile;   // both formats
  if (launch_plan(seq_lens, kv_starts, kv_ends, B, q_len, HG, max_blocks, causal ? 1 : 0, tile,
                  split_tiles, g, plan, err, stream) != cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}

namespace {

template <bool FP8>
int launch_decode_pair(const void *q, const void *kv_cache, int B, int q_len, int H,
                       int num_blocks, DecodeArgs a, mla_stream_t stream) {
  // KV latent boxes {64 columns, 64 tokens} (128B swizzle for bf16, 64B for
  // e4m3: one box row either way); KV and query rope halves {32 columns,
  // 64 tokens / 128 heads} (64B / 32B swizzle)
  CUtensorMap tm_kv, tm_kr, tm_qr;
  const CUtensorMapDataType dt =
      FP8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUtensorMapSwizzle sw_l = FP8 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
  const CUtensorMapSwizzle sw_r = FP8 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B;
  const uint64_t row_bytes = static_cast<uint64_t>(kDqk) * pair::Fmt<FP8>::kEsz;
  const uint64_t kv_dims[2] = {kDqk, static_cast<uint64_t>(num_blocks) * kPage};
  const uint64_t q_dims[2] = {kDqk, static_cast<uint64_t>(B) * q_len * H};
  const uint64_t strides[1] = {row_bytes};
  const uint32_t box_kv[2] = {64, static_cast<uint32_t>(pair::kTile)};
  const uint32_t box_kr[2] = {32, static_cast<uint32_t>(pair::kTile)};
  const uint32_t box_qr[2] = {32, 128};
  const uint32_t box_ql[2] = {64, 128};
  CUtensorMap tm_ql;
  if (!make_tmap(&tm_kv, dt, 2, kv_cache, kv_dims, strides, box_kv, sw_l) ||
      !make_tmap(&tm_kr, dt, 2, kv_cache, kv_dims, strides, box_kr, sw_r) ||
      !make_tmap(&tm_qr, dt, 2, q, q_dims, strides, box_qr, sw_r) ||
      !make_tmap(&tm_ql, dt, 2, q, q_dims, strides, box_ql, sw_l))
    return MLA_ERR_CUDA;
  if (cudaFuncSetAttribute(decode_pair_kernel<FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           pair::kSmem) != cudaSuccess)
    return MLA_ERR_CUDA;
  PairLaunch pl(a.groups, stream);
  if (cudaLaunchKernelEx(&pl.cfg, decode_pair_kernel<FP8>, tm_kv, tm_kr, tm_qr, tm_ql, a) !=
      cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}

}  // namespace

namespace {

// Host-side validation shared by mla_decode_paged and its no-allocation
// variant: everything but the workspace.
int validate_decode(const void *q, int q_dtype, float q_scale, const void *kv_cache,
                    int kv_dtype, float k_scale, const int32_t *block_table,
                    const int32_t *seq_lens, int B, int q_len, int H, int max_blocks,
                    int num_blocks, float sm_scale, int split_tiles, const void *out,
                    int out_dtype, const float *lse) {
  if (!decode_shape_ok(B, q_len, H) || max_blocks < 1 || num_blocks < 1 ||
      num_blocks >= (1 << 25) || split_tiles < 0)
    return MLA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(max_blocks) * kPage > (1ll << 30))
    return MLA_ERR_INVALID_ARG;
  if (!q || !kv_cache || !block_table || !seq_lens || !out || !lse)
    return MLA_ERR_INVALID_ARG;
  if ((q_dtype != MLA_BF16 && q_dtype != MLA_E4M3) || q_dtype != kv_dtype)
    return MLA_ERR_INVALID_ARG;
  if (out_dtype != MLA_BF16 && out_dtype != MLA_F32) return MLA_ERR_INVALID_ARG;
  if (!(sm_scale > 0.f) || !(sm_scale < INFINITY)) return MLA_ERR_INVALID_ARG;
  if (kv_dtype == MLA_E4M3 && (!(q_scale > 0.f) || !(q_scale < INFINITY) ||
                               !(k_scale > 0.f) || !(k_scale < INFINITY)))
    return MLA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv_cache) || !aligned16(out)) return MLA_ERR_INVALID_ARG;
  return MLA_OK;
}

}  // namespace

extern "C" int mla_decode_paged(const void *q, int q_dtype, float q_scale,
                                const void *kv_cache, int kv_dtype,
                                float k_scale, const int32_t *block_table,
                                const int32_t *seq_lens,
                                const int32_t *kv_starts,
                                const int32_t *kv_ends, int B, int q_len,
                                int H, int max_blocks, int num_blocks,
                                float sm_scale, int causal, int split_tiles,
                                void *out, int out_dtype, float *lse,
                                void *workspace, size_t ws_bytes,
                                mla_stream_t stream) {
  const int v = validate_decode(q, q_dtype, q_scale, kv_cache, kv_dtype, k_scale, block_table,
                                seq_lens, B, q_len, H, max_blocks, num_blocks, sm_scale,
                                split_tiles, out, out_dtype, lse);
  if (v != MLA_OK) return v;
  if (!aligned16(workspace)) return MLA_ERR_INVALID_ARG;
  const bool fp8 = kv_dtype == MLA_E4M3;
  const int g = groups_for_device();
  const WsLayout w = ws_layout(B, q_len, H, max_blocks * kPage, split_tiles, g);
  if (!workspace || ws_bytes < w.total) return MLA_ERR_WORKSPACE;
  int *err = device_error_word();
  if (!err) return MLA_ERR_CUDA;
  const int HG = (H + 127) / 128;
  const int J = B * q_len * HG;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  int32_t *plan = reinterpret_cast<int32_t *>(ws + w.plan_off);
  float *ws_o = reinterpret_cast<float *>(ws + w.o_off);
  float *ws_lse = reinterpret_cast<float *>(ws + w.lse_off);

  const int tile = pair::kTile;   // both formats
  if (launch_plan(seq_lens, kv_starts, kv_ends, B, q_len, HG, max_blocks, causal ? 1 : 0, tile,
                  split_tiles, g, plan, err, stream) != cudaSuccess)
    return MLA_ERR_CUDA;

  DecodeArgs a{};
  a.plan = plan;
  a.J = J;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.q = static_cast<const uint8_t *>(q);
  a.q_len = q_len;
  a.H = H;
  a.HG = HG;
  a.max_blocks = max_blocks;
  a.num_blocks = num_blocks;
  a.groups = g;
  a.scale_log2 = sm_scale * 1.4426950408889634f * (fp8 ? q_scale * k_scale : 1.f);
  a.out_scale = fp8 ? k_scale : 1.f;
  a.out = out;
  a.out_dtype = out_dtype;
  a.lse = lse;
  a.ws_o = ws_o;
  a.ws_lse = ws_lse;
  a.err = err;
  const int st = fp8 ? launch_decode_pair<true>(q, kv_cache, B, q_len, H, num_blocks, a, stream)
                     : launch_decode_pair<false>(q, kv_cache, B, q_len, H, num_blocks, a, stream);
  if (st != MLA_OK) return st;

  const dim3 mgrid(static_cast<unsigned>(J) * (128 / mrg::kRows));
  const int32_t *cplan = plan;
  const float *cws_lse = ws_lse;
  cudaError_t e;
  if (out_dtype == MLA_BF16) {
    // the partials were written in bf16
    constexpr int smem = mrg::Geo<__nv_bfloat16>::kSmem;
    e = cudaFuncSetAttribute(decode_merge_kernel<__nv_bfloat16>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess)
      e = launch_pdl(decode_merge_kernel<__nv_bfloat16>, mgrid, dim3(256), smem, stream, cplan, J,
                     q_len, H, HG, reinterpret_cast<const __nv_bfloat16 *>(ws_o), cws_lse,
                     static_cast<__nv_bfloat16 *>(out), lse, err);
  } else {
    constexpr int smem = mrg::Geo<float>::kSmem;
    e = cudaFuncSetAttribute(decode_merge_kernel<float>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess)
      e = launch_pdl(decode_merge_kernel<float>, mgrid, dim3(256), smem, stream, cplan, J, q_len,
                     H, HG,
                     static_cast<const float *>(ws_o), cws_lse, static_cast<float *>(out), lse,
                     err);
  }
  return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

// ------------------------------------------------- no-allocation variant
namespace {

// Scratch of mla_decode_paged_noalloc: the plan and the split partials.
static __device__ __align__(256) uint8_t g_noalloc_scratch[MLA_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch on the current device, looked up once
// per device (in host code the symbol is only a stand-in, not an address).
void *noalloc_scratch() {
  constexpr int kMaxDev = 64;
  static std::mutex mu;
  static void *addr[kMaxDev] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace

extern "C" int mla_decode_paged_noalloc(
    const void *q, int q_dtype, float q_scale, const void *kv_cache, int kv_dtype,
    float k_scale, const int32_t *block_table, const int32_t *seq_lens,
    const int32_t *kv_starts, const int32_t *kv_ends, int B, int q_len, int H,
    int max_blocks, int num_blocks, float sm_scale, int causal, int split_tiles,
    void *out, int out_dtype, float *lse, mla_stream_t stream) {
  // every argument check of mla_decode_paged first, then the scratch size
  const int v = validate_decode(q, q_dtype, q_scale, kv_cache, kv_dtype, k_scale, block_table,
                                seq_lens, B, q_len, H, max_blocks, num_blocks, sm_scale,
                                split_tiles, out, out_dtype, lse);
  if (v != MLA_OK) return v;
  const WsLayout w = ws_layout(B, q_len, H, max_blocks * kPage, split_tiles,
                               groups_for_device());
  if (w.total > MLA_NOALLOC_SCRATCH_BYTES) return MLA_ERR_WORKSPACE;
  void *ws = noalloc_scratch();
  if (!ws) return MLA_ERR_CUDA;
  return mla_decode_paged(q, q_dtype, q_scale, kv_cache, kv_dtype, k_scale,
                          block_table, seq_lens, kv_starts, kv_ends, B, q_len, H,
                          max_blocks, num_blocks, sm_scale, causal, split_tiles, out,
                          out_dtype, lse, ws, MLA_NOALLOC_SCRATCH_BYTES, stream);
}
