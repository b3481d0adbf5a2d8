// Host staging: moves a step's packed inputs from page-locked host memory
// into device memory, or its packed results back, with the SMs' own loads
// and stores over the host link instead of a copy-engine transfer.
//
// A decode step's host traffic is small (1.6 MB of query in, 1.1 MB of
// output back at B = 32, H = 128) and a copy-engine transfer of that size
// is dominated by its fixed cost; many CTAs each keeping several 16-byte
// loads in flight reach the link's bandwidth instead.  The kernel is a
// plain grid-stride copy: every thread issues its loads for one round of
// kUnroll chunks before the stores, so each SM keeps
// kThreads * kUnroll * 16 bytes in flight.
//
// No page defines this step; it is the transfer the serving loop around
// the decode chain performs ("DeepSeek MLA 在 DCP 分布式环境中的 Prefill 阶段解析",
// §MLA Prefill vs Decode: per-step query in, attention output out).
#include "common.cuh"
#include "sm100.cuh"

namespace mla {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

__global__ void __launch_bounds__(kThreads)
stage_copy_kernel(uint4 *__restrict__ dst, const uint4 *__restrict__ src, size_t n16) {
  // the source may be the previous grid's output
  sm100::grid_dep_wait();
  sm100::grid_dep_launch();
  const size_t stride = static_cast<size_t>(gridDim.x) * kThreads;
  for (size_t base = static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x; base < n16;
       base += stride * kUnroll) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const size_t i = base + u * stride;
      if (i < n16) v[u] = src[i];
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const size_t i = base + u * stride;
      if (i < n16) dst[i] = v[u];
    }
  }
}

// Device-visible address of `p` and whether it is page-locked host memory
// (true) or memory of the current device (false); false return if it is
// neither (pageable host memory, another device's memory, an unknown
// pointer).
bool classify(const void *p, int device, void **dev_ptr, bool *is_host) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();   // clear the (non-sticky) error an unknown pointer leaves
    return false;
  }
  if (a.type == cudaMemoryTypeHost) {
    if (!a.devicePointer) return false;   // page-locked but not mapped
    *dev_ptr = a.devicePointer;
    *is_host = true;
    return true;
  }
  if ((a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) && a.device == device &&
      a.devicePointer) {
    *dev_ptr = a.devicePointer;
    *is_host = false;
    return true;
  }
  return false;
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" int mla_stage_copy(void *dst, const void *src, size_t bytes, mla_stream_t stream) {
  if (bytes == 0) return MLA_OK;
  if (!dst || !src || (bytes & 15u) != 0 || !aligned16(dst) || !aligned16(src))
    return MLA_ERR_INVALID_ARG;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return MLA_ERR_CUDA;
  void *d_dst = nullptr, *d_src = nullptr;
  bool dst_host = false, src_host = false;
  if (!classify(dst, device, &d_dst, &dst_host) || !classify(src, device, &d_src, &src_host))
    return MLA_ERR_INVALID_ARG;
  if (dst_host == src_host) return MLA_ERR_INVALID_ARG;   // exactly one side is host memory
  const size_t n16 = bytes / 16;
  const size_t per_cta = static_cast<size_t>(kThreads) * kUnroll;
  const size_t want = (n16 + per_cta - 1) / per_cta;
  const int ctas = static_cast<int>(want < static_cast<size_t>(2 * device_sm_count())
                                        ? want : static_cast<size_t>(2 * device_sm_count()));
  if (launch_pdl(stage_copy_kernel, dim3(ctas), dim3(kThreads), 0,
                 static_cast<cudaStream_t>(stream), static_cast<uint4 *>(d_dst),
                 static_cast<const uint4 *>(d_src), n16) != cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}
