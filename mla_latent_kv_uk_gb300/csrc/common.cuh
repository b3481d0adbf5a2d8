// Shared host/device helpers of the GB300 absorbed-MLA library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "mla.h"

namespace mla {

constexpr int kLatent = 512;   // L
constexpr int kRope = 64;      // R
constexpr int kDqk = 576;      // L + R
constexpr int kNope = 128;     // per-head nope width
constexpr int kVhead = 128;    // per-head value width
constexpr int kPage = 64;      // tokens per cache page

// ---- host side -----------------------------------------------------------

// Device address of the library's error word for the current device.
// Returns nullptr if the symbol cannot be resolved.
int *device_error_word();

// Number of SMs of the current device (cached per device).
int device_sm_count();

// Encodes a tiled TMA descriptor; returns false on failure.  dims/strides
// follow cuTensorMapEncodeTiled (dim 0 innermost, strides in bytes for
// dims 1..rank-1).
bool make_tmap(CUtensorMap *map, CUtensorMapDataType dtype, int rank,
               const void *base, const uint64_t *dims,
               const uint64_t *strides_bytes, const uint32_t *box,
               CUtensorMapSwizzle swizzle);

// Launches `kern` on `stream` with programmatic stream serialization, so it
// may be scheduled while the previous grid in the stream is still running;
// the kernel must call griddepcontrol.wait before reading that grid's output.
template <typename... Params, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(Params...), dim3 grid, dim3 block,
                              size_t smem, cudaStream_t stream, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

inline int launch_status() {
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

inline bool aligned16(const void *p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

// ---- device side ---------------------------------------------------------

__device__ __forceinline__ void raise_error(int *err, int bits) {
  if (err) atomicOr(err, bits);
}

}  // namespace mla
