// Library-wide host plumbing: status strings, the device error word, the
// per-device SM count, TMA descriptor encoding, and the self-test of the
// kernels' bounded waits.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "sm100.cuh"

namespace {

// One error word per device (a __device__ variable has one instance per
// device context); kernels receive its address as an argument.
__device__ int g_error_word;

constexpr int kMaxDevices = 64;

struct PerDevice {
  int *err = nullptr;
  int sms = 0;
  bool init = false;
};

PerDevice g_dev[kMaxDevices];
std::mutex g_mu;

PerDevice *current() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  PerDevice &d = g_dev[dev];
  if (!d.init) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
        cudaSuccess)
      return nullptr;
    d.err = static_cast<int *>(p);
    d.sms = sms;
    d.init = true;
  }
  return &d;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

}  // namespace

namespace mla {

int *device_error_word() {
  PerDevice *d = current();
  return d ? d->err : nullptr;
}

int device_sm_count() {
  PerDevice *d = current();
  return d ? d->sms : 0;
}

bool make_tmap(CUtensorMap *map, CUtensorMapDataType dtype, int rank,
               const void *base, const uint64_t *dims,
               const uint64_t *strides_bytes, const uint32_t *box,
               CUtensorMapSwizzle swizzle) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t gdim[5], gstride[4];
  cuuint32_t bdim[5], estride[5];
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bdim[i] = box[i];
    estride[i] = 1;
    if (i + 1 < rank) gstride[i] = strides_bytes[i];
  }
  CUresult r = fn(map, dtype, static_cast<cuuint32_t>(rank),
                  const_cast<void *>(base), gdim, gstride, bdim, estride,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// One thread waits, through the kernels' bounded wait, on a barrier that
// nothing completes; when the limit runs out it reports like every kernel.
__global__ void selftest_wait_kernel(long long limit_cycles, int *err) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  sm100::mbar_init(&bar, 1);
  abort_flag = 0;
  sm100::fence_barrier_init();
  if (!sm100::mbar_wait_for(&bar, 0, &abort_flag, limit_cycles))
    raise_error(err, MLA_DEVERR_TIMEOUT);
}

}  // namespace mla

extern "C" {

int mla_selftest_wait_timeout(long long limit_cycles, mla_stream_t stream) {
  if (limit_cycles < 1 || limit_cycles > 1000000000LL) return MLA_ERR_INVALID_ARG;
  int *err = mla::device_error_word();
  if (!err) return MLA_ERR_CUDA;
  mla::selftest_wait_kernel<<<1, 32, 0, stream>>>(limit_cycles, err);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

const char *mla_status_string(int status) {
  switch (status) {
    case MLA_OK: return "ok";
    case MLA_ERR_INVALID_ARG: return "invalid argument";
    case MLA_ERR_UNSUPPORTED: return "unsupported configuration";
    case MLA_ERR_WORKSPACE: return "workspace missing or too small";
    case MLA_ERR_CUDA: return "CUDA runtime or launch error";
    default: return "unknown status";
  }
}

int mla_version(void) { return 1; }

int mla_get_device_error(int *code, mla_stream_t stream) {
  if (!code) return MLA_ERR_INVALID_ARG;
  int *w = mla::device_error_word();
  if (!w) return MLA_ERR_CUDA;
  int h = 0;
  if (cudaMemcpyAsync(&h, w, sizeof(int), cudaMemcpyDeviceToHost, stream) !=
      cudaSuccess)
    return MLA_ERR_CUDA;
  if (cudaMemsetAsync(w, 0, sizeof(int), stream) != cudaSuccess)
    return MLA_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MLA_ERR_CUDA;
  *code = h;
  return MLA_OK;
}

}  // extern "C"
