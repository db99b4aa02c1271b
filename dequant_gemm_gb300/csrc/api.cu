// The C ABI of libnf4gemm.so: host-side validation, device checks and kernel
// dispatch. Every entry point validates all of its arguments before it
// touches the device, and launches nothing on an invalid call.
#include <mutex>

#include "common.cuh"

namespace {

// Device status word: kernels whose bounded waits run out record
// NF4_ERR_DEVICE_TIMEOUT here; nf4_poll_device_status reads and clears it.
__device__ int g_device_status[2];   // status, site of the first timeout

struct DeviceInfo {
  bool checked = false;
  bool ok = false;
  int num_sms = 0;
  int* status = nullptr;  // device address of g_device_status
};

constexpr int kMaxDevices = 64;
DeviceInfo g_devices[kMaxDevices];
std::mutex g_devices_mu;

// Checks (once per device) that the current device is an sm_103 part and
// records its SM count and the device address of the status word.
nf4_status current_device(DeviceInfo** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return NF4_ERR_DEVICE;
  }
  std::lock_guard<std::mutex> lock(g_devices_mu);
  DeviceInfo& d = g_devices[dev];
  if (!d.checked) {
    int major = 0, minor = 0, sms = 0;
    bool ok = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) == cudaSuccess &&
              cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) == cudaSuccess &&
              cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess;
    ok = ok && major == 10 && minor == 3;
    void* status = nullptr;
    ok = ok && cudaGetSymbolAddress(&status, g_device_status) == cudaSuccess;
    if (!ok) cudaGetLastError();
    d.ok = ok;
    d.num_sms = sms;
    d.status = static_cast<int*>(status);
    d.checked = true;
  }
  if (!d.ok) return NF4_ERR_DEVICE;
  *out = &d;
  return NF4_OK;
}

// Token counts up to these use the streaming small-M kernels; larger ones the
// tensor-memory GEMM.
constexpr int64_t kSmallMFwd = 16;
constexpr int64_t kSmallMDx = 16;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

nf4_status check_weight(const nf4_weight* w) {
  if (!w) return NF4_ERR_NULL;
  if (w->blocksize != nf4::kBlock || w->dq_group != nf4::kGroup) return NF4_ERR_BLOCKSIZE;
  if (w->rows < 0 || w->cols < 0 || (w->cols % nf4::kBlock) != 0) return NF4_ERR_SHAPE;
  return NF4_OK;
}

nf4_status check_weight_ptrs(const nf4_weight* w) {
  if (!w->codes || !w->absmax_q || !w->absmax_scale) return NF4_ERR_NULL;
  if (!aligned16(w->codes) || !aligned16(w->absmax_q) || !aligned16(w->absmax_scale))
    return NF4_ERR_ALIGN;
  return NF4_OK;
}

nf4_status launched(cudaError_t e) {
  if (e == cudaSuccess) return NF4_OK;
  cudaGetLastError();
  return NF4_ERR_LAUNCH;
}

}  // namespace

extern "C" {

nf4_status nf4_quantize(const float* W, int64_t rows, int64_t cols, int32_t blocksize,
                        uint8_t* codes, uint8_t* absmax_q, float* absmax_scale, void* stream) {
  if (blocksize != nf4::kBlock) return NF4_ERR_BLOCKSIZE;
  if (rows < 0 || cols < 0 || (cols % nf4::kBlock) != 0) return NF4_ERR_SHAPE;
  if (rows == 0 || cols == 0) return NF4_OK;
  if (!W || !codes || !absmax_q || !absmax_scale) return NF4_ERR_NULL;
  if (!aligned16(W) || !aligned16(codes) || !aligned16(absmax_q) || !aligned16(absmax_scale))
    return NF4_ERR_ALIGN;
  DeviceInfo* d = nullptr;
  if (nf4_status s = current_device(&d)) return s;
  return launched(nf4::launch_quantize(W, rows * cols, codes, absmax_q, absmax_scale,
                                       static_cast<cudaStream_t>(stream)));
}

nf4_status nf4_dequantize(const nf4_weight* w, float* W_out, void* stream) {
  if (nf4_status s = check_weight(w)) return s;
  if (w->rows == 0 || w->cols == 0) return NF4_OK;
  if (nf4_status s = check_weight_ptrs(w)) return s;
  if (!W_out) return NF4_ERR_NULL;
  if (!aligned16(W_out)) return NF4_ERR_ALIGN;
  DeviceInfo* d = nullptr;
  if (nf4_status s = current_device(&d)) return s;
  return launched(nf4::launch_dequantize(w->codes, w->absmax_q, w->absmax_scale,
                                         w->rows * w->cols, W_out,
                                         static_cast<cudaStream_t>(stream)));
}

nf4_status nf4_matmul_fwd(const uint16_t* X, int64_t M, const nf4_weight* w, float* Y,
                          void* stream) {
  if (nf4_status s = check_weight(w)) return s;
  if (M < 0 || (w->rows % 8) != 0) return NF4_ERR_SHAPE;
  if (M == 0 || w->rows == 0) return NF4_OK;
  if (w->cols == 0) {  // an empty reduction: Y = 0
    if (!Y) return NF4_ERR_NULL;
    return launched(cudaMemsetAsync(Y, 0, static_cast<size_t>(M) * w->rows * sizeof(float),
                                    static_cast<cudaStream_t>(stream)));
  }
  if (nf4_status s = check_weight_ptrs(w)) return s;
  if (!X || !Y) return NF4_ERR_NULL;
  if (!aligned16(X) || !aligned16(Y)) return NF4_ERR_ALIGN;
  DeviceInfo* d = nullptr;
  if (nf4_status s = current_device(&d)) return s;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (M <= kSmallMFwd && w->cols <= nf4::kGemvMaxCols)
    return launched(nf4::launch_gemv_fwd(X, M, w->codes, w->absmax_q, w->absmax_scale, w->rows,
                                         w->cols, Y, d->num_sms, d->status, st));
  return launched(nf4::launch_tc_fwd(X, M, w->codes, w->absmax_q, w->absmax_scale, w->rows,
                                     w->cols, Y, d->num_sms, d->status, st));
}

nf4_status nf4_matmul_bwd_dx(const uint16_t* dY, int64_t M, const nf4_weight* w, float* dX,
                             void* stream) {
  if (nf4_status s = check_weight(w)) return s;
  if (M < 0 || (w->rows % 8) != 0) return NF4_ERR_SHAPE;
  if (M == 0 || w->cols == 0) return NF4_OK;
  if (w->rows == 0) {  // an empty reduction: dX = 0
    if (!dX) return NF4_ERR_NULL;
    return launched(cudaMemsetAsync(dX, 0, static_cast<size_t>(M) * w->cols * sizeof(float),
                                    static_cast<cudaStream_t>(stream)));
  }
  if (nf4_status s = check_weight_ptrs(w)) return s;
  if (!dY || !dX) return NF4_ERR_NULL;
  if (!aligned16(dY) || !aligned16(dX)) return NF4_ERR_ALIGN;
  DeviceInfo* d = nullptr;
  if (nf4_status s = current_device(&d)) return s;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (M <= kSmallMDx)
    return launched(nf4::launch_simt_dx(dY, M, w->codes, w->absmax_q, w->absmax_scale, w->rows,
                                        w->cols, dX, d->num_sms, st));
  return launched(nf4::launch_tc_dx(dY, M, w->codes, w->absmax_q, w->absmax_scale, w->rows,
                                    w->cols, dX, d->num_sms, d->status, st));
}

nf4_status nf4_poll_device_status_site(void* stream, int32_t* site) {
  if (site) *site = 0;
  DeviceInfo* d = nullptr;
  if (nf4_status s = current_device(&d)) return s;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) {
    cudaGetLastError();
    return NF4_ERR_LAUNCH;
  }
  int value[2] = {0, 0};
  const int zero[2] = {0, 0};
  if (cudaMemcpyAsync(value, d->status, sizeof(value), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaMemcpyAsync(d->status, zero, sizeof(zero), cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess) {
    cudaGetLastError();
    return NF4_ERR_LAUNCH;
  }
  if (site) *site = value[1];
  return value[0] == 0 ? NF4_OK : static_cast<nf4_status>(value[0]);
}

nf4_status nf4_poll_device_status(void* stream) {
  return nf4_poll_device_status_site(stream, nullptr);
}

nf4_status nf4_codebook(float* out16) {
  if (!out16) return NF4_ERR_NULL;
  for (int i = 0; i < 16; ++i) out16[i] = nf4::bits_to_float(nf4::kLevelBits[i]);
  return NF4_OK;
}

const char* nf4_status_string(nf4_status status) {
  switch (status) {
    case NF4_OK: return "ok";
    case NF4_ERR_NULL: return "a required pointer is NULL";
    case NF4_ERR_SHAPE: return "unsupported or negative shape";
    case NF4_ERR_ALIGN: return "a pointer is not 16-byte aligned";
    case NF4_ERR_BLOCKSIZE: return "blocksize must be 64 and dq_group 256";
    case NF4_ERR_DEVICE: return "no current CUDA device, or it is not sm_103";
    case NF4_ERR_LAUNCH: return "the CUDA runtime rejected a launch or the stream holds an error";
    case NF4_ERR_DEVICE_TIMEOUT: return "a kernel's bounded wait ran out";
  }
  return "unknown status";
}

}  // extern "C"
