// The C ABI of libnf4gemm.so: host-side validation, device checks and kernel
// dispatch. Every entry point validates all of its arguments before it
// touches the device, and launches nothing on an invalid call.
#include <atomic>
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
  int ordinal = -1;
};

constexpr int kMaxDevices = 64;
DeviceInfo g_devices[kMaxDevices];
std::mutex g_devices_mu;

// Limit of the tensor-core MMA issuer's stage wait, in clock cycles (about a
// second at the GB300's clocks unless a test shortens it).
constexpr long long kDefaultWaitLimit = 1ll << 31;
std::atomic<long long> g_mma_wait_limit{kDefaultWaitLimit};

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
    d.ordinal = dev;
    d.checked = true;
  }
  if (!d.ok) return NF4_ERR_DEVICE;
  *out = &d;
  return NF4_OK;
}

// Token counts up to this use the streaming small-M forward; larger ones,
// and every input gradient, the tensor-memory GEMM.
constexpr int64_t kSmallMFwd = 16;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool is_4bit(int32_t dtype) { return dtype == NF4_DTYPE_NF4 || dtype == NF4_DTYPE_FP4; }
bool valid_dtype(int32_t dtype) { return is_4bit(dtype) || dtype == NF4_DTYPE_INT8; }

nf4_status check_weight(const nf4_weight* w) {
  if (!w) return NF4_ERR_NULL;
  if (!valid_dtype(w->dtype)) return NF4_ERR_SHAPE;
  if (w->blocksize != nf4::kBlock) return NF4_ERR_BLOCKSIZE;
  if (w->dq_group != (is_4bit(w->dtype) ? nf4::kGroup : 0)) return NF4_ERR_BLOCKSIZE;
  if (w->rows < 0 || w->cols < 0 || (w->cols % nf4::kBlock) != 0) return NF4_ERR_SHAPE;
  return NF4_OK;
}

nf4_status check_weight_ptrs(const nf4_weight* w) {
  if (!w->codes || !w->absmax_scale) return NF4_ERR_NULL;
  if (is_4bit(w->dtype) && !w->absmax_q) return NF4_ERR_NULL;
  if (!aligned16(w->codes) || !aligned16(w->absmax_scale)) return NF4_ERR_ALIGN;
  if (is_4bit(w->dtype) && !aligned16(w->absmax_q)) return NF4_ERR_ALIGN;
  return NF4_OK;
}

// The CUDA error behind this thread's last NF4_ERR_LAUNCH.
thread_local cudaError_t t_last_cuda_error = cudaSuccess;

nf4_status launched(cudaError_t e) {
  if (e == cudaSuccess) return NF4_OK;
  t_last_cuda_error = e;
  cudaGetLastError();
  return NF4_ERR_LAUNCH;
}

size_t elem_bytes(int32_t e) { return e == NF4_F32 ? 4 : 2; }

// Validates one fused call without launching anything (the checks of
// matmul below, in its order).
nf4_status check_call(bool dx, const void* act, int32_t act_elem, int64_t M, const nf4_weight* w,
                      const void* out, int32_t out_elem, int32_t flags) {
  if (nf4_status s = check_weight(w)) return s;
  if (act_elem != NF4_BF16 && act_elem != NF4_F16) return NF4_ERR_SHAPE;
  if (out_elem != NF4_F32 && out_elem != NF4_BF16) return NF4_ERR_SHAPE;
  if ((flags & ~NF4_ACCUMULATE) != 0) return NF4_ERR_SHAPE;
  if (M < 0 || (w->rows % 8) != 0) return NF4_ERR_SHAPE;
  const int64_t out_cols = dx ? w->cols : w->rows, red = dx ? w->rows : w->cols;
  if (M == 0 || out_cols == 0) return NF4_OK;
  if (red == 0) return out ? NF4_OK : NF4_ERR_NULL;
  if (nf4_status s = check_weight_ptrs(w)) return s;
  if (!act || !out) return NF4_ERR_NULL;
  if (!aligned16(act) || !aligned16(out)) return NF4_ERR_ALIGN;
  return NF4_OK;
}

// One fused call as the launchers take it (after check_call).
nf4::MatmulCall make_call(const void* act, int32_t act_elem, int64_t M, const nf4_weight* w,
                          void* out, int32_t out_elem, int32_t flags, const DeviceInfo* d,
                          cudaStream_t st) {
  nf4::MatmulCall c;
  c.act = act;
  c.act_f16 = act_elem == NF4_F16;
  c.M = M;
  c.N = w->rows;
  c.K = w->cols;
  c.fmt = w->dtype;
  c.codes = w->codes;
  c.a8 = w->absmax_q;
  c.scale = w->absmax_scale;
  c.out = out;
  c.out_bf16 = out_elem == NF4_BF16;
  c.accumulate = (flags & NF4_ACCUMULATE) != 0;
  c.num_sms = d->num_sms;
  c.status = d->status;
  c.wait_limit = g_mma_wait_limit.load(std::memory_order_relaxed);
  c.device = d->ordinal;
  c.st = st;
  return c;
}

// The shared body of the fused forward and input gradient.
nf4_status matmul(bool dx, const void* act, int32_t act_elem, int64_t M, const nf4_weight* w,
                  void* out, int32_t out_elem, int32_t flags, void* stream) {
  if (nf4_status s = check_call(dx, act, act_elem, M, w, out, out_elem, flags)) return s;
  const int64_t out_cols = dx ? w->cols : w->rows, red = dx ? w->rows : w->cols;
  if (M == 0 || out_cols == 0) return NF4_OK;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (red == 0) {  // an empty reduction: the output is 0 (or unchanged when accumulating)
    if ((flags & NF4_ACCUMULATE) != 0) return NF4_OK;
    return launched(cudaMemsetAsync(out, 0, static_cast<size_t>(M) * out_cols * elem_bytes(out_elem),
                                    st));
  }
  DeviceInfo* d = nullptr;
  if (nf4_status s = current_device(&d)) return s;
  const nf4::MatmulCall c = make_call(act, act_elem, M, w, out, out_elem, flags, d, st);
  if (!dx && M <= kSmallMFwd && w->cols <= nf4::kGemvMaxCols)
    return launched(nf4::launch_gemv_fwd(c));
  return launched(dx ? nf4::launch_tc_dx(c) : nf4::launch_tc_fwd(c));
}

// Forwards of several weights sharing the activations: one small-M launch
// over all their row tiles, else one call per weight.
nf4_status matmul_group(const void* act, int32_t act_elem, int64_t M, const nf4_weight* ws,
                        int32_t count, void* const* outs, int32_t out_elem, int32_t flags,
                        void* stream) {
  if (!ws || !outs) return NF4_ERR_NULL;
  if (count < 1 || count > NF4_GROUP_MAX) return NF4_ERR_SHAPE;
  for (int i = 0; i < count; ++i) {
    if (nf4_status s = check_weight(&ws[i])) return s;
    if (ws[i].cols != ws[0].cols || ws[i].dtype != ws[0].dtype) return NF4_ERR_SHAPE;
  }
  for (int i = 0; i < count; ++i)
    if (nf4_status s = check_call(false, act, act_elem, M, &ws[i], outs[i], out_elem, flags))
      return s;
  const int64_t K = ws[0].cols;
  if (M == 0) return NF4_OK;
  if (M > kSmallMFwd || K == 0 || K > nf4::kGemvMaxCols) {
    for (int i = 0; i < count; ++i)
      if (nf4_status s = matmul(false, act, act_elem, M, &ws[i], outs[i], out_elem, flags, stream))
        return s;
    return NF4_OK;
  }
  DeviceInfo* d = nullptr;
  if (nf4_status s = current_device(&d)) return s;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  nf4::MatmulCall cs[NF4_GROUP_MAX];
  int n = 0;
  for (int i = 0; i < count; ++i)   // weights without rows have nothing to write
    if (ws[i].rows > 0) cs[n++] = make_call(act, act_elem, M, &ws[i], outs[i], out_elem, flags, d, st);
  if (n == 0) return NF4_OK;
  return launched(nf4::launch_gemv_group(cs, n));
}

nf4_status quantize(const void* W, int32_t w_elem, int64_t rows, int64_t cols, int32_t blocksize,
                    int32_t dtype, uint8_t* codes, uint8_t* absmax_q, float* absmax_scale,
                    void* stream) {
  if (blocksize != nf4::kBlock) return NF4_ERR_BLOCKSIZE;
  if (!valid_dtype(dtype) || (w_elem != NF4_F32 && w_elem != NF4_BF16)) return NF4_ERR_SHAPE;
  if (rows < 0 || cols < 0 || (cols % nf4::kBlock) != 0) return NF4_ERR_SHAPE;
  if (rows == 0 || cols == 0) return NF4_OK;
  if (!W || !codes || !absmax_scale) return NF4_ERR_NULL;
  if (is_4bit(dtype) ? !absmax_q : absmax_q != nullptr) return NF4_ERR_NULL;
  if (!aligned16(W) || !aligned16(codes) || !aligned16(absmax_scale)) return NF4_ERR_ALIGN;
  if (is_4bit(dtype) && !aligned16(absmax_q)) return NF4_ERR_ALIGN;
  DeviceInfo* d = nullptr;
  if (nf4_status s = current_device(&d)) return s;
  return launched(nf4::launch_quantize(W, w_elem == NF4_BF16, dtype, rows * cols, codes, absmax_q,
                                       absmax_scale, static_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

nf4_status nf4_quantize(const float* W, int64_t rows, int64_t cols, int32_t blocksize,
                        uint8_t* codes, uint8_t* absmax_q, float* absmax_scale, void* stream) {
  return quantize(W, NF4_F32, rows, cols, blocksize, NF4_DTYPE_NF4, codes, absmax_q, absmax_scale,
                  stream);
}

nf4_status nf4_quantize_ex(const void* W, int32_t w_elem, int64_t rows, int64_t cols,
                           int32_t blocksize, int32_t dtype, uint8_t* codes, uint8_t* absmax_q,
                           float* absmax_scale, void* stream) {
  return quantize(W, w_elem, rows, cols, blocksize, dtype, codes, absmax_q, absmax_scale, stream);
}

nf4_status nf4_dequantize_ex(const nf4_weight* w, void* W_out, int32_t out_elem, void* stream) {
  if (nf4_status s = check_weight(w)) return s;
  if (out_elem != NF4_F32 && out_elem != NF4_BF16 && out_elem != NF4_F16) return NF4_ERR_SHAPE;
  if (w->rows == 0 || w->cols == 0) return NF4_OK;
  if (nf4_status s = check_weight_ptrs(w)) return s;
  if (!W_out) return NF4_ERR_NULL;
  if (!aligned16(W_out)) return NF4_ERR_ALIGN;
  DeviceInfo* d = nullptr;
  if (nf4_status s = current_device(&d)) return s;
  return launched(nf4::launch_dequantize(w->dtype, w->codes, w->absmax_q, w->absmax_scale,
                                         w->rows * w->cols, W_out, out_elem,
                                         static_cast<cudaStream_t>(stream)));
}

nf4_status nf4_dequantize(const nf4_weight* w, float* W_out, void* stream) {
  return nf4_dequantize_ex(w, W_out, NF4_F32, stream);
}

nf4_status nf4_matmul_fwd(const uint16_t* X, int64_t M, const nf4_weight* w, float* Y,
                          void* stream) {
  return matmul(false, X, NF4_BF16, M, w, Y, NF4_F32, 0, stream);
}

nf4_status nf4_matmul_bwd_dx(const uint16_t* dY, int64_t M, const nf4_weight* w, float* dX,
                             void* stream) {
  return matmul(true, dY, NF4_BF16, M, w, dX, NF4_F32, 0, stream);
}

nf4_status nf4_matmul_fwd_group(const void* X, int32_t x_elem, int64_t M, const nf4_weight* ws,
                                int32_t count, void* const* Ys, int32_t y_elem, int32_t flags,
                                void* stream) {
  return matmul_group(X, x_elem, M, ws, count, Ys, y_elem, flags, stream);
}

nf4_status nf4_matmul_fwd_ex(const void* X, int32_t x_elem, int64_t M, const nf4_weight* w,
                             void* Y, int32_t y_elem, int32_t flags, void* stream) {
  return matmul(false, X, x_elem, M, w, Y, y_elem, flags, stream);
}

nf4_status nf4_matmul_bwd_dx_ex(const void* dY, int32_t dy_elem, int64_t M, const nf4_weight* w,
                                void* dX, int32_t dx_elem, int32_t flags, void* stream) {
  return matmul(true, dY, dy_elem, M, w, dX, dx_elem, flags, stream);
}

nf4_status nf4_poll_device_status_site(void* stream, int32_t* site) {
  if (site) *site = 0;
  DeviceInfo* d = nullptr;
  if (nf4_status s = current_device(&d)) return s;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaError_t e = cudaStreamSynchronize(st); e != cudaSuccess) return launched(e);
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

nf4_status nf4_codebook(float* out16) { return nf4_codebook_of(NF4_DTYPE_NF4, out16); }

nf4_status nf4_codebook_of(int32_t dtype, float* out16) {
  if (!out16) return NF4_ERR_NULL;
  if (!is_4bit(dtype)) return NF4_ERR_SHAPE;
  const uint32_t* lv = dtype == NF4_DTYPE_FP4 ? nf4::kFp4LevelBits : nf4::kLevelBits;
  for (int i = 0; i < 16; ++i) out16[i] = nf4::bits_to_float(lv[i]);
  return NF4_OK;
}

nf4_status nf4_set_mma_wait_limit(int64_t cycles) {
  g_mma_wait_limit.store(cycles > 0 ? cycles : kDefaultWaitLimit, std::memory_order_relaxed);
  return NF4_OK;
}

const char* nf4_last_cuda_error(void) {
  return t_last_cuda_error == cudaSuccess ? "no error" : cudaGetErrorString(t_last_cuda_error);
}

const char* nf4_status_string(nf4_status status) {
  switch (status) {
    case NF4_OK: return "ok";
    case NF4_ERR_NULL: return "a required pointer is NULL (or a pointer the data type leaves unused is not)";
    case NF4_ERR_SHAPE: return "unsupported or negative shape, data type, element type or flag";
    case NF4_ERR_ALIGN: return "a pointer is not 16-byte aligned";
    case NF4_ERR_BLOCKSIZE: return "blocksize must be 64, dq_group 256 (4-bit) or 0 (int8)";
    case NF4_ERR_DEVICE: return "no current CUDA device, or it is not sm_103";
    case NF4_ERR_LAUNCH: return "the CUDA runtime rejected a launch or the stream holds an error";
    case NF4_ERR_DEVICE_TIMEOUT: return "a kernel's bounded wait ran out";
  }
  return "unknown status";
}

}  // extern "C"
