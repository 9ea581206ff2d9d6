// maskllm_api.cu -- the C ABI declared in include/maskllm.h: argument
// validation on the host, then one kernel launch on the caller's stream.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <atomic>

#include "internal.h"
#include "maskllm.h"

namespace maskllm {

namespace {

constexpr int kMaxDevices = 64;
std::atomic<int> g_num_sms[kMaxDevices];

thread_local char t_last_cuda_error[256] = "";

maskllm_status cuda_fail(cudaError_t e) {
  const char* msg = cudaGetErrorString(e);
  strncpy(t_last_cuda_error, msg ? msg : "unknown CUDA error", sizeof(t_last_cuda_error) - 1);
  t_last_cuda_error[sizeof(t_last_cuda_error) - 1] = '\0';
  return MASKLLM_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Span {
  const void* p;
  uint64_t bytes;
};

bool overlaps(Span a, Span b) {
  if (a.p == nullptr || b.p == nullptr || a.bytes == 0 || b.bytes == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
  return a0 < b0 + b.bytes && b0 < a0 + a.bytes;
}

// Outputs must not overlap inputs nor each other.
maskllm_status check_alias(const Span* in, int n_in, const Span* out, int n_out) {
  for (int o = 0; o < n_out; ++o) {
    for (int i = 0; i < n_in; ++i)
      if (overlaps(out[o], in[i])) return MASKLLM_ERR_ALIAS;
    for (int o2 = o + 1; o2 < n_out; ++o2)
      if (overlaps(out[o], out[o2])) return MASKLLM_ERR_ALIAS;
  }
  return MASKLLM_OK;
}

maskllm_status check_shape(int64_t rows, int64_t cols) {
  if (rows < 1 || cols < 32 || cols % 32 != 0) return MASKLLM_ERR_SHAPE;
  if (rows > (int64_t(1) << 46) / cols) return MASKLLM_ERR_SHAPE;
  return MASKLLM_OK;
}

maskllm_status check_ptrs(const void* const* ptrs, int n) {
  for (int i = 0; i < n; ++i)
    if (ptrs[i] == nullptr) return MASKLLM_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i)
    if (!aligned16(ptrs[i])) return MASKLLM_ERR_ALIGNMENT;
  return MASKLLM_OK;
}

maskllm_status check_optional(const void* p) {
  return (p == nullptr || aligned16(p)) ? MASKLLM_OK : MASKLLM_ERR_ALIGNMENT;
}

maskllm_status check_temperature(float tau, float kappa) {
  if (!isfinite(tau) || !(tau > 0.0f) || !isfinite(kappa)) return MASKLLM_ERR_INVALID_ARG;
  // 1/tau must be a finite fp32 number
  if (!isfinite(static_cast<float>(1.0 / static_cast<double>(tau)))) return MASKLLM_ERR_INVALID_ARG;
  return MASKLLM_OK;
}

#define MK_TRY(expr)                      \
  do {                                    \
    const maskllm_status st_ = (expr);    \
    if (st_ != MASKLLM_OK) return st_;    \
  } while (0)

maskllm_status get_device(Device* d) {
  const cudaError_t e = current_device(d);
  return e == cudaSuccess ? MASKLLM_OK : cuda_fail(e);
}

maskllm_status finish(cudaError_t e) { return e == cudaSuccess ? MASKLLM_OK : cuda_fail(e); }

}  // namespace

cudaError_t current_device(Device* d) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  d->ordinal = dev;
  int sms = (dev >= 0 && dev < kMaxDevices) ? g_num_sms[dev].load(std::memory_order_relaxed) : 0;
  if (sms <= 0) {
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxDevices) g_num_sms[dev].store(sms, std::memory_order_relaxed);
  }
  d->num_sms = sms;
  return cudaSuccess;
}

}  // namespace maskllm

using maskllm::Span;

extern "C" {

maskllm_status maskllm_prior_init(const uint16_t* W, int64_t rows, int64_t cols, float scale,
                                  float* logits_out, maskllm_stream_t stream) {
  const void* ptrs[] = {W, logits_out};
  MK_TRY(maskllm::check_ptrs(ptrs, 2));
  MK_TRY(maskllm::check_shape(rows, cols));
  if (!isfinite(scale)) return MASKLLM_ERR_INVALID_ARG;
  const uint64_t n = static_cast<uint64_t>(rows) * static_cast<uint64_t>(cols);
  const Span in[] = {{W, 2 * n}};
  const Span out[] = {{logits_out, 6 * n}};
  MK_TRY(maskllm::check_alias(in, 1, out, 1));
  maskllm::Device d;
  MK_TRY(maskllm::get_device(&d));
  return maskllm::finish(
      maskllm::launch_prior_init(d, W, rows, cols, scale, logits_out, stream));
}

maskllm_status maskllm_forward(const uint16_t* W, const float* logits, int64_t rows,
                               int64_t cols, float tau, float kappa, maskllm_rng rng,
                               uint16_t* W_out, float* row_sq_out, float* probs_out,
                               maskllm_stream_t stream) {
  const void* ptrs[] = {W, logits, W_out};
  MK_TRY(maskllm::check_ptrs(ptrs, 3));
  MK_TRY(maskllm::check_optional(row_sq_out));
  MK_TRY(maskllm::check_optional(probs_out));
  MK_TRY(maskllm::check_shape(rows, cols));
  MK_TRY(maskllm::check_temperature(tau, kappa));
  const uint64_t n = static_cast<uint64_t>(rows) * static_cast<uint64_t>(cols);
  const Span in[] = {{W, 2 * n}, {logits, 6 * n}};
  const Span out[] = {{W_out, 2 * n},
                      {row_sq_out, 4 * static_cast<uint64_t>(rows)},
                      {probs_out, 6 * n}};
  MK_TRY(maskllm::check_alias(in, 2, out, 3));
  maskllm::Device d;
  MK_TRY(maskllm::get_device(&d));
  return maskllm::finish(maskllm::launch_forward(d, W, logits, rows, cols, tau, kappa,
                                                 {rng.seed, rng.step, rng.tensor_id}, W_out,
                                                 row_sq_out, probs_out, stream));
}

maskllm_status maskllm_backward(const uint16_t* W, const float* logits,
                                const uint16_t* grad_W_out, int64_t rows, int64_t cols,
                                float tau, float kappa, maskllm_rng rng, float reg_coeff,
                                float* dlogits_out, maskllm_stream_t stream) {
  const void* ptrs[] = {W, logits, grad_W_out, dlogits_out};
  MK_TRY(maskllm::check_ptrs(ptrs, 4));
  MK_TRY(maskllm::check_shape(rows, cols));
  MK_TRY(maskllm::check_temperature(tau, kappa));
  if (!isfinite(reg_coeff)) return MASKLLM_ERR_INVALID_ARG;
  const uint64_t n = static_cast<uint64_t>(rows) * static_cast<uint64_t>(cols);
  const Span in[] = {{W, 2 * n}, {logits, 6 * n}, {grad_W_out, 2 * n}};
  const Span out[] = {{dlogits_out, 6 * n}};
  MK_TRY(maskllm::check_alias(in, 3, out, 1));
  maskllm::Device d;
  MK_TRY(maskllm::get_device(&d));
  return maskllm::finish(maskllm::launch_backward(d, W, logits, grad_W_out, rows, cols, tau,
                                                  kappa, {rng.seed, rng.step, rng.tensor_id},
                                                  reg_coeff, dlogits_out, stream));
}

maskllm_status maskllm_hard_compress(const uint16_t* W, const float* logits, int64_t rows,
                                     int64_t cols, uint16_t* values_out, uint32_t* meta_out,
                                     uint8_t* idx_out, maskllm_stream_t stream) {
  const void* ptrs[] = {W, logits, values_out, meta_out};
  MK_TRY(maskllm::check_ptrs(ptrs, 4));
  MK_TRY(maskllm::check_optional(idx_out));
  MK_TRY(maskllm::check_shape(rows, cols));
  const uint64_t n = static_cast<uint64_t>(rows) * static_cast<uint64_t>(cols);
  const Span in[] = {{W, 2 * n}, {logits, 6 * n}};
  const Span out[] = {{values_out, n}, {meta_out, n / 8}, {idx_out, n / 4}};
  MK_TRY(maskllm::check_alias(in, 2, out, 3));
  maskllm::Device d;
  MK_TRY(maskllm::get_device(&d));
  return maskllm::finish(maskllm::launch_hard_compress(d, W, logits, rows, cols, values_out,
                                                       meta_out, idx_out, stream));
}

maskllm_status maskllm_decompress(const uint16_t* values, const uint32_t* meta, int64_t rows,
                                  int64_t cols, uint16_t* W_out, maskllm_stream_t stream) {
  const void* ptrs[] = {values, meta, W_out};
  MK_TRY(maskllm::check_ptrs(ptrs, 3));
  MK_TRY(maskllm::check_shape(rows, cols));
  const uint64_t n = static_cast<uint64_t>(rows) * static_cast<uint64_t>(cols);
  const Span in[] = {{values, n}, {meta, n / 8}};
  const Span out[] = {{W_out, 2 * n}};
  MK_TRY(maskllm::check_alias(in, 2, out, 1));
  maskllm::Device d;
  MK_TRY(maskllm::get_device(&d));
  return maskllm::finish(maskllm::launch_decompress(d, values, meta, rows, cols, W_out, stream));
}

maskllm_status maskllm_noise_words(maskllm_rng rng, int64_t group_begin, int64_t n,
                                   uint32_t* out4, maskllm_stream_t stream) {
  const void* ptrs[] = {out4};
  MK_TRY(maskllm::check_ptrs(ptrs, 1));
  if (group_begin < 0 || n < 1 || n > (int64_t(1) << 40) ||
      group_begin > (int64_t(1) << 62) - n)
    return MASKLLM_ERR_INVALID_ARG;
  maskllm::Device d;
  MK_TRY(maskllm::get_device(&d));
  return maskllm::finish(maskllm::launch_noise_words(
      d, {rng.seed, rng.step, rng.tensor_id}, group_begin, n, out4, stream));
}

maskllm_status maskllm_device_status(maskllm_stream_t stream) {
  uint32_t word = 0;
  const cudaError_t e = maskllm::read_and_clear_error_word(stream, &word);
  if (e != cudaSuccess) return maskllm::cuda_fail(e);
  return word != 0 ? MASKLLM_ERR_TIMEOUT : MASKLLM_OK;
}

const char* maskllm_status_string(maskllm_status status) {
  switch (status) {
    case MASKLLM_OK: return "MASKLLM_OK";
    case MASKLLM_ERR_INVALID_ARG: return "MASKLLM_ERR_INVALID_ARG";
    case MASKLLM_ERR_SHAPE: return "MASKLLM_ERR_SHAPE";
    case MASKLLM_ERR_ALIGNMENT: return "MASKLLM_ERR_ALIGNMENT";
    case MASKLLM_ERR_ALIAS: return "MASKLLM_ERR_ALIAS";
    case MASKLLM_ERR_CUDA: return "MASKLLM_ERR_CUDA";
    case MASKLLM_ERR_TIMEOUT: return "MASKLLM_ERR_TIMEOUT";
  }
  return "MASKLLM_UNKNOWN_STATUS";
}

const char* maskllm_last_cuda_error(void) { return maskllm::t_last_cuda_error; }

}  // extern "C"
