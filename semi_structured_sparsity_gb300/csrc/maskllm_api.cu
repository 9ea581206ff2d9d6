// maskllm_api.cu -- the C ABI declared in include/maskllm.h: argument
// validation on the host, then kernel launches on the caller's stream.
//
// Kernels: the pipelined streaming kernels (kernels_stream.cu) serve the
// prior, forward, backward, hard-compress and diagnostics calls; the others
// live in kernels_pack.cu, kernels_perm.cu and kernels_spmm.cu.
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

// Inputs and outputs of one call (all matrices of a batch together; at most
// 4 inputs (the backward with diagnostics) and 5 outputs (the forward with
// diagnostics) per matrix).
struct Spans {
  static constexpr int kCap = 8 * kMaxBatch;
  Span in[kCap];
  Span out[kCap];
  int n_in = 0, n_out = 0;
  bool full = false;
  void input(const void* p, uint64_t b) {
    if (n_in < kCap) in[n_in++] = {p, b};
    else full = true;
  }
  void output(const void* p, uint64_t b) {
    if (n_out < kCap) out[n_out++] = {p, b};
    else full = true;
  }
  // Outputs must not overlap inputs nor each other.
  maskllm_status check() const {
    if (full) return MASKLLM_ERR_INVALID_ARG;
    for (int o = 0; o < n_out; ++o) {
      for (int i = 0; i < n_in; ++i)
        if (overlaps(out[o], in[i])) return MASKLLM_ERR_ALIAS;
      for (int o2 = o + 1; o2 < n_out; ++o2)
        if (overlaps(out[o], out[o2])) return MASKLLM_ERR_ALIAS;
    }
    return MASKLLM_OK;
  }
};

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

#define MK_TRY(expr)                   \
  do {                                 \
    const maskllm_status st_ = (expr); \
    if (st_ != MASKLLM_OK) return st_; \
  } while (0)

uint64_t weights(const maskllm_matrix& m) {
  return static_cast<uint64_t>(m.rows) * static_cast<uint64_t>(m.cols);
}

// Per-operation validation of one matrix; appends its spans.
maskllm_status check_prior(const maskllm_matrix& m, Spans& sp) {
  const void* ptrs[] = {m.W, m.logits_out};
  MK_TRY(check_ptrs(ptrs, 2));
  MK_TRY(check_shape(m.rows, m.cols));
  const uint64_t n = weights(m);
  sp.input(m.W, 2 * n);
  sp.output(m.logits_out, 6 * n);
  return MASKLLM_OK;
}

maskllm_status check_forward(const maskllm_matrix& m, Spans& sp) {
  const void* ptrs[] = {m.W, m.logits, m.W_out};
  MK_TRY(check_ptrs(ptrs, 3));
  MK_TRY(check_optional(m.row_sq_out));
  MK_TRY(check_optional(m.probs_out));
  MK_TRY(check_shape(m.rows, m.cols));
  const uint64_t n = weights(m);
  sp.input(m.W, 2 * n);
  sp.input(m.logits, 6 * n);
  sp.output(m.W_out, 2 * n);
  sp.output(m.row_sq_out, 4 * static_cast<uint64_t>(m.rows));
  sp.output(m.probs_out, 6 * n);
  return MASKLLM_OK;
}

maskllm_status check_backward(const maskllm_matrix& m, Spans& sp) {
  const void* ptrs[] = {m.W, m.logits, m.grad_W_out, m.dlogits_out};
  MK_TRY(check_ptrs(ptrs, 4));
  MK_TRY(check_shape(m.rows, m.cols));
  const uint64_t n = weights(m);
  sp.input(m.W, 2 * n);
  sp.input(m.logits, 6 * n);
  sp.input(m.grad_W_out, 2 * n);
  sp.output(m.dlogits_out, 6 * n);
  return MASKLLM_OK;
}

maskllm_status check_compress(const maskllm_matrix& m, Spans& sp) {
  const void* ptrs[] = {m.W, m.logits, m.values_out, m.meta_out};
  MK_TRY(check_ptrs(ptrs, 4));
  MK_TRY(check_optional(m.idx_out));
  MK_TRY(check_shape(m.rows, m.cols));
  const uint64_t n = weights(m);
  sp.input(m.W, 2 * n);
  sp.input(m.logits, 6 * n);
  sp.output(m.values_out, n);
  sp.output(m.meta_out, n / 8);
  sp.output(m.idx_out, n / 4);
  return MASKLLM_OK;
}

maskllm_status check_prior_from_mask(const maskllm_matrix& m, Spans& sp) {
  const void* ptrs[] = {m.meta, m.logits_out};
  MK_TRY(check_ptrs(ptrs, 2));
  MK_TRY(check_shape(m.rows, m.cols));
  const uint64_t n = weights(m);
  sp.input(m.meta, n / 8);
  sp.output(m.logits_out, 6 * n);
  return MASKLLM_OK;
}

// The diagnostics' rules (maskllm_mask_stats): optional outputs, the L1
// distance needs the previous draws, rows no longer than 2^24 weights.
maskllm_status check_diagnostics(const maskllm_matrix& m, Spans& sp) {
  MK_TRY(check_optional(m.prev_idx));
  MK_TRY(check_optional(m.idx_out));
  MK_TRY(check_optional(m.l1_row_out));
  MK_TRY(check_optional(m.maxprob_row_out));
  if (m.l1_row_out != nullptr && m.prev_idx == nullptr) return MASKLLM_ERR_INVALID_ARG;
  MK_TRY(check_shape(m.rows, m.cols));
  if (m.cols > (int64_t(1) << 24)) return MASKLLM_ERR_SHAPE;
  const uint64_t n = weights(m), r4 = 4 * static_cast<uint64_t>(m.rows);
  sp.input(m.prev_idx, n / 4);
  sp.output(m.idx_out, n / 4);
  sp.output(m.l1_row_out, r4);
  sp.output(m.maxprob_row_out, r4);
  return MASKLLM_OK;
}

maskllm_status check_mask_stats(const maskllm_matrix& m, Spans& sp) {
  const void* ptrs[] = {m.logits};
  MK_TRY(check_ptrs(ptrs, 1));
  MK_TRY(check_diagnostics(m, sp));
  sp.input(m.logits, 6 * weights(m));
  return MASKLLM_OK;
}

maskllm_status check_forward_stats(const maskllm_matrix& m, Spans& sp) {
  const void* ptrs[] = {m.W, m.logits, m.W_out};
  MK_TRY(check_ptrs(ptrs, 3));
  MK_TRY(check_optional(m.row_sq_out));
  MK_TRY(check_diagnostics(m, sp));
  const uint64_t n = weights(m);
  sp.input(m.W, 2 * n);
  sp.input(m.logits, 6 * n);
  sp.output(m.W_out, 2 * n);
  sp.output(m.row_sq_out, 4 * static_cast<uint64_t>(m.rows));
  return MASKLLM_OK;
}

maskllm_status check_backward_stats(const maskllm_matrix& m, Spans& sp) {
  MK_TRY(check_backward(m, sp));
  return check_diagnostics(m, sp);
}

maskllm_status finish(cudaError_t e) { return e == cudaSuccess ? MASKLLM_OK : cuda_fail(e); }

enum class Op {
  kPrior,
  kForward,
  kBackward,
  kCompress,
  kPriorFromMask,
  kMaskStats,
  kForwardStats,
  kBackwardStats
};

struct Call {
  Op op;
  float tau = 1.0f, kappa = 0.0f, reg = 0.0f, scale = 1.0f, high = 0.0f, low = 0.0f;
  uint64_t seed = 0;
  uint32_t step = 0;
};

StreamMatrix to_stream(const maskllm_matrix& m, Op op) {
  StreamMatrix s{};
  s.W = m.W;
  s.L = m.logits;
  s.G = m.grad_W_out;
  s.rows = m.rows;
  s.cols = m.cols;
  s.tensor_id = m.tensor_id;
  switch (op) {
    case Op::kPrior: s.out0 = m.logits_out; break;
    case Op::kForward:
      s.out0 = m.W_out;
      s.out1 = m.row_sq_out;
      s.out2 = m.probs_out;
      break;
    case Op::kBackward: s.out0 = m.dlogits_out; break;
    case Op::kCompress:
      s.out0 = m.values_out;
      s.out1 = m.meta_out;
      s.out2 = m.idx_out;
      break;
    case Op::kPriorFromMask:
      s.W = m.meta;
      s.L = nullptr;
      s.G = nullptr;
      s.out0 = m.logits_out;
      break;
    case Op::kMaskStats:
      s.W = nullptr;
      s.G = m.prev_idx;
      s.out0 = m.idx_out;
      s.out1 = m.l1_row_out;
      s.out2 = m.maxprob_row_out;
      break;
    case Op::kForwardStats:
      s.G = m.prev_idx;
      s.out0 = m.W_out;
      s.out1 = m.row_sq_out;
      s.out2 = m.idx_out;
      s.out3 = m.l1_row_out;
      s.out4 = m.maxprob_row_out;
      break;
    case Op::kBackwardStats:
      s.P = m.prev_idx;
      s.out0 = m.dlogits_out;
      s.out1 = m.idx_out;
      s.out2 = m.l1_row_out;
      s.out3 = m.maxprob_row_out;
      break;
  }
  return s;
}

// The validation of one matrix for the call's operation (appends its spans).
maskllm_status check_matrix(Op op, const maskllm_matrix& m, Spans& sp) {
  switch (op) {
    case Op::kPrior: return check_prior(m, sp);
    case Op::kForward: return check_forward(m, sp);
    case Op::kBackward: return check_backward(m, sp);
    case Op::kCompress: return check_compress(m, sp);
    case Op::kPriorFromMask: return check_prior_from_mask(m, sp);
    case Op::kMaskStats: return check_mask_stats(m, sp);
    case Op::kForwardStats: return check_forward_stats(m, sp);
    case Op::kBackwardStats: return check_backward_stats(m, sp);
  }
  return MASKLLM_ERR_INVALID_ARG;
}

maskllm_status run(const Call& c, const maskllm_matrix* mats, int32_t n, cudaStream_t s) {
  if (mats == nullptr || n < 1) return MASKLLM_ERR_INVALID_ARG;
  if (c.op != Op::kPrior && c.op != Op::kCompress && c.op != Op::kPriorFromMask)
    MK_TRY(check_temperature(c.tau, c.kappa));
  if (!isfinite(c.reg) || !isfinite(c.scale) || !isfinite(c.high) || !isfinite(c.low))
    return MASKLLM_ERR_INVALID_ARG;
  // validate everything before launching anything
  for (int32_t b = 0; b < n; b += kMaxBatch) {
    const int32_t nb = n - b < kMaxBatch ? n - b : kMaxBatch;
    Spans sp;
    for (int32_t i = 0; i < nb; ++i) MK_TRY(check_matrix(c.op, mats[b + i], sp));
    MK_TRY(sp.check());
  }
  if (n > kMaxBatch) {
    // outputs of one launch must not overlap inputs or outputs of another
    for (int32_t i = 0; i < n; ++i) {
      Spans one;
      check_matrix(c.op, mats[i], one);
      for (int32_t j = 0; j < n; ++j) {
        if (j == i) continue;
        Spans other;
        check_matrix(c.op, mats[j], other);
        for (int o = 0; o < one.n_out; ++o) {
          for (int k = 0; k < other.n_in; ++k)
            if (overlaps(one.out[o], other.in[k])) return MASKLLM_ERR_ALIAS;
          for (int k = 0; k < other.n_out; ++k)
            if (overlaps(one.out[o], other.out[k])) return MASKLLM_ERR_ALIAS;
        }
      }
    }
  }
  Device d;
  cudaError_t e = current_device(&d);
  if (e != cudaSuccess) return cuda_fail(e);
  for (int32_t b = 0; b < n; b += kMaxBatch) {
    const int32_t nb = n - b < kMaxBatch ? n - b : kMaxBatch;
    StreamMatrix sm[kMaxBatch];
    bool probs = false;
    for (int32_t i = 0; i < nb; ++i) {
      sm[i] = to_stream(mats[b + i], c.op);
      probs = probs || (c.op == Op::kForward && mats[b + i].probs_out != nullptr);
    }
    const RngArgs rng{c.seed, c.step, 0};
    switch (c.op) {
      case Op::kPrior: e = stream_prior_init(d, sm, nb, c.scale, s); break;
      case Op::kForward: e = stream_forward(d, sm, nb, c.tau, c.kappa, rng, probs, s); break;
      case Op::kBackward: e = stream_backward(d, sm, nb, c.tau, c.kappa, rng, c.reg, s); break;
      case Op::kCompress: e = stream_hard_compress(d, sm, nb, s); break;
      case Op::kPriorFromMask: e = launch_prior_from_mask(d, sm, nb, c.high, c.low, s); break;
      case Op::kMaskStats: e = stream_mask_stats(d, sm, nb, c.tau, c.kappa, rng, s); break;
      case Op::kForwardStats: e = stream_forward_stats(d, sm, nb, c.tau, c.kappa, rng, s); break;
      case Op::kBackwardStats:
        e = stream_backward_stats(d, sm, nb, c.tau, c.kappa, rng, c.reg, s);
        break;
    }
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return MASKLLM_OK;
}

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

using maskllm::Call;
using maskllm::Op;

extern "C" {

maskllm_status maskllm_prior_init(const uint16_t* W, int64_t rows, int64_t cols, float scale,
                                  float* logits_out, maskllm_stream_t stream) {
  maskllm_matrix m{};
  m.W = W;
  m.rows = rows;
  m.cols = cols;
  m.logits_out = logits_out;
  Call c{Op::kPrior};
  c.scale = scale;
  return maskllm::run(c, &m, 1, stream);
}

maskllm_status maskllm_forward(const uint16_t* W, const float* logits, int64_t rows,
                               int64_t cols, float tau, float kappa, maskllm_rng rng,
                               uint16_t* W_out, float* row_sq_out, float* probs_out,
                               maskllm_stream_t stream) {
  maskllm_matrix m{};
  m.W = W;
  m.logits = logits;
  m.rows = rows;
  m.cols = cols;
  m.tensor_id = rng.tensor_id;
  m.W_out = W_out;
  m.row_sq_out = row_sq_out;
  m.probs_out = probs_out;
  Call c{Op::kForward};
  c.tau = tau;
  c.kappa = kappa;
  c.seed = rng.seed;
  c.step = rng.step;
  return maskllm::run(c, &m, 1, stream);
}

maskllm_status maskllm_backward(const uint16_t* W, const float* logits,
                                const uint16_t* grad_W_out, int64_t rows, int64_t cols,
                                float tau, float kappa, maskllm_rng rng, float reg_coeff,
                                float* dlogits_out, maskllm_stream_t stream) {
  maskllm_matrix m{};
  m.W = W;
  m.logits = logits;
  m.grad_W_out = grad_W_out;
  m.rows = rows;
  m.cols = cols;
  m.tensor_id = rng.tensor_id;
  m.dlogits_out = dlogits_out;
  Call c{Op::kBackward};
  c.tau = tau;
  c.kappa = kappa;
  c.seed = rng.seed;
  c.step = rng.step;
  c.reg = reg_coeff;
  return maskllm::run(c, &m, 1, stream);
}

maskllm_status maskllm_hard_compress(const uint16_t* W, const float* logits, int64_t rows,
                                     int64_t cols, uint16_t* values_out, uint32_t* meta_out,
                                     uint8_t* idx_out, maskllm_stream_t stream) {
  maskllm_matrix m{};
  m.W = W;
  m.logits = logits;
  m.rows = rows;
  m.cols = cols;
  m.values_out = values_out;
  m.meta_out = meta_out;
  m.idx_out = idx_out;
  return maskllm::run(Call{Op::kCompress}, &m, 1, stream);
}

maskllm_status maskllm_prior_init_batched(const maskllm_matrix* mats, int32_t n, float scale,
                                          maskllm_stream_t stream) {
  Call c{Op::kPrior};
  c.scale = scale;
  return maskllm::run(c, mats, n, stream);
}

maskllm_status maskllm_forward_batched(const maskllm_matrix* mats, int32_t n, float tau,
                                       float kappa, uint64_t seed, uint32_t step,
                                       maskllm_stream_t stream) {
  Call c{Op::kForward};
  c.tau = tau;
  c.kappa = kappa;
  c.seed = seed;
  c.step = step;
  return maskllm::run(c, mats, n, stream);
}

maskllm_status maskllm_backward_batched(const maskllm_matrix* mats, int32_t n, float tau,
                                        float kappa, uint64_t seed, uint32_t step,
                                        float reg_coeff, maskllm_stream_t stream) {
  Call c{Op::kBackward};
  c.tau = tau;
  c.kappa = kappa;
  c.seed = seed;
  c.step = step;
  c.reg = reg_coeff;
  return maskllm::run(c, mats, n, stream);
}

maskllm_status maskllm_hard_compress_batched(const maskllm_matrix* mats, int32_t n,
                                             maskllm_stream_t stream) {
  return maskllm::run(Call{Op::kCompress}, mats, n, stream);
}

maskllm_status maskllm_decompress(const uint16_t* values, const uint32_t* meta, int64_t rows,
                                  int64_t cols, uint16_t* W_out, maskllm_stream_t stream) {
  const void* ptrs[] = {values, meta, W_out};
  MK_TRY(maskllm::check_ptrs(ptrs, 3));
  MK_TRY(maskllm::check_shape(rows, cols));
  const uint64_t n = static_cast<uint64_t>(rows) * static_cast<uint64_t>(cols);
  maskllm::Spans sp;
  sp.input(values, n);
  sp.input(meta, n / 8);
  sp.output(W_out, 2 * n);
  MK_TRY(sp.check());
  maskllm::Device d;
  cudaError_t e = maskllm::current_device(&d);
  if (e != cudaSuccess) return maskllm::cuda_fail(e);
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
  cudaError_t e = maskllm::current_device(&d);
  if (e != cudaSuccess) return maskllm::cuda_fail(e);
  return maskllm::finish(maskllm::launch_noise_words(
      d, {rng.seed, rng.step, rng.tensor_id}, group_begin, n, out4, stream));
}

maskllm_status maskllm_prior_from_mask(const uint32_t* meta, int64_t rows, int64_t cols,
                                       float high, float low, float* logits_out,
                                       maskllm_stream_t stream) {
  maskllm_matrix m{};
  m.meta = meta;
  m.rows = rows;
  m.cols = cols;
  m.logits_out = logits_out;
  Call c{Op::kPriorFromMask};
  c.high = high;
  c.low = low;
  return maskllm::run(c, &m, 1, stream);
}

maskllm_status maskllm_prior_from_mask_batched(const maskllm_matrix* mats, int32_t n, float high,
                                               float low, maskllm_stream_t stream) {
  Call c{Op::kPriorFromMask};
  c.high = high;
  c.low = low;
  return maskllm::run(c, mats, n, stream);
}

maskllm_status maskllm_mask_stats_batched(const maskllm_matrix* mats, int32_t n, float tau,
                                          float kappa, uint64_t seed, uint32_t step,
                                          maskllm_stream_t stream) {
  Call c{Op::kMaskStats};
  c.tau = tau;
  c.kappa = kappa;
  c.seed = seed;
  c.step = step;
  return maskllm::run(c, mats, n, stream);
}

maskllm_status maskllm_forward_stats_batched(const maskllm_matrix* mats, int32_t n, float tau,
                                             float kappa, uint64_t seed, uint32_t step,
                                             maskllm_stream_t stream) {
  Call c{Op::kForwardStats};
  c.tau = tau;
  c.kappa = kappa;
  c.seed = seed;
  c.step = step;
  return maskllm::run(c, mats, n, stream);
}

maskllm_status maskllm_backward_stats_batched(const maskllm_matrix* mats, int32_t n, float tau,
                                              float kappa, uint64_t seed, uint32_t step,
                                              float reg_coeff, maskllm_stream_t stream) {
  Call c{Op::kBackwardStats};
  c.tau = tau;
  c.kappa = kappa;
  c.seed = seed;
  c.step = step;
  c.reg = reg_coeff;
  return maskllm::run(c, mats, n, stream);
}

maskllm_status maskllm_backward_stats(const uint16_t* W, const float* logits,
                                      const uint16_t* grad_W_out, const uint8_t* prev_idx,
                                      int64_t rows, int64_t cols, float tau, float kappa,
                                      maskllm_rng rng, float reg_coeff, float* dlogits_out,
                                      uint8_t* idx_out, uint32_t* l1_row_out,
                                      float* maxprob_row_out, maskllm_stream_t stream) {
  maskllm_matrix m{};
  m.W = W;
  m.logits = logits;
  m.grad_W_out = grad_W_out;
  m.prev_idx = prev_idx;
  m.rows = rows;
  m.cols = cols;
  m.tensor_id = rng.tensor_id;
  m.dlogits_out = dlogits_out;
  m.idx_out = idx_out;
  m.l1_row_out = l1_row_out;
  m.maxprob_row_out = maxprob_row_out;
  return maskllm_backward_stats_batched(&m, 1, tau, kappa, rng.seed, rng.step, reg_coeff, stream);
}

maskllm_status maskllm_mask_stats(const float* logits, const uint8_t* prev_idx, int64_t rows,
                                  int64_t cols, float tau, float kappa, maskllm_rng rng,
                                  uint8_t* idx_out, uint32_t* l1_row_out,
                                  float* maxprob_row_out, maskllm_stream_t stream) {
  maskllm_matrix m{};
  m.logits = logits;
  m.prev_idx = prev_idx;
  m.rows = rows;
  m.cols = cols;
  m.tensor_id = rng.tensor_id;
  m.idx_out = idx_out;
  m.l1_row_out = l1_row_out;
  m.maxprob_row_out = maxprob_row_out;
  Call c{Op::kMaskStats};
  c.tau = tau;
  c.kappa = kappa;
  c.seed = rng.seed;
  c.step = rng.step;
  return maskllm::run(c, &m, 1, stream);
}

}  // extern "C"

namespace maskllm {
namespace {

maskllm_status check_perm_shape(int64_t rows, int64_t cols) {
  MK_TRY(check_shape(rows, cols));
  if (cols > kPermMaxCols || rows > kPermMaxRows) return MASKLLM_ERR_SHAPE;
  return MASKLLM_OK;
}

}  // namespace
}  // namespace maskllm

extern "C" {

maskllm_status maskllm_perm_shift(const uint16_t* W, int64_t rows, int64_t cols,
                                  int32_t* shift_out, maskllm_stream_t stream) {
  const void* ptrs[] = {W, shift_out};
  MK_TRY(maskllm::check_ptrs(ptrs, 2));
  MK_TRY(maskllm::check_perm_shape(rows, cols));
  maskllm::Spans sp;
  sp.input(W, 2 * static_cast<uint64_t>(rows) * cols);
  sp.output(shift_out, 4);
  MK_TRY(sp.check());
  maskllm::Device d;
  cudaError_t e = maskllm::current_device(&d);
  if (e != cudaSuccess) return maskllm::cuda_fail(e);
  return maskllm::finish(maskllm::perm_shift(d, W, rows, cols, shift_out, stream));
}

maskllm_status maskllm_perm_metric(const uint16_t* W, int64_t rows, int64_t cols,
                                   const int32_t* perm, const int32_t* shift,
                                   uint64_t* metric_out, maskllm_stream_t stream) {
  const void* ptrs[] = {W, perm, shift, metric_out};
  MK_TRY(maskllm::check_ptrs(ptrs, 4));
  MK_TRY(maskllm::check_perm_shape(rows, cols));
  maskllm::Spans sp;
  sp.input(W, 2 * static_cast<uint64_t>(rows) * cols);
  sp.input(perm, 4 * static_cast<uint64_t>(cols));
  sp.input(shift, 4);
  sp.output(metric_out, 8);
  MK_TRY(sp.check());
  maskllm::Device d;
  cudaError_t e = maskllm::current_device(&d);
  if (e != cudaSuccess) return maskllm::cuda_fail(e);
  return maskllm::finish(maskllm::perm_metric(d, W, rows, cols, perm, shift, metric_out, stream));
}

maskllm_status maskllm_permute_columns(const uint16_t* W, int64_t rows, int64_t cols,
                                       const int32_t* perm, uint16_t* W_out,
                                       maskllm_stream_t stream) {
  const void* ptrs[] = {W, perm, W_out};
  MK_TRY(maskllm::check_ptrs(ptrs, 3));
  MK_TRY(maskllm::check_perm_shape(rows, cols));
  const uint64_t n = static_cast<uint64_t>(rows) * cols;
  maskllm::Spans sp;
  sp.input(W, 2 * n);
  sp.input(perm, 4 * static_cast<uint64_t>(cols));
  sp.output(W_out, 2 * n);
  MK_TRY(sp.check());
  maskllm::Device d;
  cudaError_t e = maskllm::current_device(&d);
  if (e != cudaSuccess) return maskllm::cuda_fail(e);
  return maskllm::finish(maskllm::permute_columns(d, W, rows, cols, perm, W_out, stream));
}

int64_t maskllm_perm_workspace_bytes(int64_t rows, int64_t cols) {
  if (maskllm::check_perm_shape(rows, cols) != MASKLLM_OK) return 0;
  return maskllm::perm_workspace_bytes(rows, cols);
}

maskllm_status maskllm_perm_swap_gains(const uint16_t* W, int64_t rows, int64_t cols,
                                       const int32_t* perm, void* workspace,
                                       int64_t workspace_bytes, int64_t* gains_out,
                                       int32_t* info_out, int32_t* shift_out,
                                       maskllm_stream_t stream) {
  const void* ptrs[] = {W, perm, workspace, gains_out, info_out};
  MK_TRY(maskllm::check_ptrs(ptrs, 5));
  MK_TRY(maskllm::check_optional(shift_out));
  MK_TRY(maskllm::check_perm_shape(rows, cols));
  const int64_t need = maskllm::perm_workspace_bytes(rows, cols);
  if (workspace_bytes < need) return MASKLLM_ERR_INVALID_ARG;
  maskllm::Spans sp;
  sp.input(W, 2 * static_cast<uint64_t>(rows) * cols);
  sp.input(perm, 4 * static_cast<uint64_t>(cols));
  sp.output(workspace, static_cast<uint64_t>(need));
  sp.output(gains_out, 8 * static_cast<uint64_t>(cols) * cols);
  sp.output(info_out, 4);
  sp.output(shift_out, 4);
  MK_TRY(sp.check());
  maskllm::Device d;
  cudaError_t e = maskllm::current_device(&d);
  if (e != cudaSuccess) return maskllm::cuda_fail(e);
  return maskllm::finish(maskllm::perm_swap_gains(d, W, rows, cols, perm, workspace, gains_out,
                                                  info_out, shift_out, stream));
}

maskllm_status maskllm_perm_search(const uint16_t* W, int64_t rows, int64_t cols, int32_t* perm,
                                   int32_t max_swaps, void* workspace, int64_t workspace_bytes,
                                   int32_t* swaps_out, int64_t* gains_out,
                                   int32_t* n_swaps_out, int32_t* shift_out,
                                   maskllm_stream_t stream) {
  const void* ptrs[] = {W, perm, workspace, n_swaps_out};
  MK_TRY(maskllm::check_ptrs(ptrs, 4));
  MK_TRY(maskllm::check_optional(swaps_out));
  MK_TRY(maskllm::check_optional(gains_out));
  MK_TRY(maskllm::check_optional(shift_out));
  MK_TRY(maskllm::check_perm_shape(rows, cols));
  if (max_swaps < 0) return MASKLLM_ERR_INVALID_ARG;
  const int64_t need = maskllm::perm_workspace_bytes(rows, cols);
  if (workspace_bytes < need) return MASKLLM_ERR_INVALID_ARG;
  maskllm::Spans sp;
  sp.input(W, 2 * static_cast<uint64_t>(rows) * cols);
  sp.output(perm, 4 * static_cast<uint64_t>(cols));
  sp.output(workspace, static_cast<uint64_t>(need));
  sp.output(swaps_out, 8 * static_cast<uint64_t>(max_swaps));
  sp.output(gains_out, 8 * static_cast<uint64_t>(max_swaps));
  sp.output(n_swaps_out, 4);
  sp.output(shift_out, 4);
  MK_TRY(sp.check());
  maskllm::Device d;
  cudaError_t e = maskllm::current_device(&d);
  if (e != cudaSuccess) return maskllm::cuda_fail(e);
  return maskllm::finish(maskllm::perm_search(d, W, rows, cols, perm, max_swaps, workspace,
                                              swaps_out, gains_out, n_swaps_out, shift_out,
                                              stream));
}

maskllm_status maskllm_forward_stats(const uint16_t* W, const float* logits,
                                     const uint8_t* prev_idx, int64_t rows, int64_t cols,
                                     float tau, float kappa, maskllm_rng rng, uint16_t* W_out,
                                     float* row_sq_out, uint8_t* idx_out, uint32_t* l1_row_out,
                                     float* maxprob_row_out, maskllm_stream_t stream) {
  maskllm_matrix m{};
  m.W = W;
  m.logits = logits;
  m.prev_idx = prev_idx;
  m.rows = rows;
  m.cols = cols;
  m.tensor_id = rng.tensor_id;
  m.W_out = W_out;
  m.row_sq_out = row_sq_out;
  m.idx_out = idx_out;
  m.l1_row_out = l1_row_out;
  m.maxprob_row_out = maxprob_row_out;
  Call c{Op::kForwardStats};
  c.tau = tau;
  c.kappa = kappa;
  c.seed = rng.seed;
  c.step = rng.step;
  return maskllm::run(c, &m, 1, stream);
}

maskllm_status maskllm_set_wait_timeout(uint64_t nanoseconds) {
  maskllm::stream_set_wait_ns(nanoseconds);
  return MASKLLM_OK;
}

maskllm_status maskllm_test_withhold_loads(int32_t enable) {
  maskllm::stream_set_withhold_loads(enable != 0);
  return MASKLLM_OK;
}

maskllm_status maskllm_test_spmm_tile_n(int32_t n) {
  if (n != 0 && (n < 128 || n > 256 || n % 32 != 0)) return MASKLLM_ERR_INVALID_ARG;
  maskllm::spmm_force_tile_width(n);
  return MASKLLM_OK;
}

maskllm_status maskllm_device_status(maskllm_stream_t stream) {
  uint32_t b = 0, c = 0, g = 0;
  cudaError_t e = maskllm::read_and_clear_stream_error(stream, &b);
  if (e == cudaSuccess) e = maskllm::read_and_clear_perm_error(stream, &c);
  if (e == cudaSuccess) e = maskllm::read_and_clear_spmm_error(stream, &g);
  if (e != cudaSuccess) return maskllm::cuda_fail(e);
  if ((b | g) != 0) return MASKLLM_ERR_TIMEOUT;
  return c != 0 ? MASKLLM_ERR_INVALID_ARG : MASKLLM_OK;
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

extern "C" maskllm_status maskllm_spmm(const uint16_t* values, const uint32_t* meta, int64_t M,
                                       int64_t K, const uint16_t* B, int64_t N, float* C,
                                       maskllm_stream_t stream) {
  const void* ptrs[] = {values, meta, B, C};
  MK_TRY(maskllm::check_ptrs(ptrs, 4));
  if (M < 1 || N < 1 || K < 32 || K % 32 != 0) return MASKLLM_ERR_SHAPE;
  const int64_t lim = (int64_t(1) << 31) - 1;
  // the grid holds one CTA pair per 256 rows of C in x and 256 columns in y
  if (M > lim || N > lim || K > lim || (N + 255) / 256 > 65535) return MASKLLM_ERR_SHAPE;
  maskllm::Spans sp;
  sp.input(values, static_cast<uint64_t>(M) * static_cast<uint64_t>(K));
  sp.input(meta, static_cast<uint64_t>(M) * static_cast<uint64_t>(K) / 8);
  sp.input(B, 2 * static_cast<uint64_t>(N) * static_cast<uint64_t>(K));
  sp.output(C, 4 * static_cast<uint64_t>(M) * static_cast<uint64_t>(N));
  MK_TRY(sp.check());
  maskllm::Device d;
  cudaError_t e = maskllm::current_device(&d);
  if (e != cudaSuccess) return maskllm::cuda_fail(e);
  return maskllm::finish(
      maskllm::spmm(d, values, meta, M, K, B, N, C, maskllm::stream_wait_ns(), stream));
}

// ---- Permutation search without caller memory -----------------------------
// For callers that cannot allocate device memory themselves (see
// maskllm_perm_search_static in maskllm.h): the search's scratch lives in a
// fixed array of this library's own device memory.

namespace maskllm {

static __device__ __align__(256) unsigned char
    g_perm_static_scratch[MASKLLM_PERM_SEARCH_STATIC_BYTES];

namespace {

// Devices on which a lookup of the array's address has succeeded once.
std::atomic<bool> g_perm_static_seen[kMaxDevices];

// Device address of the array on the current device `dev`.  In host code the
// array's name is only a host-side stand-in, never an address a kernel may
// use.  The address is looked up on every call (a lookup allocates nothing):
// after cudaDeviceReset, or with another context current, the module may sit
// elsewhere, and a remembered address would point at memory that is not the
// array.  The first lookup on a device may load the module, which must not
// happen inside a stream capture: that case is refused before any lookup.
maskllm_status perm_static_scratch(int dev, cudaStream_t s, void** addr) {
  if (dev < 0 || dev >= kMaxDevices) return cuda_fail(cudaErrorInvalidDevice);
  if (!g_perm_static_seen[dev].load(std::memory_order_acquire)) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    const cudaError_t e = cudaStreamIsCapturing(s, &cap);
    if (e != cudaSuccess) return cuda_fail(e);
    if (cap != cudaStreamCaptureStatusNone) return MASKLLM_ERR_INVALID_ARG;
  }
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_perm_static_scratch);
  if (e != cudaSuccess) return cuda_fail(e);
  g_perm_static_seen[dev].store(true, std::memory_order_release);
  *addr = p;
  return MASKLLM_OK;
}

}  // namespace
}  // namespace maskllm

extern "C" maskllm_status maskllm_perm_search_static(const uint16_t* W, int64_t rows,
                                                     int64_t cols, int32_t* perm,
                                                     int32_t max_swaps, int32_t* swaps_out,
                                                     int64_t* gains_out, int32_t* n_swaps_out,
                                                     int32_t* shift_out,
                                                     maskllm_stream_t stream) {
  const void* ptrs[] = {W, perm, n_swaps_out};
  MK_TRY(maskllm::check_ptrs(ptrs, 3));
  MK_TRY(maskllm::check_optional(swaps_out));
  MK_TRY(maskllm::check_optional(gains_out));
  MK_TRY(maskllm::check_optional(shift_out));
  MK_TRY(maskllm::check_perm_shape(rows, cols));
  if (max_swaps < 0) return MASKLLM_ERR_INVALID_ARG;
  if (maskllm::perm_workspace_bytes(rows, cols) > MASKLLM_PERM_SEARCH_STATIC_BYTES)
    return MASKLLM_ERR_SHAPE;
  maskllm::Spans sp;
  sp.input(W, 2 * static_cast<uint64_t>(rows) * cols);
  sp.output(perm, 4 * static_cast<uint64_t>(cols));
  sp.output(swaps_out, 8 * static_cast<uint64_t>(max_swaps));
  sp.output(gains_out, 8 * static_cast<uint64_t>(max_swaps));
  sp.output(n_swaps_out, 4);
  sp.output(shift_out, 4);
  MK_TRY(sp.check());
  maskllm::Device d;
  cudaError_t e = maskllm::current_device(&d);
  if (e != cudaSuccess) return maskllm::cuda_fail(e);
  void* scratch = nullptr;
  MK_TRY(maskllm::perm_static_scratch(d.ordinal, stream, &scratch));
  return maskllm::finish(maskllm::perm_search(d, W, rows, cols, perm, max_swaps, scratch,
                                              swaps_out, gains_out, n_swaps_out, shift_out,
                                              stream));
}
