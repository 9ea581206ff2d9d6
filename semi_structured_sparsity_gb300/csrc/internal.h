// internal.h -- launchers shared between the C-ABI layer and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace maskllm {

struct Device {
  int ordinal;
  int num_sms;
};

// The current device and its SM count (cached per device).
cudaError_t current_device(Device* d);

struct RngArgs {
  uint64_t seed;
  uint32_t step;
  uint32_t tensor_id;
};

cudaError_t launch_decompress(const Device& d, const uint16_t* values, const uint32_t* meta,
                              int64_t rows, int64_t cols, uint16_t* W_out, cudaStream_t s);
cudaError_t launch_noise_words(const Device& d, RngArgs rng, int64_t group_begin, int64_t n,
                               uint32_t* out4, cudaStream_t s);

// ---- pipelined streaming kernels (kernels_stream.cu) ----------------------

constexpr int kMaxBatch = 16;   // matrices per launch

struct StreamMatrix {
  const void* W;      // bf16 [rows, cols]
  const void* L;      // fp32 [rows, cols/4, 6]
  const void* G;      // bf16 [rows, cols] (backward)
  void* out0;         // prior: logits; forward: W'; backward: dlogits; compress: values
  void* out1;         // forward: row_sq (nullable); compress: codes
  void* out2;         // forward: probs (nullable); compress: idx (nullable)
  void* out3 = nullptr;   // forward with diagnostics: L1 distance per row (u32)
  void* out4 = nullptr;   // forward with diagnostics: max-probability sum per row (fp32)
  const void* P = nullptr;   // backward with diagnostics: previous draws (u8 per group)
  int64_t rows;
  int64_t cols;
  uint32_t tensor_id;
};

cudaError_t stream_prior_init(const Device& d, const StreamMatrix* m, int n, float scale,
                              cudaStream_t s);
cudaError_t stream_forward(const Device& d, const StreamMatrix* m, int n, float tau, float kappa,
                           RngArgs rng, bool probs, cudaStream_t s);
cudaError_t stream_backward(const Device& d, const StreamMatrix* m, int n, float tau, float kappa,
                            RngArgs rng, float reg_coeff, cudaStream_t s);
cudaError_t stream_hard_compress(const Device& d, const StreamMatrix* m, int n, cudaStream_t s);
// G = previous draws (u8 per group, nullable); out0 = draws (nullable);
// out1 = L1 distance per row (u32, needs G); out2 = max-probability sum per row
cudaError_t stream_mask_stats(const Device& d, const StreamMatrix* m, int n, float tau, float kappa,
                              RngArgs rng, cudaStream_t s);
// The forward (out0 = W', out1 = row_sq) with the diagnostics of
// stream_mask_stats in the same pass: G = previous draws, out2 = draws,
// out3 = L1 per row, out4 = max-probability sum per row (all nullable).
cudaError_t stream_forward_stats(const Device& d, const StreamMatrix* m, int n, float tau,
                                 float kappa, RngArgs rng, cudaStream_t s);
// The backward (out0 = dlogits) with the diagnostics in the same pass: P =
// previous draws, out1 = draws, out2 = L1 per row, out3 = max-probability
// sum per row (all nullable; out2 needs P).
cudaError_t stream_backward_stats(const Device& d, const StreamMatrix* m, int n, float tau,
                                  float kappa, RngArgs rng, float reg_coeff, cudaStream_t s);
// Logits from 2:4 codes, up to kMaxBatch matrices in one launch
// (kernels_pack.cu): W = the codes (u32 [rows, cols/32]), out0 = logits.
cudaError_t launch_prior_from_mask(const Device& d, const StreamMatrix* m, int n, float high,
                                   float low, cudaStream_t s);
// ---- channel permutation before pruning (kernels_perm.cu) -----------------

constexpr int32_t kPermBadPermutation = -1;   // search / gains outcome codes
constexpr int32_t kPermNonFinite = -2;
constexpr int32_t kPermShiftNonFinite = -2147483647 - 1;   // shift of a non-finite matrix
constexpr int64_t kPermMaxCols = 32768;
constexpr int64_t kPermMaxRows = int64_t(1) << 24;

// Control block of one search or gains call, in the caller's workspace.
struct PermCtl {
  unsigned long long key;   // best swap of the step (0: none)
  uint32_t tiles_done;      // tiles of the best-pair scan finished this step
  uint32_t maxbits;         // largest |w| bit pattern
  uint32_t flags;           // bit 0: bad permutation
  int32_t shift;
  int32_t code;             // 0, kPermBadPermutation or kPermNonFinite
  int32_t done;
  int32_t n_swaps;
  int32_t rec_a, rec_b;     // the swap applied in this step
};

int64_t perm_workspace_bytes(int64_t rows, int64_t cols);
cudaError_t perm_search(const Device& d, const uint16_t* W, int64_t rows, int64_t cols,
                        int32_t* perm, int32_t max_swaps, void* workspace, int32_t* swaps_out,
                        int64_t* gains_out, int32_t* n_swaps_out, int32_t* shift_out,
                        cudaStream_t s);
cudaError_t perm_swap_gains(const Device& d, const uint16_t* W, int64_t rows, int64_t cols,
                            const int32_t* perm, void* workspace, int64_t* gains_out,
                            int32_t* info_out, int32_t* shift_out, cudaStream_t s);
cudaError_t perm_shift(const Device& d, const uint16_t* W, int64_t rows, int64_t cols,
                       int32_t* shift_out, cudaStream_t s);
cudaError_t perm_metric(const Device& d, const uint16_t* W, int64_t rows, int64_t cols,
                        const int32_t* perm, const int32_t* shift, uint64_t* metric_out,
                        cudaStream_t s);
cudaError_t permute_columns(const Device& d, const uint16_t* W, int64_t rows, int64_t cols,
                            const int32_t* perm, uint16_t* W_out, cudaStream_t s);
cudaError_t read_and_clear_perm_error(cudaStream_t s, uint32_t* value);

// ---- 2:4 sparse x dense product (kernels_spmm.cu) ------------------------
// C [M, N] fp32 = A B^T, A as values bf16 [M, K/2] + codes u32 [M, K/32],
// B bf16 [N, K].  Returns cudaErrorInvalidValue when the tensor maps cannot
// be encoded.
// Test hook: every later sparse product uses tile width n (128..256, a
// multiple of 32), or chooses it per call again when n == 0.
void spmm_force_tile_width(int n);
cudaError_t spmm(const Device& d, const uint16_t* values, const uint32_t* meta, int64_t M,
                 int64_t K, const uint16_t* B, int64_t N, float* C, uint64_t wait_ns,
                 cudaStream_t s);
cudaError_t read_and_clear_spmm_error(cudaStream_t s, uint32_t* value);

void stream_set_wait_ns(uint64_t ns);
uint64_t stream_wait_ns();
void stream_set_withhold_loads(int on);
cudaError_t read_and_clear_stream_error(cudaStream_t s, uint32_t* value);

}  // namespace maskllm
