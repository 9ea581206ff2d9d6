// kernels_mask.cu -- magnitude prior, forward and backward of the
// differentiable 2:4 mask.
//
// "MaskLLM: Learnable Semi-Structured Sparsity for Large Language Models":
// Fig. 3 (per-group categorical distribution over the 2:4 candidates, Gumbel
// softmax, weighted average of the candidates; all differentiable), Fig. 5
// (logit scale kappa), Table 2 (prior masks initialise the logits), Table 3
// (weight regularisation).  "Accelerating Sparse Deep Neural Networks",
// Sec. 4.1 (magnitude pruning keeps the two largest of four).
//
// All three kernels are HBM-bound streams (8, 10 and 16 bytes per weight).
// One work item is two groups (8 weights): one 16-byte load of W, three
// 16-byte loads of logits, 16-byte stores.  The Gumbel quantile table
// (64 KB) is copied into shared memory once per CTA of a persistent grid.
#include "device_common.cuh"
#include "internal.h"

namespace maskllm {

// Gumbel(0,1) quantiles at the midpoints of 2^14 cells of (0,1), fl32 of
// -ln(-ln((i + 0.5) / 2^14)) computed in double; generated at build time.
__device__ __align__(16) float g_gumbel_table[kTableSize] = {
#include "gumbel_table.inc"
};

// Set by a bounded device-side wait that gave up; read by the host through
// read_and_clear_error_word().
__device__ uint32_t g_error_word = 0;

namespace {

constexpr int kThreads = 512;           // threads per CTA of the mask kernels
constexpr int kCtasPerSm = 2;           // 2 x (64 KB table + 4 KB) shared memory

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// ---------------------------------------------------------------------------
// Magnitude prior: L_c = fl(scale * fl(|w_i| + |w_j|)).
// ---------------------------------------------------------------------------

__device__ __forceinline__ void prior_group(float a0, float a1, float a2, float a3, float s,
                                            float out[kCand]) {
  out[0] = __fmul_rn(s, __fadd_rn(a0, a1));
  out[1] = __fmul_rn(s, __fadd_rn(a0, a2));
  out[2] = __fmul_rn(s, __fadd_rn(a0, a3));
  out[3] = __fmul_rn(s, __fadd_rn(a1, a2));
  out[4] = __fmul_rn(s, __fadd_rn(a1, a3));
  out[5] = __fmul_rn(s, __fadd_rn(a2, a3));
}

__global__ void __launch_bounds__(256) prior_kernel(const uint4* __restrict__ W,
                                                    float4* __restrict__ L, int64_t items,
                                                    float scale) {
  for (int64_t q = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; q < items;
       q += (int64_t)gridDim.x * blockDim.x) {
    const uint4 w = __ldcs(W + q);
    float a[kCand], b[kCand];
    prior_group(fabsf(bf16_lo(w.x)), fabsf(bf16_hi(w.x)), fabsf(bf16_lo(w.y)),
                fabsf(bf16_hi(w.y)), scale, a);
    prior_group(fabsf(bf16_lo(w.z)), fabsf(bf16_hi(w.z)), fabsf(bf16_lo(w.w)),
                fabsf(bf16_hi(w.w)), scale, b);
    float4* o = L + 3 * q;
    __stcs(o + 0, make_float4(a[0], a[1], a[2], a[3]));
    __stcs(o + 1, make_float4(a[4], a[5], b[0], b[1]));
    __stcs(o + 2, make_float4(b[2], b[3], b[4], b[5]));
  }
}

// ---------------------------------------------------------------------------
// Forward.
// ---------------------------------------------------------------------------

struct FwdParams {
  const uint4* __restrict__ W;
  const float4* __restrict__ L;
  uint4* __restrict__ Wout;
  float* __restrict__ row_sq;   // nullable
  float4* __restrict__ probs;   // nullable
  int64_t rows;
  int32_t ipr;                  // items (pairs of groups) per row = cols / 8
  int32_t seg;                  // threads that share one row in a pass
  int32_t rows_per_pass;
  float kappa;
  float rho;
  uint32_t step;
  uint32_t tensor_id;
  RoundKeys keys;
};

// One group: returns the two packed bf16 words of W' and adds sum x^2.
template <bool kProbs>
__device__ __forceinline__ void fwd_group(const FwdParams& p, const float* tab, uint64_t gidx,
                                          const float L[kCand], uint32_t w01, uint32_t w23,
                                          uint32_t& o01, uint32_t& o23, float& acc,
                                          float prob_out[kCand]) {
  float g[kCand], e[kCand], inv, num[4], M[4];
  gumbel6(group_words(gidx, p.step, p.tensor_id, p.keys), tab, g);
  softmax6(L, g, p.kappa, p.rho, e, inv, num);
  soft_mask4(num, inv, M);
  const float x0 = __fmul_rn(bf16_lo(w01), M[0]);
  const float x1 = __fmul_rn(bf16_hi(w01), M[1]);
  const float x2 = __fmul_rn(bf16_lo(w23), M[2]);
  const float x3 = __fmul_rn(bf16_hi(w23), M[3]);
  o01 = pack_bf16x2_rn(x0, x1);
  o23 = pack_bf16x2_rn(x2, x3);
  acc = __fmaf_rn(x0, x0, acc);
  acc = __fmaf_rn(x1, x1, acc);
  acc = __fmaf_rn(x2, x2, acc);
  acc = __fmaf_rn(x3, x3, acc);
  if (kProbs) {
#pragma unroll
    for (int c = 0; c < kCand; ++c) prob_out[c] = e[c] * inv;
  }
}

template <bool kProbs>
__device__ __forceinline__ void fwd_item(const FwdParams& p, const float* tab, int64_t q,
                                         float& acc) {
  const uint4 w = __ldcs(p.W + q);
  const float4 a = __ldcs(p.L + 3 * q);
  const float4 b = __ldcs(p.L + 3 * q + 1);
  const float4 c = __ldcs(p.L + 3 * q + 2);
  const float La[kCand] = {a.x, a.y, a.z, a.w, b.x, b.y};
  const float Lb[kCand] = {b.z, b.w, c.x, c.y, c.z, c.w};
  uint4 o;
  float pa[kCand], pb[kCand];
  fwd_group<kProbs>(p, tab, 2 * static_cast<uint64_t>(q), La, w.x, w.y, o.x, o.y, acc, pa);
  fwd_group<kProbs>(p, tab, 2 * static_cast<uint64_t>(q) + 1, Lb, w.z, w.w, o.z, o.w, acc, pb);
  __stcs(p.Wout + q, o);
  if (kProbs) {
    float4* d = p.probs + 3 * q;
    d[0] = make_float4(pa[0], pa[1], pa[2], pa[3]);
    d[1] = make_float4(pa[4], pa[5], pb[0], pb[1]);
    d[2] = make_float4(pb[2], pb[3], pb[4], pb[5]);
  }
}

// Persistent grid; CTA b owns the contiguous rows [rows*b/G, rows*(b+1)/G).
// A pass covers rows_per_pass rows: either one row whose items are strided
// over all threads (seg = kThreads), or several short rows of seg = ipr
// threads each.  Each thread sums x^2 over its items in a fixed order; the
// row total is then a fixed-order lane-strided sum of the per-thread values
// and a butterfly over the warp -- deterministic for a given cols.
template <bool kProbs>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) fwd_kernel(const FwdParams p) {
  extern __shared__ __align__(16) float smem[];
  float* tab = smem;
  float* part = smem + kTableSize;  // [2][kThreads]
  load_table(tab, g_gumbel_table);
  __syncthreads();

  const int64_t r0 = p.rows * blockIdx.x / gridDim.x;
  const int64_t r1 = p.rows * (blockIdx.x + 1) / gridDim.x;
  const int t = threadIdx.x;
  const int seg_id = t / p.seg;
  const int seg_pos = t - seg_id * p.seg;
  const int warp = t >> 5, lane = t & 31;
  int buf = 0;
  for (int64_t rb = r0; rb < r1; rb += p.rows_per_pass) {
    float acc = 0.f;
    const int64_t r = rb + seg_id;
    if (seg_id < p.rows_per_pass && r < r1) {
      for (int i = seg_pos; i < p.ipr; i += p.seg) fwd_item<kProbs>(p, tab, r * p.ipr + i, acc);
    }
    if (p.row_sq != nullptr) {
      float* pb = part + buf * kThreads;
      pb[t] = acc;
      __syncthreads();
      for (int j = warp; j < p.rows_per_pass && rb + j < r1; j += kThreads / 32) {
        float s = 0.f;
        for (int k = lane; k < p.seg; k += 32) s += pb[j * p.seg + k];
        s = warp_sum(s);
        if (lane == 0) p.row_sq[rb + j] = s;
      }
      buf ^= 1;
    }
  }
}

// ---------------------------------------------------------------------------
// Backward.
// ---------------------------------------------------------------------------

struct BwdParams {
  const uint4* __restrict__ W;
  const float4* __restrict__ L;
  const uint4* __restrict__ G;
  float4* __restrict__ dL;
  int64_t items;
  float kappa;
  float rho;
  float dz_dlogit;   // fl32(kappa * rho)
  float two_reg;     // 2 * reg_coeff
  uint32_t step;
  uint32_t tensor_id;
  RoundKeys keys;
};

template <bool kReg>
__device__ __forceinline__ void bwd_group(const BwdParams& p, const float* tab, uint64_t gidx,
                                          const float L[kCand], uint32_t w01, uint32_t w23,
                                          uint32_t g01, uint32_t g23, float out[kCand]) {
  float g[kCand], e[kCand], inv, num[4];
  gumbel6(group_words(gidx, p.step, p.tensor_id, p.keys), tab, g);
  softmax6(L, g, p.kappa, p.rho, e, inv, num);
  const float w[4] = {bf16_lo(w01), bf16_hi(w01), bf16_lo(w23), bf16_hi(w23)};
  float t[4] = {bf16_lo(g01), bf16_hi(g01), bf16_lo(g23), bf16_hi(g23)};
  if (kReg) {
    float M[4];
    soft_mask4(num, inv, M);
#pragma unroll
    for (int j = 0; j < 4; ++j) t[j] = __fmaf_rn(p.two_reg, __fmul_rn(w[j], M[j]), t[j]);
  }
  float h[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) h[j] = t[j] * w[j];
  const float dp[kCand] = {h[0] + h[1], h[0] + h[2], h[0] + h[3],
                           h[1] + h[2], h[1] + h[3], h[2] + h[3]};
  float pr[kCand];
  float r = 0.f;
#pragma unroll
  for (int c = 0; c < kCand; ++c) {
    pr[c] = e[c] * inv;
    r = __fmaf_rn(pr[c], dp[c], r);
  }
#pragma unroll
  for (int c = 0; c < kCand; ++c) out[c] = (p.dz_dlogit * pr[c]) * (dp[c] - r);
}

template <bool kReg>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) bwd_kernel(const BwdParams p) {
  extern __shared__ __align__(16) float smem[];
  float* tab = smem;
  load_table(tab, g_gumbel_table);
  __syncthreads();
  for (int64_t q = blockIdx.x * (int64_t)kThreads + threadIdx.x; q < p.items;
       q += (int64_t)gridDim.x * kThreads) {
    const uint4 w = __ldcs(p.W + q);
    const uint4 gr = __ldcs(p.G + q);
    const float4 a = __ldcs(p.L + 3 * q);
    const float4 b = __ldcs(p.L + 3 * q + 1);
    const float4 c = __ldcs(p.L + 3 * q + 2);
    const float La[kCand] = {a.x, a.y, a.z, a.w, b.x, b.y};
    const float Lb[kCand] = {b.z, b.w, c.x, c.y, c.z, c.w};
    float da[kCand], db[kCand];
    bwd_group<kReg>(p, tab, 2 * static_cast<uint64_t>(q), La, w.x, w.y, gr.x, gr.y, da);
    bwd_group<kReg>(p, tab, 2 * static_cast<uint64_t>(q) + 1, Lb, w.z, w.w, gr.z, gr.w, db);
    float4* d = p.dL + 3 * q;
    __stcs(d + 0, make_float4(da[0], da[1], da[2], da[3]));
    __stcs(d + 1, make_float4(da[4], da[5], db[0], db[1]));
    __stcs(d + 2, make_float4(db[2], db[3], db[4], db[5]));
  }
}

constexpr size_t kFwdSmem = (kTableSize + 2 * kThreads) * sizeof(float);
constexpr size_t kBwdSmem = kTableSize * sizeof(float);

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(bytes));
}

float reciprocal_fp32(float tau) { return static_cast<float>(1.0 / static_cast<double>(tau)); }

}  // namespace

cudaError_t launch_prior_init(const Device& d, const uint16_t* W, int64_t rows, int64_t cols,
                              float scale, float* logits, cudaStream_t s) {
  const int64_t items = rows * cols / 8;
  const int64_t want = (items + 255) / 256;
  const int grid = static_cast<int>(want < 8LL * d.num_sms ? want : 8LL * d.num_sms);
  prior_kernel<<<grid, 256, 0, s>>>(reinterpret_cast<const uint4*>(W),
                                    reinterpret_cast<float4*>(logits), items, scale);
  return cudaGetLastError();
}

cudaError_t launch_forward(const Device& d, const uint16_t* W, const float* logits, int64_t rows,
                           int64_t cols, float tau, float kappa, RngArgs rng, uint16_t* W_out,
                           float* row_sq, float* probs, cudaStream_t s) {
  FwdParams p;
  p.W = reinterpret_cast<const uint4*>(W);
  p.L = reinterpret_cast<const float4*>(logits);
  p.Wout = reinterpret_cast<uint4*>(W_out);
  p.row_sq = row_sq;
  p.probs = reinterpret_cast<float4*>(probs);
  p.rows = rows;
  p.ipr = static_cast<int32_t>(cols / 8);
  if (p.ipr >= kThreads) {
    p.seg = kThreads;
    p.rows_per_pass = 1;
  } else {
    p.seg = p.ipr;
    p.rows_per_pass = kThreads / p.ipr;
  }
  p.kappa = kappa;
  p.rho = reciprocal_fp32(tau);
  p.step = rng.step;
  p.tensor_id = rng.tensor_id;
  p.keys = make_round_keys(rng.seed);
  const int64_t passes = (rows + p.rows_per_pass - 1) / p.rows_per_pass;
  const int64_t cap = static_cast<int64_t>(kCtasPerSm) * d.num_sms;
  const int grid = static_cast<int>(passes < cap ? passes : cap);
  cudaError_t e;
  if (probs != nullptr) {
    if ((e = set_smem(fwd_kernel<true>, kFwdSmem)) != cudaSuccess) return e;
    fwd_kernel<true><<<grid, kThreads, kFwdSmem, s>>>(p);
  } else {
    if ((e = set_smem(fwd_kernel<false>, kFwdSmem)) != cudaSuccess) return e;
    fwd_kernel<false><<<grid, kThreads, kFwdSmem, s>>>(p);
  }
  return cudaGetLastError();
}

cudaError_t launch_backward(const Device& d, const uint16_t* W, const float* logits,
                            const uint16_t* G, int64_t rows, int64_t cols, float tau, float kappa,
                            RngArgs rng, float reg_coeff, float* dlogits, cudaStream_t s) {
  BwdParams p;
  p.W = reinterpret_cast<const uint4*>(W);
  p.L = reinterpret_cast<const float4*>(logits);
  p.G = reinterpret_cast<const uint4*>(G);
  p.dL = reinterpret_cast<float4*>(dlogits);
  p.items = rows * cols / 8;
  p.kappa = kappa;
  p.rho = reciprocal_fp32(tau);
  p.dz_dlogit = static_cast<float>(static_cast<double>(kappa) * static_cast<double>(p.rho));
  p.two_reg = 2.0f * reg_coeff;
  p.step = rng.step;
  p.tensor_id = rng.tensor_id;
  p.keys = make_round_keys(rng.seed);
  const int64_t want = (p.items + kThreads - 1) / kThreads;
  const int64_t cap = static_cast<int64_t>(kCtasPerSm) * d.num_sms;
  const int grid = static_cast<int>(want < cap ? want : cap);
  cudaError_t e;
  if (reg_coeff != 0.0f) {
    if ((e = set_smem(bwd_kernel<true>, kBwdSmem)) != cudaSuccess) return e;
    bwd_kernel<true><<<grid, kThreads, kBwdSmem, s>>>(p);
  } else {
    if ((e = set_smem(bwd_kernel<false>, kBwdSmem)) != cudaSuccess) return e;
    bwd_kernel<false><<<grid, kThreads, kBwdSmem, s>>>(p);
  }
  return cudaGetLastError();
}

cudaError_t read_and_clear_error_word(cudaStream_t s, uint32_t* value) {
  uint32_t zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(value, g_error_word, sizeof(uint32_t), 0,
                                            cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return e;
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return e;
  if (*value != 0) {
    e = cudaMemcpyToSymbolAsync(g_error_word, &zero, sizeof(uint32_t), 0, cudaMemcpyHostToDevice,
                                s);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(s);
  }
  return e;
}

}  // namespace maskllm
