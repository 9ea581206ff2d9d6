// kernels_pack.cu -- the inverse of 2:4 compression, logits from a given
// mask, and the noise-word export.
//
// "Accelerating Sparse Deep Neural Networks", Sec. 3.1: a 2:4 matrix is
// stored as the two kept values of each group of four plus 2 bits per kept
// value giving its position; the constant sparsity of every group means
// fixed offsets and no data-dependent indirection.  (The compression itself
// is a streaming kernel, kernels_stream.cu.)
//
// Decompression: one work item is 8 groups = 32 weights = one 32-bit
// metadata word: 32 bytes of values and 4 bytes of metadata in, 64 bytes of
// W out.
#include "device_common.cuh"
#include "internal.h"

namespace maskllm {
namespace {

__global__ void __launch_bounds__(256) decompress_kernel(const uint4* __restrict__ vals,
                                                         const uint32_t* __restrict__ meta,
                                                         uint4* __restrict__ W, int64_t items) {
  for (int64_t q = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; q < items;
       q += (int64_t)gridDim.x * blockDim.x) {
    const uint4 v0 = __ldcs(vals + 2 * q);
    const uint4 v1 = __ldcs(vals + 2 * q + 1);
    const uint32_t code_word = __ldcs(meta + q);
    const uint32_t vv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    uint32_t o[16];
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      const uint32_t code = (code_word >> (4 * g)) & 0xFu;
      const uint32_t i = code & 3u, j = code >> 2;
      const uint32_t a = vv[g] & 0xFFFFu, b = vv[g] >> 16;
      uint32_t e[4];
#pragma unroll
      for (uint32_t k = 0; k < 4; ++k) e[k] = (k == i) ? a : ((k == j) ? b : 0u);
      o[2 * g] = e[0] | (e[1] << 16);
      o[2 * g + 1] = e[2] | (e[3] << 16);
    }
#pragma unroll
    for (int v = 0; v < 4; ++v)
      __stcs(W + 4 * q + v, make_uint4(o[4 * v], o[4 * v + 1], o[4 * v + 2], o[4 * v + 3]));
  }
}

// Logits from a given mask ("MaskLLM" project page, Table 2: learned masks
// start from a prior mask): high on the candidate a group's 4-bit code names,
// low on the other five; a code naming no candidate gives low everywhere.
// Candidate of each code, one nibble per code (0xF = none):
// 0x4 -> c0, 0x8 -> c1, 0xC -> c2, 0x9 -> c3, 0xD -> c4, 0xE -> c5.
constexpr uint64_t kCandOfCode = 0xF542FF31FFF0FFFFull;
constexpr int kPfmThreads = 256;
// Tiles whose code bytes a warp loads at once before it writes any of them:
// one load latency per run instead of per tile (the reads wait behind the
// kernel's writes in DRAM).  218 -> 194 us for the LLaMA-2-7B block; 8 tiles
// ahead measured 204 us (53 registers), 16 ahead 195 us.
constexpr int kPfmAhead = 4;

// A batch of matrices as one list of warp tiles: a tile is 32 code bytes
// (64 groups) of one matrix; matrix m owns tiles [tile_begin[m],
// tile_begin[m + 1]).
struct PfmBatch {
  const uint8_t* meta[kMaxBatch];   // code bytes: group k at nibble k % 2 of byte k / 2
  float4* L[kMaxBatch];             // logits, 6 floats per group
  int64_t items[kMaxBatch];         // code bytes (pairs of groups) of the matrix
  int64_t tile_begin[kMaxBatch + 1];
  int64_t run_begin[kMaxBatch + 1];   // runs of kPfmAhead tiles of one matrix
  int32_t n;
  float high, low;
};

// Each warp takes runs of kPfmAhead tiles of one matrix in a grid-stride
// loop (ascending, so the matrix of the next run is found by moving forward
// through run_begin): it loads the code bytes of the run's tiles, then for
// each tile every thread writes the 48 bytes of logits of its two groups
// into a warp-private shared buffer, and the warp stores the buffer with
// 16-byte stores that are contiguous across lanes.
__global__ void __launch_bounds__(kPfmThreads) prior_from_mask_kernel(const __grid_constant__
                                                                      PfmBatch p) {
  __shared__ __align__(16) float4 buf[kPfmThreads / 32][96];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t warps_total = static_cast<int64_t>(gridDim.x) * (kPfmThreads / 32);
  const int64_t runs = p.run_begin[p.n];
  int m = 0;
  for (int64_t run = blockIdx.x * (int64_t)(kPfmThreads / 32) + warp; run < runs;
       run += warps_total) {
    while (run >= p.run_begin[m + 1]) ++m;
    const int64_t tile0 = (run - p.run_begin[m]) * kPfmAhead;   // matrix-local
    const int64_t tiles_m = p.tile_begin[m + 1] - p.tile_begin[m];
    uint32_t b[kPfmAhead];
#pragma unroll
    for (int j = 0; j < kPfmAhead; ++j) {
      const int64_t item = (tile0 + j) * 32 + lane;
      b[j] = (tile0 + j < tiles_m && item < p.items[m]) ? __ldcs(p.meta[m] + item) : 0u;
    }
#pragma unroll
    for (int j = 0; j < kPfmAhead; ++j) {
      const int64_t local = tile0 + j;
      if (local >= tiles_m) break;
      const int64_t left = p.items[m] - local * 32;    // items in this tile (<= 32 used)
      const int n_items = static_cast<int>(left < 32 ? left : 32);
      if (lane < n_items) {
        float v[12];
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          const uint32_t cand =
              static_cast<uint32_t>(kCandOfCode >> (4 * ((b[j] >> (4 * g)) & 0xFu))) & 0xFu;
#pragma unroll
          for (int c = 0; c < kCand; ++c)
            v[6 * g + c] = (static_cast<uint32_t>(c) == cand) ? p.high : p.low;
        }
        buf[warp][3 * lane + 0] = make_float4(v[0], v[1], v[2], v[3]);
        buf[warp][3 * lane + 1] = make_float4(v[4], v[5], v[6], v[7]);
        buf[warp][3 * lane + 2] = make_float4(v[8], v[9], v[10], v[11]);
      }
      __syncwarp();
      float4* dst = p.L[m] + 3 * local * 32;
#pragma unroll
      for (int k = 0; k < 3; ++k) {
        const int q = lane + 32 * k;                    // 16-byte chunk of the tile
        if (q < 3 * n_items) __stcs(dst + q, buf[warp][q]);
      }
      __syncwarp();
    }
  }
}

struct NoiseParams {
  uint4* out;
  int64_t group_begin;
  int64_t n;
  uint32_t step;
  uint32_t tensor_id;
  RoundKeys keys;
};

__global__ void __launch_bounds__(256) noise_words_kernel(const NoiseParams p) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < p.n;
       i += (int64_t)gridDim.x * blockDim.x) {
    p.out[i] = group_words(static_cast<uint64_t>(p.group_begin + i), p.step, p.tensor_id, p.keys);
  }
}

int grid_for(int64_t items, int threads, const Device& d, int per_sm) {
  const int64_t want = (items + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(per_sm) * d.num_sms;
  return static_cast<int>(want < cap ? want : cap);
}

}  // namespace

cudaError_t launch_decompress(const Device& d, const uint16_t* values, const uint32_t* meta,
                              int64_t rows, int64_t cols, uint16_t* W_out, cudaStream_t s) {
  const int64_t items = rows * cols / 32;
  decompress_kernel<<<grid_for(items, 256, d, 8), 256, 0, s>>>(
      reinterpret_cast<const uint4*>(values), meta, reinterpret_cast<uint4*>(W_out), items);
  return cudaGetLastError();
}

cudaError_t launch_prior_from_mask(const Device& d, const StreamMatrix* mats, int n, float high,
                                   float low, cudaStream_t s) {
  if (n < 1 || n > kMaxBatch) return cudaErrorInvalidValue;
  PfmBatch p;
  p.n = n;
  p.high = high;
  p.low = low;
  p.tile_begin[0] = 0;
  for (int i = 0; i < n; ++i) {
    p.meta[i] = static_cast<const uint8_t*>(mats[i].W);
    p.L[i] = static_cast<float4*>(mats[i].out0);
    p.items[i] = mats[i].rows * mats[i].cols / 8;   // code bytes = pairs of groups
    p.tile_begin[i + 1] = p.tile_begin[i] + (p.items[i] + 31) / 32;
  }
  p.run_begin[0] = 0;
  for (int i = 0; i < n; ++i)
    p.run_begin[i + 1] = p.run_begin[i] +
                         (p.tile_begin[i + 1] - p.tile_begin[i] + kPfmAhead - 1) / kPfmAhead;
  const int64_t want = (p.run_begin[n] + kPfmThreads / 32 - 1) / (kPfmThreads / 32);
  const int64_t cap = 8LL * d.num_sms;
  prior_from_mask_kernel<<<static_cast<int>(want < cap ? want : cap), kPfmThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_noise_words(const Device& d, RngArgs rng, int64_t group_begin, int64_t n,
                               uint32_t* out4, cudaStream_t s) {
  NoiseParams p;
  p.out = reinterpret_cast<uint4*>(out4);
  p.group_begin = group_begin;
  p.n = n;
  p.step = rng.step;
  p.tensor_id = rng.tensor_id;
  p.keys = make_round_keys(rng.seed);
  noise_words_kernel<<<grid_for(n, 256, d, 8), 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace maskllm
