// kernels_perm.cu -- channel permutation before 2:4 pruning: the quality
// metric, the gain of every channel swap, and a steepest-ascent swap search.
//
// "Accelerating Sparse Deep Neural Networks", Sec. 4.1 (and its Fig. 5):
// permuting the input channels (columns) of a weight matrix before 2:4
// magnitude pruning raises the magnitude that the pruning keeps; the layer
// that produces those channels is permuted alike, so the product is
// unchanged.  "Channel Permutations for N:M Sparsity" (abstract): a quality
// metric judges a permutation; a search looks for good ones.
//
// Definitions (slot i of the permuted matrix holds channel perm[i]):
//   q(w)      = floor(|w| 2^k),  k = 31 - ceil(log2 rows) - floor(log2 max|w|)
//   metric    = sum over rows and groups of the two largest q of the group
//   gain(a,b) = metric after exchanging the channels of slots a and b, minus
//               the metric before (0 for two slots of one group)
//   search    = apply the swap of largest gain (ties: smallest a, then
//               smallest b, a < b) while some gain is positive, at most
//               max_swaps times.
// k makes every column sum of q over the rows smaller than 2^32, and all the
// arithmetic below is on integers, so the results do not depend on the order
// of any addition.
//
// Decomposition.  Let the three values of a group other than slot a's be
// o1 >= o2 >= o3; with value v in slot a the group keeps o1 + max(o2, v).  So
// with
//   V[r][i] = q(W[r][perm[i]])                        value in slot i
//   S[r][i] = median of the three V of slot i's group-mates
//   E[a][b] = sum over r of max(S[r][a], V[r][b])     (slot a receives b)
// the gain is (E[a][b] - E[a][a]) + (E[b][a] - E[b][b]) for slots of
// different groups: o1 cancels.  E is a max-plus "product" of S and V over
// the rows, computed by a tiled kernel; after a swap of slots a and b the
// columns a and b of V, hence of E, trade places, and S changes only for the
// three group-mates of a and of b, whose six rows of E are recomputed.  One
// search step is three kernels: best (a persistent scan of the 32 x 32 tiles
// of pairs, each block's largest gain, then the largest of those), apply (the
// swap and the cheap updates), rows (the six E rows).  All of them return at
// once when the search has stopped,
// so the host enqueues max_swaps steps without waiting for any of them.
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace maskllm {

// bit 0: a permutation entry out of [0, cols) (metric and column-permute
// calls; such entries read as zero)
__device__ uint32_t g_perm_error_word = 0;

namespace {

constexpr uint32_t kKeyIndexBits = 30;   // a << 15 | b, cols <= 32768
constexpr unsigned long long kKeyIndexMask = (1ull << kKeyIndexBits) - 1;

// Fixed-point shift of a matrix whose largest magnitude has bf16 bits
// `maxbits` (sign cleared, finite).
__device__ __forceinline__ int32_t shift_of(uint32_t maxbits, int64_t rows) {
  if (maxbits == 0) return 0;
  const int ef = static_cast<int>(maxbits >> 7);
  const int e = ef ? ef - 127 : (31 - __clz(static_cast<int>(maxbits & 0x7Fu))) - 133;
  const int lr = rows <= 1 ? 0 : 64 - __clzll(static_cast<long long>(rows - 1));
  return 31 - lr - e;
}

// q(w) = floor(|w| 2^k) of a bf16 bit pattern: |w| = m 2^e2 with an integer
// significand m (8 bits for normal numbers, the 7 stored bits for
// subnormals), so q is a shift of m.  Saturates should a caller's k be too
// large for w.
__device__ __forceinline__ uint32_t fixed_of(uint32_t bits, int32_t k) {
  const uint32_t b = bits & 0x7FFFu;
  const uint32_t ef = b >> 7;
  const uint32_t m = ef ? (0x80u | (b & 0x7Fu)) : (b & 0x7Fu);
  const int sh = (ef ? static_cast<int>(ef) - 134 : -133) + k;
  if (sh >= 0) {
    if (sh >= 32) return m ? 0xFFFFFFFFu : 0u;
    const uint64_t v = static_cast<uint64_t>(m) << sh;
    return v > 0xFFFFFFFFull ? 0xFFFFFFFFu : static_cast<uint32_t>(v);
  }
  return sh <= -32 ? 0u : m >> (-sh);
}

__device__ __forceinline__ uint32_t median3(uint32_t x, uint32_t y, uint32_t z) {
  return max(min(x, y), min(max(x, y), z));
}

// Sum of the two largest of four.
__device__ __forceinline__ uint32_t top2(uint32_t q0, uint32_t q1, uint32_t q2, uint32_t q3) {
  const uint32_t h01 = max(q0, q1), l01 = min(q0, q1);
  const uint32_t h23 = max(q2, q3), l23 = min(q2, q3);
  return max(h01, h23) + max(min(h01, h23), max(l01, l23));
}

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long w = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    v = w > v ? w : v;
  }
  return v;
}

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

__device__ __forceinline__ uint32_t warp_max_u32(uint32_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// ---------------------------------------------------------------------------
// Set-up: permutation check and largest magnitude.
// ---------------------------------------------------------------------------

// Largest magnitude bit pattern of W (n weights, n % 8 == 0) into *maxbits;
// when perm is given, also marks each entry in `seen` and raises
// PermCtl::flags bit 0 for an entry out of range or seen twice.
__global__ void __launch_bounds__(256) perm_scan_kernel(const uint4* __restrict__ W, int64_t n8,
                                                        const int32_t* __restrict__ perm,
                                                        int32_t cols, uint32_t* seen,
                                                        uint32_t* maxbits, uint32_t* flags) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t t0 = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  if (perm != nullptr) {
    for (int64_t i = t0; i < cols; i += stride) {
      const int32_t p = perm[i];
      if (p < 0 || p >= cols) {
        atomicOr(flags, 1u);
      } else {
        const uint32_t bit = 1u << (p & 31);
        if (atomicOr(&seen[p >> 5], bit) & bit) atomicOr(flags, 1u);
      }
    }
  }
  uint32_t mx = 0;
  for (int64_t i = t0; i < n8; i += stride) {
    const uint4 v = W[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) mx = max(mx, max(w[j] & 0x7FFFu, (w[j] >> 16) & 0x7FFFu));
  }
  mx = warp_max_u32(mx);
  if ((threadIdx.x & 31) == 0 && mx != 0) atomicMax(maxbits, mx);
}

// V and S of every row (one block per row at a time; the row is staged in
// shared memory so the permuted reads stay on chip).  Block 0 also settles
// the status: a bad permutation or a non-finite weight stops everything.
__global__ void __launch_bounds__(256) perm_prepare_kernel(const uint16_t* __restrict__ W,
                                                           int64_t rows, int32_t cols,
                                                           const int32_t* __restrict__ perm,
                                                           uint32_t* __restrict__ S,
                                                           uint32_t* __restrict__ V,
                                                           PermCtl* ctl) {
  extern __shared__ __align__(16) uint16_t row[];
  const uint32_t mb = ctl->maxbits;
  const uint32_t flags = ctl->flags | (mb >= 0x7F80u ? 2u : 0u);
  const int32_t k = flags ? 0 : shift_of(mb, rows);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    ctl->shift = k;
    ctl->code = (flags & 1u) ? kPermBadPermutation : (flags ? kPermNonFinite : 0);
    if (flags) ctl->done = 1;
  }
  if (flags) return;
  const int32_t n8 = cols / 8, ng = cols / 4;
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    const uint4* src = reinterpret_cast<const uint4*>(W + r * cols);
    for (int i = threadIdx.x; i < n8; i += blockDim.x) reinterpret_cast<uint4*>(row)[i] = src[i];
    __syncthreads();
    for (int g = threadIdx.x; g < ng; g += blockDim.x) {
      const int4 p = reinterpret_cast<const int4*>(perm)[g];
      const uint32_t q0 = fixed_of(row[p.x], k), q1 = fixed_of(row[p.y], k);
      const uint32_t q2 = fixed_of(row[p.z], k), q3 = fixed_of(row[p.w], k);
      reinterpret_cast<uint4*>(V + r * cols)[g] = make_uint4(q0, q1, q2, q3);
      reinterpret_cast<uint4*>(S + r * cols)[g] =
          make_uint4(median3(q1, q2, q3), median3(q0, q2, q3), median3(q0, q1, q3),
                     median3(q0, q1, q2));
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// E[a][b] = sum_r max(S[r][a], V[r][b]): 128 x 128 tiles of E per block, 16
// rows of S and V per step through shared memory (double-buffered through
// registers), 8 x 8 outputs per thread.  The sums are exact (below 2^32 by
// the choice of k).
// ---------------------------------------------------------------------------

constexpr int kTile = 128;
constexpr int kKStep = 16;

// acc + x * one as an integer multiply-add.  The loop is bound by the
// integer ALU pipe, which issues the max; with `one` a run-time 1 the adds go
// to the FMA pipe instead of competing with the max for the ALU pipe.
__device__ __forceinline__ uint32_t mad_u32(uint32_t x, uint32_t one, uint32_t acc) {
  uint32_t r;
  asm("mad.lo.u32 %0, %1, %2, %3;" : "=r"(r) : "r"(x), "r"(one), "r"(acc));
  return r;
}

// Two blocks per SM (128 registers): the max-and-add loop is bound by the
// integer pipe's latency with one block of 8 warps (set-up 5.5 -> 4.65 ms on
// 4096 x 4096).
__global__ void __launch_bounds__(256, 2) perm_table_kernel(const uint32_t* __restrict__ S,
                                                         const uint32_t* __restrict__ V,
                                                         uint32_t* __restrict__ E, int64_t rows,
                                                         int32_t cols, uint32_t one,
                                                         const PermCtl* ctl) {
  if (ctl->done) return;
  __shared__ __align__(16) uint32_t sS[2][kKStep][kTile];
  __shared__ __align__(16) uint32_t sV[2][kKStep][kTile];
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int64_t a0 = static_cast<int64_t>(blockIdx.y) * kTile;
  const int64_t b0 = static_cast<int64_t>(blockIdx.x) * kTile;

  uint4 ls[2], lv[2];
  auto fetch = [&](int64_t r0) {
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int e = tid + 256 * u, kr = e >> 5, c4 = (e & 31) * 4;
      const int64_t r = r0 + kr;
      const bool in_r = r < rows;
      ls[u] = (in_r && a0 + c4 < cols)
                  ? *reinterpret_cast<const uint4*>(S + r * cols + a0 + c4)
                  : make_uint4(0, 0, 0, 0);
      lv[u] = (in_r && b0 + c4 < cols)
                  ? *reinterpret_cast<const uint4*>(V + r * cols + b0 + c4)
                  : make_uint4(0, 0, 0, 0);
    }
  };
  auto stash = [&](int buf) {
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int e = tid + 256 * u, kr = e >> 5, c4 = (e & 31) * 4;
      *reinterpret_cast<uint4*>(&sS[buf][kr][c4]) = ls[u];
      *reinterpret_cast<uint4*>(&sV[buf][kr][c4]) = lv[u];
    }
  };

  uint32_t acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0;

  fetch(0);
  stash(0);
  __syncthreads();
  const int64_t nk = (rows + kKStep - 1) / kKStep;
  for (int64_t kt = 0; kt < nk; ++kt) {
    const int buf = static_cast<int>(kt & 1);
    if (kt + 1 < nk) fetch((kt + 1) * kKStep);
#pragma unroll
    for (int kk = 0; kk < kKStep; kk += 2) {
      uint32_t s0[8], s1[8], v0[8], v1[8];
      const uint4 sa = *reinterpret_cast<const uint4*>(&sS[buf][kk][ty * 4]);
      const uint4 sb = *reinterpret_cast<const uint4*>(&sS[buf][kk][64 + ty * 4]);
      const uint4 sc = *reinterpret_cast<const uint4*>(&sS[buf][kk + 1][ty * 4]);
      const uint4 sd = *reinterpret_cast<const uint4*>(&sS[buf][kk + 1][64 + ty * 4]);
      const uint4 va = *reinterpret_cast<const uint4*>(&sV[buf][kk][tx * 4]);
      const uint4 vb = *reinterpret_cast<const uint4*>(&sV[buf][kk][64 + tx * 4]);
      const uint4 vc = *reinterpret_cast<const uint4*>(&sV[buf][kk + 1][tx * 4]);
      const uint4 vd = *reinterpret_cast<const uint4*>(&sV[buf][kk + 1][64 + tx * 4]);
      s0[0] = sa.x; s0[1] = sa.y; s0[2] = sa.z; s0[3] = sa.w;
      s0[4] = sb.x; s0[5] = sb.y; s0[6] = sb.z; s0[7] = sb.w;
      s1[0] = sc.x; s1[1] = sc.y; s1[2] = sc.z; s1[3] = sc.w;
      s1[4] = sd.x; s1[5] = sd.y; s1[6] = sd.z; s1[7] = sd.w;
      v0[0] = va.x; v0[1] = va.y; v0[2] = va.z; v0[3] = va.w;
      v0[4] = vb.x; v0[5] = vb.y; v0[6] = vb.z; v0[7] = vb.w;
      v1[0] = vc.x; v1[1] = vc.y; v1[2] = vc.z; v1[3] = vc.w;
      v1[4] = vd.x; v1[5] = vd.y; v1[6] = vd.z; v1[7] = vd.w;
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          acc[i][j] = mad_u32(max(s0[i], v0[j]), one, acc[i][j]);
          acc[i][j] = mad_u32(max(s1[i], v1[j]), one, acc[i][j]);
        }
    }
    if (kt + 1 < nk) stash(buf ^ 1);
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int64_t a = a0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
    if (a >= cols) continue;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int64_t b = b0 + h * 64 + tx * 4;
      if (b < cols)
        *reinterpret_cast<uint4*>(E + a * cols + b) =
            make_uint4(acc[i][4 * h], acc[i][4 * h + 1], acc[i][4 * h + 2], acc[i][4 * h + 3]);
    }
  }
}

// Gains of all pairs from E (32 x 32 tiles; the transposed tile through
// shared memory).  0 for two slots of one group.
__global__ void __launch_bounds__(256) perm_gains_kernel(const uint32_t* __restrict__ E,
                                                         int32_t cols, int64_t* __restrict__ gains,
                                                         const PermCtl* ctl) {
  if (ctl->code != 0) return;
  __shared__ uint32_t T[32][33], U[32][33], dA[32], dB[32];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int64_t a0 = static_cast<int64_t>(blockIdx.y) * 32, b0 = static_cast<int64_t>(blockIdx.x) * 32;
  for (int i = ty; i < 32; i += 8) {
    T[i][tx] = E[(a0 + i) * cols + b0 + tx];
    U[i][tx] = E[(b0 + i) * cols + a0 + tx];
  }
  if (threadIdx.x < 32) dA[tx] = E[(a0 + tx) * (cols + 1)];
  else if (threadIdx.x < 64) dB[tx] = E[(b0 + tx) * (cols + 1)];
  __syncthreads();
  for (int i = ty; i < 32; i += 8) {
    const int64_t a = a0 + i, b = b0 + tx;
    int64_t g = 0;
    if ((a >> 2) != (b >> 2))
      g = (static_cast<int64_t>(T[i][tx]) - dA[i]) + (static_cast<int64_t>(U[tx][i]) - dB[tx]);
    gains[a * cols + b] = g;
  }
}

// ---------------------------------------------------------------------------
// One search step.
// ---------------------------------------------------------------------------

// The best swap: largest positive gain, then smallest a * 2^15 + b, as one
// 64-bit key (gain << 30 | (2^30 - 1 - (a << 15 | b))).  A persistent grid
// walks the 32 x 32 tiles of slot pairs with tA <= tB (grid-stride over all
// tA, tB; the others are skipped), double-buffering each tile pair's two E
// tiles and diagonal entries with per-thread asynchronous copies so the next
// tile's loads overlap this tile's gains.  Each thread keeps its best gain
// and index, each block writes its largest key (0: none) to its slot of
// `tile_best`, and the last block to finish (a counter, no waiting) reduces
// them into ctl->key and resets the counter.
struct BestTile {
  uint32_t T[32][32];   // E[a0 + i][b0 + j], read along rows
  uint32_t U[32][33];   // E[b0 + i][a0 + j], read along columns (padded)
  uint32_t dA[32], dB[32];
};

__device__ __forceinline__ void cp_async_4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__global__ void __launch_bounds__(256) perm_best_kernel(const uint32_t* __restrict__ E,
                                                        int32_t cols,
                                                        unsigned long long* __restrict__ tile_best,
                                                        PermCtl* ctl) {
  if (ctl->done) return;
  __shared__ __align__(16) BestTile buf[2];
  __shared__ unsigned long long red[8];
  __shared__ int last;
  const int nt = cols / 32;
  const int ntiles = nt * nt;
  const int tid = threadIdx.x, tx = tid & 31, ty = tid >> 5, lane = tid & 31;
  // the next tile pair with tA <= tB at or after t (grid stride), or ntiles
  auto next_tile = [&](int t) {
    while (t < ntiles && t / nt > t % nt) t += gridDim.x;
    return t < ntiles ? t : ntiles;
  };
  auto issue = [&](int t, BestTile& b) {
    const int64_t a0 = static_cast<int64_t>(t / nt) * 32, b0 = static_cast<int64_t>(t % nt) * 32;
    // T: 32 rows x 128 bytes, one 16-byte piece per thread
    const int r = tid >> 3, q = (tid & 7) * 4;
    cp_async_16(&b.T[r][q], E + (a0 + r) * cols + b0 + q);
    // U: 1024 words into the padded rows, four per thread
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int e = tid + 256 * k, rr = e >> 5, cc = e & 31;
      cp_async_4(&b.U[rr][cc], E + (b0 + rr) * cols + a0 + cc);
    }
    if (tid < 32)
      cp_async_4(&b.dA[tid], E + (a0 + tid) * (cols + 1));
    else if (tid < 64)
      cp_async_4(&b.dB[tid - 32], E + (b0 + tid - 32) * (cols + 1));
  };

  int64_t best_g = 0;
  int best_i = 0;
  int t = next_tile(blockIdx.x);
  if (t < ntiles) issue(t, buf[0]);
  cp_async_commit();
  for (int k = 0; t < ntiles; ++k) {
    const int tn = next_tile(t + gridDim.x);
    if (tn < ntiles) issue(tn, buf[(k + 1) & 1]);
    cp_async_commit();
    cp_async_wait<1>();   // this tile's copies (all but the newest group)
    __syncthreads();
    const BestTile& b = buf[k & 1];
    const int ia0 = (t / nt) * 32, ib = (t % nt) * 32 + tx;   // slot numbers < 2^15
    const int64_t db = b.dB[tx];
#pragma unroll
    for (int i = ty; i < 32; i += 8) {
      const int ia = ia0 + i;
      if (ia < ib && (ia >> 2) != (ib >> 2)) {
        const int64_t g =
            (static_cast<int64_t>(b.T[i][tx]) - b.dA[i]) + (static_cast<int64_t>(b.U[tx][i]) - db);
        const int idx = (ia << 15) | ib;
        if (g > best_g || (g == best_g && g > 0 && idx < best_i)) {
          best_g = g;
          best_i = idx;
        }
      }
    }
    __syncthreads();   // before the next issue overwrites this buffer
    t = tn;
  }
  cp_async_wait<0>();
  unsigned long long best =
      best_g > 0 ? (static_cast<unsigned long long>(best_g) << kKeyIndexBits) |
                       (kKeyIndexMask - static_cast<unsigned long long>(best_i))
                 : 0ull;
  best = warp_max_u64(best);
  if (lane == 0) red[ty] = best;
  __syncthreads();
  const uint32_t nblocks = gridDim.x;
  if (tid == 0) {
    unsigned long long m = 0;
    for (int w = 0; w < 8; ++w) m = red[w] > m ? red[w] : m;
    tile_best[blockIdx.x] = m;
    __threadfence();
    last = atomicAdd(&ctl->tiles_done, 1u) == nblocks - 1;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  unsigned long long m = 0;
  for (uint32_t i = tid; i < nblocks; i += blockDim.x) {
    const unsigned long long kk = *reinterpret_cast<volatile const unsigned long long*>(tile_best + i);
    m = kk > m ? kk : m;
  }
  m = warp_max_u64(m);
  if (lane == 0) red[ty] = m;
  __syncthreads();
  if (tid == 0) {
    unsigned long long kk = 0;
    for (int w = 0; w < 8; ++w) kk = red[w] > kk ? red[w] : kk;
    ctl->key = kk;
    ctl->tiles_done = 0;
  }
}

// Applies the step's best swap (or stops the search when there is none):
// the permutation and the log; V's columns a and b, the S of the two groups
// (thread r: row r); E's columns a and b in every row that is not recomputed
// (thread t: row t), and zeroes the six E rows the next kernel accumulates.
__global__ void __launch_bounds__(256) perm_apply_kernel(int32_t* __restrict__ perm,
                                                         uint32_t* __restrict__ S,
                                                         uint32_t* __restrict__ V,
                                                         uint32_t* __restrict__ E, int64_t rows,
                                                         int32_t cols, PermCtl* ctl,
                                                         int32_t* __restrict__ swaps_log,
                                                         int64_t* __restrict__ gains_log) {
  if (ctl->done) return;
  const unsigned long long key = ctl->key;
  const int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  if (key == 0) {
    if (t == 0) ctl->done = 1;
    return;
  }
  const uint32_t code = static_cast<uint32_t>(kKeyIndexMask - (key & kKeyIndexMask));
  const int a = static_cast<int>(code >> 15), b = static_cast<int>(code & 0x7FFFu);
  const int ga = a >> 2, gb = b >> 2;
  if (t < rows) {
    uint32_t* Vr = V + t * cols;
    uint32_t* Sr = S + t * cols;
    const uint32_t va = Vr[a];
    Vr[a] = Vr[b];
    Vr[b] = va;
    const int gs[2] = {ga, gb};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint4 q = reinterpret_cast<const uint4*>(Vr)[gs[h]];
      reinterpret_cast<uint4*>(Sr)[gs[h]] =
          make_uint4(median3(q.y, q.z, q.w), median3(q.x, q.z, q.w), median3(q.x, q.y, q.w),
                     median3(q.x, q.y, q.z));
    }
  }
  if (t < cols) {
    const int g = static_cast<int>(t >> 2);
    const bool mate = (g == ga || g == gb) && t != a && t != b;
    if (!mate) {
      uint32_t* Er = E + t * cols;
      const uint32_t ea = Er[a];
      Er[a] = Er[b];
      Er[b] = ea;
    }
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int x = 4 * (h ? gb : ga) + j;
        if (x != a && x != b) E[static_cast<int64_t>(x) * cols + t] = 0u;
      }
  }
  if (t == 0) {
    const int32_t pa = perm[a];
    perm[a] = perm[b];
    perm[b] = pa;
    const int32_t n = ctl->n_swaps;
    if (swaps_log != nullptr) {
      swaps_log[2 * n] = a;
      swaps_log[2 * n + 1] = b;
    }
    if (gains_log != nullptr) gains_log[n] = static_cast<int64_t>(key >> kKeyIndexBits);
    ctl->n_swaps = n + 1;
    ctl->rec_a = a;
    ctl->rec_b = b;
  }
}

// Recomputes the six E rows of the group-mates of the swapped slots: block
// (x, y) takes 512 columns and one slice of the rows; the six S values of
// each row are staged in shared memory; partial sums are added with integer
// atomics (exact, so the order does not matter).  Also clears the best-swap
// key for the next step.
constexpr int kRowsChunk = 256;

__global__ void __launch_bounds__(256) perm_rows_kernel(const uint32_t* __restrict__ S,
                                                        const uint32_t* __restrict__ V,
                                                        uint32_t* __restrict__ E, int64_t rows,
                                                        int32_t cols, int64_t rows_per_slice,
                                                        PermCtl* ctl) {
  if (ctl->done) return;
  const int a = ctl->rec_a, b = ctl->rec_b;
  // the i-th group-mate: i < 3 in a's group, i >= 3 in b's, skipping a and b
  auto mate = [&](int i) {
    const int s = i < 3 ? a : b, j = i < 3 ? i : i - 3;
    return 4 * (s >> 2) + j + (j >= (s & 3) ? 1 : 0);
  };
  __shared__ __align__(16) uint32_t sx[kRowsChunk][8];
  const int64_t c = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 2;
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * rows_per_slice;
  const int64_t r1 = min(rows, r0 + rows_per_slice);
  uint32_t acc[6][2];
#pragma unroll
  for (int i = 0; i < 6; ++i) acc[i][0] = acc[i][1] = 0;
  for (int64_t rc = r0; rc < r1; rc += kRowsChunk) {
    const int n = static_cast<int>(min(static_cast<int64_t>(kRowsChunk), r1 - rc));
    __syncthreads();
    for (int e = threadIdx.x; e < n * 6; e += blockDim.x) {
      const int rr = e / 6, i = e - 6 * (e / 6);
      sx[rr][i] = S[(rc + rr) * cols + mate(i)];
    }
    __syncthreads();
    if (c < cols) {
      int rr = 0;
      // eight rows' loads in flight per thread before any is used
      for (; rr + 7 < n; rr += 8) {
        uint2 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          v[j] = *reinterpret_cast<const uint2*>(V + (rc + rr + j) * cols + c);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
#pragma unroll
          for (int i = 0; i < 6; ++i) {
            const uint32_t s = sx[rr + j][i];
            acc[i][0] += max(s, v[j].x);
            acc[i][1] += max(s, v[j].y);
          }
        }
      }
      for (; rr < n; ++rr) {
        const uint2 v = *reinterpret_cast<const uint2*>(V + (rc + rr) * cols + c);
#pragma unroll
        for (int i = 0; i < 6; ++i) {
          acc[i][0] += max(sx[rr][i], v.x);
          acc[i][1] += max(sx[rr][i], v.y);
        }
      }
    }
  }
  if (c < cols) {
#pragma unroll
    for (int i = 0; i < 6; ++i) {
      const int64_t x = mate(i);
      atomicAdd(&E[x * cols + c], acc[i][0]);
      atomicAdd(&E[x * cols + c + 1], acc[i][1]);
    }
  }
}

// The call's outcome: the number of swaps, or the status code; the shift.
__global__ void perm_finish_kernel(const PermCtl* ctl, int32_t* n_swaps_out, int32_t* shift_out) {
  if (threadIdx.x != 0) return;
  if (n_swaps_out != nullptr) *n_swaps_out = ctl->code != 0 ? ctl->code : ctl->n_swaps;
  if (shift_out != nullptr) *shift_out = ctl->shift;
}

// ---------------------------------------------------------------------------
// Stand-alone pieces: shift, metric, column permutation.
// ---------------------------------------------------------------------------

__global__ void perm_shift_finish_kernel(int32_t* shift, int64_t rows) {
  if (threadIdx.x != 0) return;
  const uint32_t mb = static_cast<uint32_t>(*shift);
  *shift = mb >= 0x7F80u ? kPermShiftNonFinite : shift_of(mb, rows);
}

// Fixed-point metric of a permutation: one group per thread and step,
// 64-bit sums per warp, one atomic add per warp.
__global__ void __launch_bounds__(256) perm_metric_kernel(const uint16_t* __restrict__ W,
                                                          int64_t rows, int32_t cols,
                                                          const int32_t* __restrict__ perm,
                                                          const int32_t* __restrict__ shift,
                                                          unsigned long long* out) {
  const int32_t k = *shift;
  const int64_t ng = cols / 4, total = rows * ng;
  unsigned long long acc = 0;
  bool bad = false;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / ng, g = i - r * ng;
    const int4 p = reinterpret_cast<const int4*>(perm)[g];
    const int pj[4] = {p.x, p.y, p.z, p.w};
    uint32_t q[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const bool in = pj[j] >= 0 && pj[j] < cols;
      bad |= !in;
      q[j] = in ? fixed_of(W[r * cols + pj[j]], k) : 0u;
    }
    acc += top2(q[0], q[1], q[2], q[3]);
  }
  if (bad) atomicOr(&g_perm_error_word, 1u);
  acc = warp_sum_u64(acc);
  if ((threadIdx.x & 31) == 0 && acc != 0) atomicAdd(out, acc);
}

// W_out[r][i] = W[r][perm[i]], one row per block at a time through shared
// memory, 8 outputs (16 bytes) per thread and step.
__global__ void __launch_bounds__(256) permute_columns_kernel(const uint16_t* __restrict__ W,
                                                              int64_t rows, int32_t cols,
                                                              const int32_t* __restrict__ perm,
                                                              uint16_t* __restrict__ W_out) {
  extern __shared__ __align__(16) uint16_t row[];
  const int32_t n8 = cols / 8;
  bool bad = false;
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    const uint4* src = reinterpret_cast<const uint4*>(W + r * cols);
    for (int i = threadIdx.x; i < n8; i += blockDim.x) reinterpret_cast<uint4*>(row)[i] = src[i];
    __syncthreads();
    for (int i = threadIdx.x; i < n8; i += blockDim.x) {
      const int4 p0 = reinterpret_cast<const int4*>(perm)[2 * i];
      const int4 p1 = reinterpret_cast<const int4*>(perm)[2 * i + 1];
      const int p[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
      uint32_t o[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const bool in0 = p[2 * h] >= 0 && p[2 * h] < cols;
        const bool in1 = p[2 * h + 1] >= 0 && p[2 * h + 1] < cols;
        bad |= !(in0 && in1);
        const uint32_t lo = in0 ? row[p[2 * h]] : 0u, hi = in1 ? row[p[2 * h + 1]] : 0u;
        o[h] = lo | (hi << 16);
      }
      reinterpret_cast<uint4*>(W_out + r * cols)[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    __syncthreads();
  }
  if (bad) atomicOr(&g_perm_error_word, 1u);
}

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

struct Workspace {
  uint32_t* E;
  uint32_t* S;
  uint32_t* V;
  unsigned long long* tile_best;
  PermCtl* ctl;
  uint32_t* seen;
};

Workspace carve(void* ws, int64_t rows, int64_t cols) {
  uint8_t* p = static_cast<uint8_t*>(ws);
  Workspace w;
  w.E = reinterpret_cast<uint32_t*>(p);
  p += round_up(cols * cols * 4, 256);
  w.S = reinterpret_cast<uint32_t*>(p);
  p += round_up(rows * cols * 4, 256);
  w.V = reinterpret_cast<uint32_t*>(p);
  p += round_up(rows * cols * 4, 256);
  w.tile_best = reinterpret_cast<unsigned long long*>(p);
  p += round_up((cols / 32) * (cols / 32 + 1) / 2 * 8, 256);
  w.ctl = reinterpret_cast<PermCtl*>(p);
  p += round_up(static_cast<int64_t>(sizeof(PermCtl)), 256);
  w.seen = reinterpret_cast<uint32_t*>(p);
  return w;
}

int blocks_for(int64_t n, int threads, int64_t cap) {
  const int64_t b = (n + threads - 1) / threads;
  return static_cast<int>(b < 1 ? 1 : (b > cap ? cap : b));
}

// Scan, V/S and E of the starting permutation (shared by search and gains).
cudaError_t prepare_table(const Device& d, const uint16_t* W, int64_t rows, int64_t cols,
                          const int32_t* perm, const Workspace& w, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(w.ctl, 0, sizeof(PermCtl), s);
  if (e == cudaSuccess) e = cudaMemsetAsync(w.seen, 0, round_up(cols, 32) / 8, s);
  if (e != cudaSuccess) return e;
  const int64_t n8 = rows * cols / 8;
  perm_scan_kernel<<<blocks_for(n8, 256, 8LL * d.num_sms), 256, 0, s>>>(
      reinterpret_cast<const uint4*>(W), n8, perm, static_cast<int32_t>(cols), w.seen,
      &w.ctl->maxbits, &w.ctl->flags);
  const size_t row_bytes = static_cast<size_t>(cols) * 2;
  e = cudaFuncSetAttribute(perm_prepare_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(row_bytes));
  if (e != cudaSuccess) return e;
  perm_prepare_kernel<<<blocks_for(rows, 1, 4LL * d.num_sms), 256, row_bytes, s>>>(
      W, rows, static_cast<int32_t>(cols), perm, w.S, w.V, w.ctl);
  const int nt = static_cast<int>((cols + kTile - 1) / kTile);
  perm_table_kernel<<<dim3(nt, nt), 256, 0, s>>>(w.S, w.V, w.E, rows, static_cast<int32_t>(cols),
                                                 1u, w.ctl);
  return cudaGetLastError();
}

}  // namespace

int64_t perm_workspace_bytes(int64_t rows, int64_t cols) {
  return round_up(cols * cols * 4, 256) + 2 * round_up(rows * cols * 4, 256) +
         round_up((cols / 32) * (cols / 32 + 1) / 2 * 8, 256) +
         round_up(static_cast<int64_t>(sizeof(PermCtl)), 256) + round_up(cols, 32) / 8;
}

cudaError_t perm_search(const Device& d, const uint16_t* W, int64_t rows, int64_t cols,
                        int32_t* perm, int32_t max_swaps, void* workspace, int32_t* swaps_out,
                        int64_t* gains_out, int32_t* n_swaps_out, int32_t* shift_out,
                        cudaStream_t s) {
  const Workspace w = carve(workspace, rows, cols);
  cudaError_t e = prepare_table(d, W, rows, cols, perm, w, s);
  if (e != cudaSuccess) return e;
  const int32_t c = static_cast<int32_t>(cols);
  // persistent scan: eight blocks per SM (59.5 us per step against 62.5
  // with four), at most one per tile pair and no more than tile_best holds
  // (nt (nt + 1) / 2 slots)
  const int64_t nt = cols / 32;
  int64_t best_blocks = 8LL * d.num_sms;
  if (best_blocks > nt * (nt + 1) / 2) best_blocks = nt * (nt + 1) / 2;
  const unsigned best_grid = static_cast<unsigned>(best_blocks);
  const int apply_blocks = blocks_for(rows > cols ? rows : cols, 256, 1LL << 30);
  const int col_blocks = static_cast<int>((cols + 511) / 512);
  // about four blocks of row slices per SM (eight rows' loads in flight per
  // thread); twice as many slices measured slower: their partial rows cost
  // more integer atomics than the extra blocks hide
  int64_t slices = (4LL * d.num_sms + col_blocks - 1) / col_blocks;
  const int64_t max_slices = (rows + 31) / 32;
  if (slices > max_slices) slices = max_slices;
  if (slices < 1) slices = 1;
  const int64_t rows_per_slice = (rows + slices - 1) / slices;
  slices = (rows + rows_per_slice - 1) / rows_per_slice;
  for (int32_t it = 0; it < max_swaps; ++it) {
    perm_best_kernel<<<best_grid, 256, 0, s>>>(w.E, c, w.tile_best, w.ctl);
    perm_apply_kernel<<<apply_blocks, 256, 0, s>>>(perm, w.S, w.V, w.E, rows, c, w.ctl, swaps_out,
                                                   gains_out);
    perm_rows_kernel<<<dim3(col_blocks, static_cast<unsigned>(slices)), 256, 0, s>>>(
        w.S, w.V, w.E, rows, c, rows_per_slice, w.ctl);
    if ((it & 255) == 255 && (e = cudaGetLastError()) != cudaSuccess) return e;
  }
  perm_finish_kernel<<<1, 32, 0, s>>>(w.ctl, n_swaps_out, shift_out);
  return cudaGetLastError();
}

cudaError_t perm_swap_gains(const Device& d, const uint16_t* W, int64_t rows, int64_t cols,
                            const int32_t* perm, void* workspace, int64_t* gains_out,
                            int32_t* info_out, int32_t* shift_out, cudaStream_t s) {
  const Workspace w = carve(workspace, rows, cols);
  cudaError_t e = prepare_table(d, W, rows, cols, perm, w, s);
  if (e != cudaSuccess) return e;
  const int nt = static_cast<int>(cols / 32);
  perm_gains_kernel<<<dim3(nt, nt), 256, 0, s>>>(w.E, static_cast<int32_t>(cols), gains_out,
                                                 w.ctl);
  perm_finish_kernel<<<1, 32, 0, s>>>(w.ctl, info_out, shift_out);
  return cudaGetLastError();
}

cudaError_t perm_shift(const Device& d, const uint16_t* W, int64_t rows, int64_t cols,
                       int32_t* shift_out, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(shift_out, 0, sizeof(int32_t), s);
  if (e != cudaSuccess) return e;
  const int64_t n8 = rows * cols / 8;
  perm_scan_kernel<<<blocks_for(n8, 256, 8LL * d.num_sms), 256, 0, s>>>(
      reinterpret_cast<const uint4*>(W), n8, nullptr, static_cast<int32_t>(cols), nullptr,
      reinterpret_cast<uint32_t*>(shift_out), nullptr);
  perm_shift_finish_kernel<<<1, 32, 0, s>>>(shift_out, rows);
  return cudaGetLastError();
}

cudaError_t perm_metric(const Device& d, const uint16_t* W, int64_t rows, int64_t cols,
                        const int32_t* perm, const int32_t* shift, uint64_t* metric_out,
                        cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(metric_out, 0, sizeof(uint64_t), s);
  if (e != cudaSuccess) return e;
  perm_metric_kernel<<<blocks_for(rows * cols / 4, 256, 8LL * d.num_sms), 256, 0, s>>>(
      W, rows, static_cast<int32_t>(cols), perm, shift,
      reinterpret_cast<unsigned long long*>(metric_out));
  return cudaGetLastError();
}

cudaError_t permute_columns(const Device& d, const uint16_t* W, int64_t rows, int64_t cols,
                            const int32_t* perm, uint16_t* W_out, cudaStream_t s) {
  const size_t row_bytes = static_cast<size_t>(cols) * 2;
  cudaError_t e = cudaFuncSetAttribute(
      permute_columns_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
      static_cast<int>(row_bytes));
  if (e != cudaSuccess) return e;
  permute_columns_kernel<<<blocks_for(rows, 1, 4LL * d.num_sms), 256, row_bytes, s>>>(
      W, rows, static_cast<int32_t>(cols), perm, W_out);
  return cudaGetLastError();
}

cudaError_t read_and_clear_perm_error(cudaStream_t s, uint32_t* value) {
  uint32_t zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(value, g_perm_error_word, sizeof(uint32_t), 0,
                                            cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return e;
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return e;
  if (*value != 0) {
    e = cudaMemcpyToSymbolAsync(g_perm_error_word, &zero, sizeof(uint32_t), 0,
                                cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(s);
  }
  return e;
}

}  // namespace maskllm
