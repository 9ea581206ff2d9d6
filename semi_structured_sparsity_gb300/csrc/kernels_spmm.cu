// kernels_spmm.cu -- 2:4 sparse x dense product on the fifth-generation
// tensor cores: C[M, N] = A[M, K] B[N, K]^T, fp32 out, where A is given in
// the compressed form the hard mask produces (values bf16 [M, K/2] + 4-bit
// position codes u32 [M, K/32], group k of a row at bits 4(k % 8) of word
// k / 8) and B is dense bf16 [N, K].
//
// "Accelerating Sparse Deep Neural Networks", Sec. 3.1 (two kept values of
// every group of four plus 2 bits of position per kept value) and Sec. 3.2
// (the sparse tensor core multiplies a 2:4 sparse first operand by a dense
// second operand and skips the zeros: twice the math throughput of the dense
// product).
//
// One CTA per 128 x 256 tile of C (tcgen05.mma.sp, kind::f16, cta_group::1:
// M = 128, N = 256, K = 32 per instruction; the fp32 accumulator is 256
// columns of tensor memory).  K advances 64 per pipeline stage (two MMAs);
// four stages of shared memory.
//   warp 0     TMA: per stage one box of A values (128 rows x 32 values, 64
//              bytes a row, 64-byte swizzle) and one of B (256 rows x 64
//              values, 128 bytes a row, 128-byte swizzle), the K-major
//              swizzled layouts the MMA reads (8-row groups 512 / 1024 bytes
//              apart; the MMA's K offset inside the swizzle row is added to
//              the descriptor's start address).
//   warp 1     allocates tensor memory; one thread issues the MMAs, commits
//              each stage's MMAs to the stage's "empty" barrier and the last
//              ones to "done".
//   warps 4-7  one tensor-memory lane per thread.  Per stage they write the
//              stage's metadata into tensor memory (two 32-bit columns at a
//              64-column-aligned base; the MMA's selector field picks the
//              column of its K = 32 block).  The sparse MMA reads the
//              metadata of a 16-row block interleaved: lane i < 8 holds the
//              k 0..15 halves of rows i (low 16 bits) and i + 8 (high), lane
//              8 + i the k 16..31 halves of the same rows -- built here from
//              the plain row-major codes with two byte permutes.  Then the
//              epilogue: tensor memory -> registers -> C (fp32, row-major).
// Every wait is bounded (pipeline.cuh); on a timeout the CTA raises its abort
// flag and the device error word, waits (bounded) for copies and MMAs in
// flight, frees its tensor memory and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "internal.h"
#include "pipeline.cuh"

namespace maskllm {

// bit 0: a wait of the sparse product kernel gave up
__device__ uint32_t g_spmm_error_word = 0;

namespace {

constexpr int kBM = 128, kBN = 256, kBK = 64;   // tile of C; dense K per stage
constexpr int kStages = 4;
constexpr int kThreads = 256;
constexpr uint32_t kABytes = kBM * (kBK / 2) * 2;   // 8 KB of values per stage
constexpr uint32_t kBBytes = kBN * kBK * 2;         // 32 KB of B per stage
constexpr uint32_t kARowBytes = kBK;                // 32 compressed values
constexpr uint32_t kBRowBytes = kBK * 2;            // 64 values
constexpr int kMetaAhead = 8;                       // stages of metadata loaded ahead
constexpr uint32_t kTmemCols = 512;                 // D: 0..255, metadata: 256 + 64 s
constexpr uint32_t kMetaCol0 = 256;

struct SmemLayout {
  static constexpr uint32_t kA = 0;
  static constexpr uint32_t kB = kStages * kABytes;
  static constexpr uint32_t kBar = kB + kStages * kBBytes;
  // tma_full[s], meta_full[s], empty[s], done
  static constexpr uint32_t kTmemSlot = kBar + (3 * kStages + 1) * 8;
  static constexpr uint32_t kAbort = kTmemSlot + 4;
  static constexpr uint32_t kBytes = kAbort + 4 + 1024;   // + alignment slack
};

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int32_t x,
                                            int32_t y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Shared-memory matrix descriptor of a K-major swizzled tile: start address,
// stride between 8-row groups, the fixed field value 1 at bit 46 and the
// swizzle mode in bits 61-63 (2: 128-byte rows, 4: 64-byte rows).  The
// leading byte offset is unused: one MMA's K extent lies inside a swizzle
// row.  Tile bases are aligned to the swizzle pattern (8 rows).
__device__ __forceinline__ uint64_t smem_desc_sw(uint32_t saddr, uint32_t group_stride,
                                                 uint32_t mode) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
         (static_cast<uint64_t>((group_stride >> 4) & 0x3FFFu) << 32) | (1ull << 46) |
         (static_cast<uint64_t>(mode) << 61);
}
constexpr uint32_t kSwizzle128 = 2, kSwizzle64 = 4;

// Instruction descriptor: sparse (bit 2) with selector `sel`, fp32 D, bf16 A
// and B, both K-major, N = 256, M = 128.
__host__ __device__ constexpr uint32_t idesc_sparse(uint32_t sel) {
  return (sel & 3u) | (1u << 2) | (1u << 4) | (1u << 7) | (1u << 10) |
         ((static_cast<uint32_t>(kBN) >> 3) << 17) | ((static_cast<uint32_t>(kBM) >> 4) << 24);
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void mma_sparse(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t meta_tmem, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %5, 0;\n\t"
      "tcgen05.mma.sp.cta_group::1.kind::f16 [%0], %1, %2, [%3], %4, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(meta_tmem), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void raise(volatile int* abort_flag) {
  *abort_flag = 1;
  atomicOr(&g_spmm_error_word, 1u);
}

__global__ void __launch_bounds__(kThreads, 1)
    spmm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                const uint32_t* __restrict__ meta, float* __restrict__ C, int32_t M, int32_t N,
                int32_t K, uint64_t wait_ns) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SmemLayout::kBar);
  uint64_t* tma_full = bars;
  uint64_t* meta_full = bars + kStages;
  uint64_t* empty = bars + 2 * kStages;
  uint64_t* done = bars + 3 * kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SmemLayout::kTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SmemLayout::kAbort);
  const uint32_t sA = smem_u32(smem + SmemLayout::kA);
  const uint32_t sB = smem_u32(smem + SmemLayout::kB);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.y * kBM, n0 = blockIdx.x * kBN;
  const int nk = (K + kBK - 1) / kBK;   // K % 32 == 0; a half stage reads zeros
  const int kw = K / 32;                // metadata words per row

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&tma_full[s], 1);
      mbar_init(&meta_full[s], 4);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---- TMA producer ----
    int issued = 0;
    if (lane == 0) {
      for (int kt = 0; kt < nk; ++kt) {
        const int s = kt % kStages;
        if (kt >= kStages &&
            !mbar_wait_bounded(&empty[s], ((kt / kStages) - 1) & 1, wait_ns, abort_flag)) {
          raise(abort_flag);
          break;
        }
        mbar_arrive_expect_tx(&tma_full[s], kABytes + kBBytes);
        tma_load_2d(sA + s * kABytes, &map_a, kt * (kBK / 2), m0, &tma_full[s]);
        tma_load_2d(sB + s * kBBytes, &map_b, kt * kBK, n0, &tma_full[s]);
        issued = kt + 1;
      }
      if (*abort_flag) {
        // wait (bounded) for the copies still landing in shared memory
        for (int kt = issued > kStages ? issued - kStages : 0; kt < issued; ++kt) {
          int never = 0;
          mbar_wait_bounded(&tma_full[kt % kStages], (kt / kStages) & 1, wait_ns, &never);
        }
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer ----
    if (lane == 0) {
      for (int kt = 0; kt < nk; ++kt) {
        const int s = kt % kStages;
        const uint32_t ph = (kt / kStages) & 1;
        if (!mbar_wait_bounded(&tma_full[s], ph, wait_ns, abort_flag) ||
            !mbar_wait_bounded(&meta_full[s], ph, wait_ns, abort_flag)) {
          raise(abort_flag);
          break;
        }
        tc_fence_after();
        const uint32_t a = sA + s * kABytes, b = sB + s * kBBytes;
        const uint32_t meta_t = tmem + kMetaCol0 + 64u * s;
        // the second K = 32 block of the last stage is absent when K % 64 == 32
        const int nkb = (2 * kt + 1 < kw) ? 2 : 1;
        for (int kb = 0; kb < nkb; ++kb) {
          // K block kb: 16 compressed values (32 bytes) of A, 32 values (64
          // bytes) of B into the swizzle row
          const uint64_t ad = smem_desc_sw(a + kb * 32, 8 * kARowBytes, kSwizzle64);
          const uint64_t bd = smem_desc_sw(b + kb * 64, 8 * kBRowBytes, kSwizzle128);
          mma_sparse(tmem, ad, bd, meta_t, idesc_sparse(kb), (kt | kb) != 0);
        }
        mma_commit(&empty[s]);
      }
      // completes when every MMA issued above has (also after an abort)
      mma_commit(done);
    }
  } else if (warp >= 4) {
    // ---- metadata, then epilogue; thread q owns tensor-memory lane q ----
    const int q = threadIdx.x - 128;
    const int quad = warp & 3;   // lanes 32 quad .. 32 quad + 31 (== q >> 5)
    const int blk = q >> 4, i = q & 15;
    const int ra = m0 + 16 * blk + (i & 7), rb = ra + 8;
    const bool hi = i >= 8;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * quad) << 16);
    // the two words of stage kt for this lane: low 16 bits from row ra, high
    // 16 bits from row rb, the k 0..15 or k 16..31 halves
    auto fetch = [&](int kt, uint32_t (&w)[2]) {
#pragma unroll
      for (int kb = 0; kb < 2; ++kb) {
        const int word = 2 * kt + kb;
        const uint32_t wa = (ra < M && word < kw) ? __ldg(meta + static_cast<int64_t>(ra) * kw + word) : 0u;
        const uint32_t wb = (rb < M && word < kw) ? __ldg(meta + static_cast<int64_t>(rb) * kw + word) : 0u;
        w[kb] = hi ? __byte_perm(wa, wb, 0x7632) : __byte_perm(wa, wb, 0x5410);
      }
    };
    uint32_t ring[kMetaAhead][2];
#pragma unroll
    for (int u = 0; u < kMetaAhead; ++u) fetch(u, ring[u]);
    bool ok = true;
    for (int kt0 = 0; kt0 < nk && ok; kt0 += kMetaAhead) {
#pragma unroll
      for (int u = 0; u < kMetaAhead; ++u) {
        const int kt = kt0 + u;
        if (kt >= nk || !ok) break;
        const int s = kt % kStages;
        if (kt >= kStages) {
          ok = mbar_wait_bounded(&empty[s], ((kt / kStages) - 1) & 1, wait_ns, abort_flag);
          ok = __all_sync(0xFFFFFFFFu, ok);
          if (!ok) {
            if (lane == 0) raise(abort_flag);
            break;
          }
          tc_fence_after();
        }
        asm volatile("tcgen05.st.sync.aligned.32x32b.x2.b32 [%0], {%1, %2};" ::"r"(
                         lane_base + kMetaCol0 + 64u * s),
                     "r"(ring[u][0]), "r"(ring[u][1])
                     : "memory");
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&meta_full[s]);
        fetch(kt + kMetaAhead, ring[u]);   // zeros past the end
      }
    }
    // epilogue
    if (ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait_bounded(done, 0, wait_ns, abort_flag));
    if (!ok && lane == 0) raise(abort_flag);
    if (ok) {
      tc_fence_after();
      const int m = m0 + q;
      float* crow = C + static_cast<int64_t>(m) * N;
      const bool vec = (N % 4) == 0;
#pragma unroll 1
      for (int c0 = 0; c0 < kBN; c0 += 32) {
        uint32_t v[32];
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
            "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
            : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
              "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
              "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]),
              "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
              "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]),
              "=r"(v[31])
            : "r"(lane_base + static_cast<uint32_t>(c0)));
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        if (m < M) {
          const int n = n0 + c0;
          if (vec && n + 32 <= N) {
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              __stcs(reinterpret_cast<float4*>(crow + n + j),
                     make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]),
                                 __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3])));
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (n + j < N) crow[n + j] = __uint_as_float(v[j]);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    // every MMA issued has completed (bounded wait) before the memory goes
    if (*abort_flag) {
      int never = 0;
      mbar_wait_bounded(done, 0, wait_ns, &never);
    }
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

// ---- host side ----------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D bf16 tensor map over [rows, cols] row-major with a box of box_cols
// values (box_cols * 2 bytes = the swizzle row) x box_rows rows.
bool make_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, uint32_t box_cols,
              uint32_t box_rows, CUtensorMapSwizzle swizzle) {
  const PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t elem[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            elem, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t spmm(const Device&, const uint16_t* values, const uint32_t* meta, int64_t M, int64_t K,
                 const uint16_t* B, int64_t N, float* C, uint64_t wait_ns, cudaStream_t s) {
  CUtensorMap map_a, map_b;
  if (!make_map(&map_a, values, M, K / 2, kBK / 2, kBM, CU_TENSOR_MAP_SWIZZLE_64B) ||
      !make_map(&map_b, B, N, K, kBK, kBN, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const uint32_t smem = SmemLayout::kBytes;
  cudaError_t e =
      cudaFuncSetAttribute(spmm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>((N + kBN - 1) / kBN), static_cast<unsigned>((M + kBM - 1) / kBM));
  spmm_kernel<<<grid, kThreads, smem, s>>>(map_a, map_b, meta, C, static_cast<int32_t>(M),
                                           static_cast<int32_t>(N), static_cast<int32_t>(K),
                                           wait_ns);
  return cudaGetLastError();
}

cudaError_t read_and_clear_spmm_error(cudaStream_t s, uint32_t* value) {
  uint32_t zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(value, g_spmm_error_word, sizeof(uint32_t), 0,
                                            cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return e;
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return e;
  if (*value != 0) {
    e = cudaMemcpyToSymbolAsync(g_spmm_error_word, &zero, sizeof(uint32_t), 0,
                                cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(s);
  }
  return e;
}

}  // namespace maskllm
