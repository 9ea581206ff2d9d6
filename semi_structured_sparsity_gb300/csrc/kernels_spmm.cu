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
// A cluster of two CTAs (one per SM) computes a 256 x 256 tile of C with the
// pair form of the sparse MMA (tcgen05.mma.sp.cta_group::2, kind::f16: M =
// 256, 128 rows in each SM; N = 256, each SM holding 128 rows of B; K = 32 per
// instruction; the fp32 accumulator is 256 columns of each SM's tensor
// memory).  Per SM and MMA the tensor core reads 4 KB of A and 8 KB of B from
// shared memory, against 4 + 16 KB for a single-SM M = 128 tile.  K advances
// 128 per stage (four MMAs); four stages.
//   warp 0     (both CTAs) copies its own tiles per stage: two boxes of A
//              values (128 rows x 32 values, 64-byte rows, 64-byte swizzle)
//              and two of B (128 rows x 64 values, 128-byte rows, 128-byte
//              swizzle), the K-major swizzled layouts the MMA reads.
//   warp 1     allocates the pair's tensor memory (both CTAs together); in
//              rank 0 one thread waits for each stage, copies the stage's
//              metadata into tensor memory (tcgen05.cp, performed in order
//              before its later MMAs; two sets of metadata columns, and
//              before reusing a set it waits for the commit of the MMAs
//              that read it two stages earlier), issues the four MMAs and
//              commits them to the stage's "empty" barrier in both CTAs,
//              the last to "done".
//   warp 2     (rank 1) forwards "this CTA's copies landed" to rank 0.
//   warps 4-7  one tensor-memory lane per thread.  Per stage they write the
//              stage's metadata into shared memory in the order the sparse
//              MMA reads it from tensor memory: per 16-row block lane i < 8
//              holds the k 0..15 halves of rows i (low 16 bits) and i + 8
//              (high), lane 8 + i the k 16..31 halves of the same rows --
//              built from the plain row-major codes with two byte permutes.
//   warps 4-11 the epilogue: tensor memory -> registers -> shared memory
//              (32-column boxes, 128-byte swizzle) -> bulk tensor stores of
//              C, each box sent as soon as it is staged (the first half of
//              the tile's columns by warps 4-7, the rest by warps 8-11).
// The tile is bn columns wide (bn = 256, 224, ..., 128, each CTA holding bn/2
// rows of B): the host picks the width that minimises the modelled time of
// the tile waves, e.g. 224 for 4096 x 4096 (304 tiles = 4 full waves of 76
// pairs instead of 256 tiles = 3.4 waves; 94.5 against 96.6 us).
// Every wait is bounded (pipeline.cuh); on a timeout the CTA raises its own
// and its peer's abort flag and the device error word, waits (bounded) for
// copies and MMAs in flight, and the pair frees its tensor memory together.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "pipeline.cuh"

namespace maskllm {

// bit 0: a wait of the sparse product kernel gave up
__device__ uint32_t g_spmm_error_word = 0;

namespace {

// A CTA pair computes one 256 x 256 tile of C: CTA rank r of the cluster owns
// rows 128 r .. 128 r + 127 of the tile (its own A rows, its own accumulator
// lanes) and holds rows 128 r .. 128 r + 127 of the tile's 256 B rows.
// kBN is the widest tile of C; a launch takes a width bn <= kBN (a multiple
// of 32) chosen against the number of tile waves (spmm_tile_width)
constexpr int kPairM = 256, kBM = 128, kBN = 256, kBNHalf = 128;
constexpr int kBK = 128;      // dense K per stage: four K = 32 MMAs
constexpr int kHalfK = 64;    // dense K per copy box (one 128-byte row of B)
constexpr int kStages = 4;
constexpr int kThreads = 384;
constexpr uint32_t kABox = kBM * (kHalfK / 2) * 2;   // 8 KB: 128 rows x 32 values
constexpr uint32_t kBBox = kBNHalf * kHalfK * 2;     // 16 KB: up to 128 rows x 64 values
constexpr uint32_t kAStage = 2 * kABox, kBStage = 2 * kBBox;
constexpr uint32_t kARowBytes = 64, kBRowBytes = 128;
constexpr uint32_t kMetaBlock = 128 * 16;            // 16 bytes per tensor-memory lane
constexpr uint32_t kMetaStage = 2 * kMetaBlock;
constexpr int kMetaAhead = 4;                        // stages of metadata words in registers
constexpr uint32_t kTmemCols = 512;                  // D: 0..255, metadata: 256 + 128 p + 64 h
constexpr uint32_t kMetaCol0 = 256;
constexpr uint32_t kOutBox = kBM * 32 * 4;           // 16 KB: 128 rows x 32 fp32

struct SmemLayout {
  static constexpr uint32_t kA = 0;
  static constexpr uint32_t kB = kStages * kAStage;
  static constexpr uint32_t kMeta = kB + kStages * kBStage;
  static constexpr uint32_t kBar = kMeta + kStages * kMetaStage;
  // full[s], empty[s], done
  static constexpr int kNumBars = 2 * kStages + 1;
  static constexpr uint32_t kTmemSlot = kBar + kNumBars * 8;
  static constexpr uint32_t kAbort = kTmemSlot + 4;
  static constexpr uint32_t kBytes = kAbort + 4 + 1024;   // + alignment slack
};
static_assert((kBN / 32) * kOutBox <= SmemLayout::kMeta, "C staging fits in the tile stages");

// Arrivals on rank 0's full[s] per stage: its own expect-tx arrival, rank 1's
// forwarded "copies landed", and one per metadata warp of both CTAs.
constexpr uint32_t kFullArrivalsRank0 = 1 + 1 + 8;

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// Arrive on an mbarrier of any CTA of the cluster (shared::cluster address).
// Default semantics: a cluster-scope release would also wait for this
// thread's global loads still in flight (the metadata prefetch).  What the
// arrivals publish is ordered before them by fence.proxy.async (metadata in
// shared memory) or was observed complete on a barrier (copies).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int32_t x,
                                            int32_t y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int32_t x, int32_t y,
                                             uint32_t src) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(x), "r"(y), "r"(src)
      : "memory");
}

// Shared-memory matrix descriptor of a K-major tile: start address, leading
// (K-direction) and stride (8-row group) byte offsets, the fixed field value
// 1 at bit 46 and the swizzle mode in bits 61-63 (0: none, 2: 128-byte rows,
// 4: 64-byte rows).  In a swizzled tile one MMA's K extent lies inside a
// swizzle row (the leading offset is unused) and the MMA's K offset is added
// to the start address; tile bases are aligned to the swizzle pattern.  In
// the pair instructions the same descriptor addresses the same offset in both
// CTAs.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lead, uint32_t stride,
                                              uint32_t mode) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
         (static_cast<uint64_t>((lead >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((stride >> 4) & 0x3FFFu) << 32) | (1ull << 46) |
         (static_cast<uint64_t>(mode) << 61);
}
constexpr uint32_t kSwizzleNone = 0, kSwizzle128 = 2, kSwizzle64 = 4;

// Instruction descriptor: sparse (bit 2) with selector `sel`, fp32 D, bf16 A
// and B, both K-major, N = bn, M = 256 (the pair's rows).
__host__ __device__ constexpr uint32_t idesc_sparse(uint32_t sel, uint32_t bn) {
  return (sel & 3u) | (1u << 2) | (1u << 4) | (1u << 7) | (1u << 10) | ((bn >> 3) << 17) |
         ((static_cast<uint32_t>(kPairM) >> 4) << 24);
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void mma_sparse_pair(uint32_t d_tmem, uint64_t a_desc,
                                                uint64_t b_desc, uint32_t meta_tmem,
                                                uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %5, 0;\n\t"
      "tcgen05.mma.sp.cta_group::2.kind::f16 [%0], %1, %2, [%3], %4, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(meta_tmem), "r"(idesc), "r"(acc)
      : "memory");
}

// Shared memory -> tensor memory, 128 lanes x 128 bits, in both CTAs of the
// pair (each from its own shared memory into its own tensor memory).  Issued
// by the MMA thread, it is performed in order with that thread's MMAs.
__device__ __forceinline__ void tmem_copy_pair(uint32_t taddr, uint64_t s_desc) {
  asm volatile("tcgen05.cp.cta_group::2.128x128b [%0], %1;" ::"r"(taddr), "l"(s_desc) : "memory");
}

// Arrives once on the barrier at the same offset in both CTAs of the pair
// when every earlier pair operation of this thread has completed.
__device__ __forceinline__ void mma_commit_pair_both(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)),
      "h"(static_cast<uint16_t>(3))
      : "memory");
}

// Raises this CTA's and the peer's abort flags and the device error word.
__device__ __forceinline__ void raise(volatile int* abort_flag, uint32_t peer) {
  *abort_flag = 1;
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(
                   map_to_rank(smem_u32(const_cast<int*>(abort_flag)), peer)),
               "r"(1)
               : "memory");
  atomicOr(&g_spmm_error_word, 1u);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    spmm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                const __grid_constant__ CUtensorMap map_c, const uint32_t* __restrict__ meta,
                float* __restrict__ C, int32_t M, int32_t N, int32_t K, int32_t bn,
                int32_t tma_store, uint64_t wait_ns) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base (the same offset in every CTA)
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SmemLayout::kBar);
  uint64_t* full = bars;              // rank 0: the stage is ready for the pair's MMAs
                                      // rank 1: this CTA's copies of the stage landed
  uint64_t* empty = bars + kStages;   // both: the pair's MMAs are done with the stage
  uint64_t* done = empty + kStages;   // both: every MMA complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SmemLayout::kTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SmemLayout::kAbort);
  const uint32_t sA = smem_u32(smem + SmemLayout::kA);
  const uint32_t sB = smem_u32(smem + SmemLayout::kB);
  const uint32_t sMeta = smem_u32(smem + SmemLayout::kMeta);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank(), peer = rank ^ 1u;
  const int m0 = (blockIdx.x >> 1) * kPairM + static_cast<int>(rank) * kBM;   // this CTA's rows
  const int n0 = blockIdx.y * bn;
  const uint32_t b_box = static_cast<uint32_t>(bn / 2) * kHalfK * 2;   // this CTA's B rows
  const int nk = (K + kBK - 1) / kBK;
  const int kw = K / 32;   // K % 32 == 0: metadata words per row

  // copies of stage kt of this CTA's tiles: one or two 64-deep halves
  // (K % 32 == 0; a half past K reads zeros), counted on full[kt % kStages]
  auto issue_stage = [&](int kt) {
    const int s = kt % kStages;
    const int nbox = (K - kt * kBK > kHalfK) ? 2 : 1;
    const uint32_t bar = smem_u32(&full[s]);
    mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(nbox) * (kABox + b_box));
    for (int h = 0; h < nbox; ++h) {
      tma_load_2d(sA + s * kAStage + h * kABox, &map_a, kt * (kBK / 2) + h * (kHalfK / 2), m0,
                  bar);
      tma_load_2d(sB + s * kBStage + h * kBBox, &map_b, kt * kBK + h * kHalfK,
                  n0 + static_cast<int>(rank) * (bn / 2), bar);
    }
  };
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], rank == 0 ? kFullArrivalsRank0 : 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    // the pair allocates together: one warp of each CTA, the same columns
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  // both CTAs' barriers are initialised before either touches the other's
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---- copies of this CTA's tiles (each CTA's own copy engine) ----
    int issued = 0;
    if (lane == 0) {
      for (int kt = 0; kt < nk; ++kt) {
        const int s = kt % kStages;
        if (kt >= kStages &&
            !mbar_wait_bounded(&empty[s], ((kt / kStages) - 1) & 1, wait_ns, abort_flag)) {
          raise(abort_flag, peer);
          break;
        }
        issue_stage(kt);
        issued = kt + 1;
      }
      if (*abort_flag) {
        // wait (bounded) for the copies still landing in this CTA.  Rank 0's
        // stage barrier also counts arrivals from the metadata warps and
        // rank 1 that an abort may have stopped: such a wait runs to its
        // limit (up to kStages x wait_ns in all), long after the copies
        // themselves have landed.
        for (int kt = issued > kStages ? issued - kStages : 0; kt < issued; ++kt) {
          int never = 0;
          mbar_wait_bounded(&full[kt % kStages], (kt / kStages) & 1, wait_ns, &never);
        }
      }
    }
  } else if (warp == 2 && rank == 1) {
    // ---- forwards "copies landed" to rank 0's stage barrier ----
    if (lane == 0) {
      for (int kt = 0; kt < nk; ++kt) {
        const int s = kt % kStages;
        if (!mbar_wait_bounded(&full[s], (kt / kStages) & 1, wait_ns, abort_flag)) {
          raise(abort_flag, peer);
          break;
        }
        mbar_arrive_remote(map_to_rank(smem_u32(&full[s]), 0));
      }
    }
  } else if (warp == 1 && rank == 0) {
    // ---- the pair's MMAs ----
    if (lane == 0) {
      for (int kt = 0; kt < nk; ++kt) {
        const int s = kt % kStages;
        if (!mbar_wait_bounded(&full[s], (kt / kStages) & 1, wait_ns, abort_flag)) {
          raise(abort_flag, peer);
          break;
        }
        // The copy below overwrites the metadata columns that the MMAs of
        // stage kt - 2 read, and a tcgen05.cp is not ordered after earlier
        // MMAs of the same thread: wait for their commit (that stage's
        // "empty" phase), normally complete long before.
        if (kt >= 2 && !mbar_wait_bounded(&empty[(kt - 2) % kStages], ((kt - 2) / kStages) & 1,
                                          wait_ns, abort_flag)) {
          raise(abort_flag, peer);
          break;
        }
        tc_fence_after();
        // the stage's metadata into tensor memory: two 4-column blocks at
        // 64-aligned columns (K blocks 0, 1 and 2, 3), alternating by stage
        const uint32_t meta_t = tmem + kMetaCol0 + 128u * (kt & 1);
        const uint32_t ms = sMeta + s * kMetaStage;
        tmem_copy_pair(meta_t, smem_desc(ms, 2048, 128, kSwizzleNone));
        tmem_copy_pair(meta_t + 64, smem_desc(ms + kMetaBlock, 2048, 128, kSwizzleNone));
        const uint32_t a = sA + s * kAStage, b = sB + s * kBStage;
        const int nkb = min(4, kw - 4 * kt);
        for (int kb = 0; kb < nkb; ++kb) {
          // K block kb: half kb / 2, position kb % 2 in the swizzle row (16
          // compressed values = 32 bytes of A, 32 values = 64 bytes of B)
          const int h = kb >> 1, sub = kb & 1;
          const uint64_t ad =
              smem_desc(a + h * kABox + sub * 32, 0, 8 * kARowBytes, kSwizzle64);
          const uint64_t bd =
              smem_desc(b + h * kBBox + sub * 64, 0, 8 * kBRowBytes, kSwizzle128);
          mma_sparse_pair(tmem, ad, bd, meta_t + 64u * h,
                          idesc_sparse(sub, static_cast<uint32_t>(bn)), (kt | kb) != 0);
        }
        mma_commit_pair_both(&empty[s]);
      }
      // completes when every MMA issued above has (also after an abort)
      mma_commit_pair_both(done);
    }
  } else if (warp >= 4) {
    // ---- warps 4-7: metadata, then the epilogue of the tile's first
    //      columns; warps 8-11: the epilogue of the others.  Thread q of a
    //      group owns tensor-memory lane q. ----
    const int g = (warp - 4) >> 2;
    const int q = (threadIdx.x - 128) & 127;
    const int quad = warp & 3;   // lanes 32 quad .. 32 quad + 31 (== q >> 5)
    const int blk = q >> 4, i = q & 15;
    const int ra = m0 + 16 * blk + (i & 7), rb = ra + 8;
    const bool hi = i >= 8;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * quad) << 16);
    // The sparse MMA reads the metadata of a 16-row block interleaved: lane
    // i < 8 holds the k 0..15 halves of rows i (low 16 bits) and i + 8
    // (high), lane 8 + i the k 16..31 halves of the same rows.  The four
    // words of stage kt for this lane, one per K = 32 block:
    auto fetch = [&](int kt, uint32_t (&w)[4]) {
#pragma unroll
      for (int kb = 0; kb < 4; ++kb) {
        const int word = 4 * kt + kb;
        const uint32_t wa = (ra < M && word < kw) ? __ldg(meta + static_cast<int64_t>(ra) * kw + word) : 0u;
        const uint32_t wb = (rb < M && word < kw) ? __ldg(meta + static_cast<int64_t>(rb) * kw + word) : 0u;
        w[kb] = hi ? __byte_perm(wa, wb, 0x7632) : __byte_perm(wa, wb, 0x5410);
      }
    };
    uint32_t ring[kMetaAhead][4] = {};
    if (g == 0) {
#pragma unroll
      for (int u = 0; u < kMetaAhead; ++u) fetch(u, ring[u]);
    }
    const uint32_t full0 = map_to_rank(smem_u32(&full[0]), 0);
    bool ok = true;
    for (int kt0 = 0; kt0 < nk && ok && g == 0; kt0 += kMetaAhead) {
#pragma unroll
      for (int u = 0; u < kMetaAhead; ++u) {
        const int kt = kt0 + u;
        if (kt >= nk || !ok) break;
        const int s = kt % kStages;
        if (kt >= kStages) {
          ok = mbar_wait_bounded(&empty[s], ((kt / kStages) - 1) & 1, wait_ns, abort_flag);
          ok = __all_sync(0xFFFFFFFFu, ok);
          if (!ok) {
            if (lane == 0) raise(abort_flag, peer);
            break;
          }
        }
        // lane q's 16-byte rows of the stage's two metadata blocks
        uint8_t* ms = smem + SmemLayout::kMeta + s * kMetaStage + 16 * q;
        sts128(ms, make_uint4(ring[u][0], ring[u][1], 0u, 0u));
        sts128(ms + kMetaBlock, make_uint4(ring[u][2], ring[u][3], 0u, 0u));
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(full0 + 8u * s);
        fetch(kt + kMetaAhead, ring[u]);   // zeros past the end
      }
    }
    // epilogue: tensor memory -> registers -> C, 32 columns at a time
    if (ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait_bounded(done, 0, wait_ns, abort_flag));
    if (!ok && lane == 0) raise(abort_flag, peer);
    if (ok) tc_fence_after();
    const int m = m0 + q;
    float* crow = C + static_cast<int64_t>(m) * N;
    // bn / 32 boxes of 32 columns: the first half (rounded up) for group 0
    const int nb = bn / 32, nb0 = (nb + 1) / 2;
    const int cb_end = g == 0 ? nb0 : nb - nb0;
#pragma unroll 1
    for (int cb = 0; cb < cb_end; ++cb) {
      const int c = g * nb0 + cb;   // box of columns 32 c .. 32 c + 31
      if (ok) {
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
            : "r"(lane_base + static_cast<uint32_t>(32 * c)));
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        if (tma_store) {
          // staged for a bulk store: box c (128 rows x 128 bytes, 128-byte
          // swizzle: 16-byte chunk j of row q at chunk j ^ (q % 8))
          uint8_t* row = smem + c * kOutBox + 128 * q;
#pragma unroll
          for (int j = 0; j < 8; ++j)
            sts128(row + 16 * (j ^ (q & 7)),
                   make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
        } else if (m < M) {
          const int n = n0 + 32 * c;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (n + j < N) crow[n + j] = __uint_as_float(v[j]);
        }
      }
      if (tma_store) {
        fence_proxy_async_smem();
        __syncwarp();
        // every warp of the group arrives here, whatever happened above;
        // the box leaves as soon as it is staged
        if (g == 0)
          asm volatile("bar.sync 1, 128;" ::: "memory");
        else
          asm volatile("bar.sync 2, 128;" ::: "memory");
        if (q == 0 && !*abort_flag && m0 < M && n0 + 32 * c < N)
          tma_store_2d(&map_c, n0 + 32 * c, m0, smem_u32(smem + c * kOutBox));
      }
    }
    if (tma_store && q == 0) {
      // the stores have read shared memory before the CTA may leave; their
      // writes to C complete on their own
      bulk_commit();
      bulk_wait_reads();
    }
  }
  if (warp == 1 && rank == 0 && *abort_flag) {
    // every MMA issued has completed (bounded wait) before either CTA's
    // tensor memory or shared memory goes
    int never = 0;
    mbar_wait_bounded(done, 0, wait_ns, &never);
  }
  tc_fence_before();
  __syncwarp();
  // neither CTA leaves while the other may still reach its shared or tensor
  // memory
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem),
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

// 2-D tensor map over [rows, cols] row-major (bf16 or fp32) with a box of
// box_cols values (box_cols x element size = the swizzle row) x box_rows rows.
bool make_map(CUtensorMap* map, CUtensorMapDataType type, uint32_t elem_bytes, const void* base,
              int64_t rows, int64_t cols, uint32_t box_cols, uint32_t box_rows,
              CUtensorMapSwizzle swizzle) {
  const PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * elem_bytes};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t elem[2] = {1, 1};
  return fn(map, type, 2, const_cast<void*>(base), dims, strides, box, elem,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tile width of C for an M x N x K product on `sms` SMs: the width w in 256,
// 224, 192, 160, 128 with the least modelled time, waves(w) * (7.2 + K /
// 4096 * (12.6 + 0.0172 w)) microseconds per wave of CTA pairs -- fitted to
// the measured times of every width on 4096 x 4096 x 4096 and 4096 x 11008 x
// 4096 (a narrower tile saves little per wave: the per-stage waits, commits
// and copies of A do not shrink with it) -- the wider tile on a tie.
int spmm_tile_width(int64_t M, int64_t N, int64_t K, int sms) {
  const int64_t pairs = std::max<int64_t>(1, sms / 2);
  const int64_t rows = (M + kPairM - 1) / kPairM;
  int best = kBN;
  double best_t = 0.0;
  for (int w = kBN; w >= 128; w -= 32) {
    const int64_t tiles = rows * ((N + w - 1) / w);
    const int64_t waves = (tiles + pairs - 1) / pairs;
    const double t = static_cast<double>(waves) *
                     (7.2 + static_cast<double>(K) / 4096.0 * (12.6 + 0.0172 * w));
    if (w == kBN || t < best_t) {
      best = w;
      best_t = t;
    }
  }
  return best;
}

// test hook: a forced tile width, 0 = chosen per call (set and read from any
// host thread)
std::atomic<int> g_spmm_tile_n{0};

}  // namespace

void spmm_force_tile_width(int n) { g_spmm_tile_n.store(n, std::memory_order_relaxed); }

cudaError_t spmm(const Device& d, const uint16_t* values, const uint32_t* meta, int64_t M,
                 int64_t K, const uint16_t* B, int64_t N, float* C, uint64_t wait_ns,
                 cudaStream_t s) {
  const int forced = g_spmm_tile_n.load(std::memory_order_relaxed);
  const int bn = forced != 0 ? forced : spmm_tile_width(M, N, K, d.num_sms);
  CUtensorMap map_a, map_b, map_c;
  if (!make_map(&map_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, values, M, K / 2, kHalfK / 2, kBM,
                CU_TENSOR_MAP_SWIZZLE_64B) ||
      !make_map(&map_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B, N, K, kHalfK,
                static_cast<uint32_t>(bn / 2), CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  // C leaves through bulk stores when its rows are 16-byte multiples on a
  // 16-byte aligned base; otherwise each thread stores its row directly
  std::memset(&map_c, 0, sizeof(map_c));
  const bool tma_store =
      (N % 4) == 0 && (reinterpret_cast<uintptr_t>(C) % 16) == 0 &&
      make_map(&map_c, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, C, M, N, 32, kBM,
               CU_TENSOR_MAP_SWIZZLE_128B);
  const uint32_t smem = SmemLayout::kBytes;
  cudaError_t e =
      cudaFuncSetAttribute(spmm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // x: two CTAs (one cluster) per 256 rows of C; y: bn columns of C
  const dim3 grid(static_cast<unsigned>(2 * ((M + kPairM - 1) / kPairM)),
                  static_cast<unsigned>((N + bn - 1) / bn));
  spmm_kernel<<<grid, kThreads, smem, s>>>(map_a, map_b, map_c, meta, C, static_cast<int32_t>(M),
                                           static_cast<int32_t>(N), static_cast<int32_t>(K), bn,
                                           tma_store ? 1 : 0, wait_ns);
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
