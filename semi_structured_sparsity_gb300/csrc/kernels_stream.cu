// kernels_stream.cu -- the four hot-path kernels as persistent, bulk-copy
// pipelined streams over a batch of matrices.
//
// "MaskLLM: Learnable Semi-Structured Sparsity for Large Language Models",
// Fig. 3 (Gumbel-softmax draw over the 2:4 candidates of every group of four,
// weighted average of the candidate masks, all differentiable), Fig. 5
// (kappa), Table 2 (prior masks), Table 3 (weight regularisation);
// "Accelerating Sparse Deep Neural Networks", Sec. 3.1 (compressed 2:4
// storage) and Sec. 4.1 (magnitude pruning).
//
// Structure (one CTA per SM: 1 producer warp + 16 consumer warps):
//   * Work is a list of chunks.  A chunk is up to 1024 consecutive groups of
//     one row, or several whole short rows (<= 1024 groups).  The chunks of a
//     launch are those of up to 16 matrices, concatenated; CTA b takes a
//     contiguous range of them, cut at row boundaries, so every row is
//     finished inside one CTA (its sum of squares needs no cross-CTA step)
//     and the CTAs carry equal byte counts to within one row.
//   * The producer warp copies each chunk's inputs (W: 8 bytes per group,
//     logits: 24, upstream gradient: 8) from global into a ring of shared
//     stages (4 stages of 32-40 KB) with bulk copies completing on the stage's
//     "full" mbarrier.  (Deeper rings, 5-6 stages where shared memory allows,
//     measured no faster.)
//   * Consumer thread t owns groups 2t and 2t+1 of every chunk: it reads them
//     from shared memory, computes, and either stores its results straight to
//     global memory (16-byte coalesced stores) or writes them back into the
//     stage, from where the producer bulk-stores the whole chunk.  Each
//     consumer warp then arrives on the stage's "empty" mbarrier.
//   * After a stage's empty barrier completes, the producer finishes that
//     chunk: it sums the per-thread row partials (left in the threads' W
//     slots) in a fixed order (forward) and issues the bulk store of staged
//     outputs, then refills the stage.
//   * Every wait is bounded (pipeline.cuh).  On a timeout the CTA raises an
//     abort flag, sets the device error word, the producer waits (bounded)
//     for its copies still in flight, and all warps return.
#include <atomic>
#include <cstddef>

#include "device_common.cuh"
#include "internal.h"
#include "pipeline.cuh"

namespace maskllm {

__device__ __align__(16) float g_gumbel_table_s[kTableSize] = {
#include "gumbel_table.inc"
};

// Bit 0: a consumer's wait for a stage's copies timed out; bit 1: the
// producer's wait for a stage's release timed out; bit 2: the final drain of
// in-flight copies timed out.
__device__ uint32_t g_stream_error_word = 0;

namespace {

constexpr int kChunkGroups = 1024;           // groups per chunk
constexpr int kMaxMats = kMaxBatch;

struct MatDesc {
  const void* W;          // bf16 [rows, cols]
  const void* L;          // fp32 [rows, cols/4, 6]
  const void* G;          // bf16 [rows, cols] (backward)
  void* out0;             // prior: logits; forward: W'; backward: dlogits; compress: values
  void* out1;             // forward: row_sq; compress: codes
  void* out2;             // forward: probs; compress: idx; forward + stats: draws
  void* out3;             // forward + stats: L1 per row
  void* out4;             // forward + stats: max-probability sum per row
  int64_t rows;           // rows; flat chunking: chunks
  int64_t unit_begin;     // first unit of this matrix in the launch's unit list
  int64_t chunk_begin;    // first chunk of this matrix in the launch's chunk list
  int32_t gpr;            // groups per row (cols / 4)
  int32_t cpr;            // chunks per row when a row spans >= 1 chunk, else 0
  int32_t rpc;            // rows per chunk when rows are short, else 0; flat
                          // chunking: the groups of the last chunk
  uint32_t tensor_id;
};

struct Scalars {
  float kappa;
  float rho;
  float dz_dlogit;
  float two_reg;
  float scale;
  uint32_t step;
  RoundKeys keys;
};

struct StreamParams {
  MatDesc mats[kMaxMats];
  int32_t nmats;
  int64_t total_units;
  int64_t total_chunks;
  uint64_t wait_ns;        // bound of every pipeline wait
  uint64_t drain_ns;       // bound of the final wait for copies in flight
  int32_t withhold_loads;  // test hook: no copies are issued
  Scalars s;
  int32_t flat;            // the matrices are chunked flat (must equal Op::kFlat)
  // the backward with diagnostics: each matrix's previous draws (u8 per
  // group, nullable)
  const void* prev[kMaxMats];
};

// Where the Philox round keys sit in the parameter block matters: with the
// keys on an 8-byte boundary the forward measured 2% slower (376 -> 384 us
// on the LLaMA-2-7B block) and the fused diagnostics 3% slower, the same
// code otherwise.  New fields go after `s`.
static_assert(offsetof(StreamParams, s) % 8 == 4 && offsetof(Scalars, keys) % 8 == 0,
              "round keys at 4 mod 8 in the parameter block");

struct Chunk {
  int32_t mat;
  int32_t ng;       // groups in the chunk
  int64_t g0;       // first group, matrix-local
  int64_t row0;     // first row
  int32_t nrows;    // whole rows ending in this chunk (0 when a long row continues)
  int32_t obuf;     // staged outputs: which of the stage's output buffers
};

__device__ __forceinline__ int64_t units_of(const MatDesc& d) {
  return d.cpr > 0 ? d.rows : (d.rows + d.rpc - 1) / d.rpc;
}

// Walks the chunks of units [u, u_end) of the launch's unit list.  kFlat:
// the matrices are chunked flat (describe()), so a matrix's last chunk may
// be ragged.
template <bool kFlat>
struct ChunkIter {
  const StreamParams* p;
  int32_t m;
  int64_t lu;       // unit within matrix m
  int32_t j;        // chunk within the unit (long rows)
  int64_t left;     // units left

  __device__ void init(const StreamParams* pp, int64_t u, int64_t u_end) {
    p = pp;
    left = u_end - u;
    m = 0;
    while (m + 1 < p->nmats && p->mats[m + 1].unit_begin <= u) ++m;
    lu = u - p->mats[m].unit_begin;
    j = 0;
  }

  __device__ bool next(Chunk& c) {
    if (left <= 0) return false;
    const MatDesc& d = p->mats[m];
    c.mat = m;
    if (d.cpr > 0) {
      c.row0 = lu;
      c.g0 = lu * d.gpr + static_cast<int64_t>(j) * kChunkGroups;
      if constexpr (kFlat) {
        c.ng = lu + 1 == d.rows ? d.rpc : kChunkGroups;   // a ragged last chunk
      } else {
        const int64_t rest = d.gpr - static_cast<int64_t>(j) * kChunkGroups;   // of the row
        c.ng = static_cast<int32_t>(rest < kChunkGroups ? rest : kChunkGroups);
      }
      const bool last = (j + 1 == d.cpr);
      c.nrows = last ? 1 : 0;
      if (last) {
        j = 0;
        ++lu;
        --left;
      } else {
        ++j;
      }
    } else {
      c.row0 = lu * d.rpc;
      const int64_t r_rest = d.rows - c.row0;
      c.nrows = static_cast<int32_t>(r_rest < d.rpc ? r_rest : d.rpc);
      c.g0 = c.row0 * d.gpr;
      c.ng = c.nrows * d.gpr;
      ++lu;
      --left;
    }
    if (lu >= units_of(d) && left > 0) {
      ++m;
      lu = 0;
      j = 0;
    }
    return true;
  }
};

// First unit of CTA b: the unit boundary at or after chunk total*b/G.
__device__ int64_t cta_first_unit(const StreamParams& p, int64_t b, int64_t G) {
  if (b >= G) return p.total_units;
  const int64_t target = p.total_chunks * b / G;   // total_chunks < 2^44, b < 2^16
  int m = 0;
  while (m + 1 < p.nmats && p.mats[m + 1].chunk_begin <= target) ++m;
  const MatDesc& d = p.mats[m];
  const int64_t t = target - d.chunk_begin;
  const int64_t per_unit = d.cpr > 0 ? d.cpr : 1;
  int64_t u = (t + per_unit - 1) / per_unit;
  const int64_t nu = units_of(d);
  if (u > nu) u = nu;
  return d.unit_begin + u;
}

// The launch's chunk index of the first chunk of unit u (u may be the total).
__device__ int64_t chunk_index(const StreamParams& p, int64_t u) {
  int m = 0;
  while (m + 1 < p.nmats && p.mats[m + 1].unit_begin <= u) ++m;
  const MatDesc& d = p.mats[m];
  return d.chunk_begin + (u - d.unit_begin) * (d.cpr > 0 ? d.cpr : 1);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

__device__ __forceinline__ void raise_abort(volatile int* abort_flag, uint32_t bit) {
  *abort_flag = 1;
  atomicOr(&g_stream_error_word, bit);
}

// ---------------------------------------------------------------------------
// Fragments: consumer thread t of a GPT-groups-per-thread kernel owns groups
// GPT*t .. GPT*t + GPT - 1 of every chunk (8 bytes of W and 24 bytes of
// logits per group, contiguous in the stage).
// ---------------------------------------------------------------------------

template <int GPT>
__device__ __forceinline__ void load_w(const uint8_t* base, int t, uint32_t w[2 * GPT]) {
  if constexpr (GPT == 2) {
    const uint4 v = *reinterpret_cast<const uint4*>(base + 16 * t);
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  } else {
    const uint2 v = *reinterpret_cast<const uint2*>(base + 8 * t);
    w[0] = v.x; w[1] = v.y;
  }
}

template <int GPT>
__device__ __forceinline__ void load_l(const uint8_t* base, int t, float L[6 * GPT]) {
  if constexpr (GPT == 2) {
    const float4* q = reinterpret_cast<const float4*>(base + 48 * t);
    const float4 a = q[0], b = q[1], c = q[2];
    L[0] = a.x; L[1] = a.y; L[2] = a.z; L[3] = a.w; L[4] = b.x; L[5] = b.y;
    L[6] = b.z; L[7] = b.w; L[8] = c.x; L[9] = c.y; L[10] = c.z; L[11] = c.w;
  } else {
    const float2* q = reinterpret_cast<const float2*>(base + 24 * t);
    const float2 a = q[0], b = q[1], c = q[2];
    L[0] = a.x; L[1] = a.y; L[2] = b.x; L[3] = b.y; L[4] = c.x; L[5] = c.y;
  }
}

// 24*GPT bytes (GPT groups of six fp32 values) to shared or global memory.
template <int GPT>
__device__ __forceinline__ void store_l(void* base_bytes, int64_t t, const float L[6 * GPT]) {
  if constexpr (GPT == 2) {
    float4* q = reinterpret_cast<float4*>(static_cast<uint8_t*>(base_bytes) + 48 * t);
    q[0] = make_float4(L[0], L[1], L[2], L[3]);
    q[1] = make_float4(L[4], L[5], L[6], L[7]);
    q[2] = make_float4(L[8], L[9], L[10], L[11]);
  } else {
    float2* q = reinterpret_cast<float2*>(static_cast<uint8_t*>(base_bytes) + 24 * t);
    q[0] = make_float2(L[0], L[1]);
    q[1] = make_float2(L[2], L[3]);
    q[2] = make_float2(L[4], L[5]);
  }
}

// 8*GPT bytes of bf16 W' words to global memory, streaming.
template <int GPT>
__device__ __forceinline__ void store_w_global(void* out, int64_t t, const uint32_t o[2 * GPT]) {
  if constexpr (GPT == 2)
    __stcs(static_cast<uint4*>(out) + t, make_uint4(o[0], o[1], o[2], o[3]));
  else
    __stcs(static_cast<uint2*>(out) + t, make_uint2(o[0], o[1]));
}

// ---------------------------------------------------------------------------
// Per-op policies (GPT = groups per consumer thread).
//   kTable      the Gumbel table is loaded into shared memory
//   kRowQuantities  per-row sums the consumers leave as per-thread partials
//               (at kPartOffset + t * kPartStride + 4 q of the stage) for the
//               producer to reduce and hand to write_row()
//   kStaged     consumers write the chunk's output into the stage; the
//               producer bulk-stores it (kOutBytesPerGroup bytes per group
//               from stage offset kOutOffset to out0)
//   kWarpWide   consume() is called by every lane, active or not
// ---------------------------------------------------------------------------

template <int GPT_, int kStages_>
struct OpBase {
  static constexpr int kGPT = GPT_;
  static constexpr int kConsumers = kChunkGroups / GPT_;
  static constexpr int kConsumerWarps = kConsumers / 32;
  static constexpr int kThreads = kConsumers + 32;   // + the producer warp
  static constexpr int kStages = kStages_;
  // per-row sums: none by default (see FwdOp, StatsOp)
  static constexpr int kRowQuantities = 0;
  static constexpr uint32_t kPartOffset = 0;
  static constexpr uint32_t kPartStride = 0;
  __device__ static bool want_row(const MatDesc&, int) { return false; }
  __device__ static void write_row(const MatDesc&, int64_t, int, float) {}
  // the refill of a stage touches nothing the retirement of its previous
  // chunk reads (partials): the producer issues the copies first and retires
  // the old chunk while they are in flight.  Not for staged outputs: a bulk
  // store queued behind the refill's copies leaves the stage later (the
  // prior measured 17% slower that way).
  static constexpr bool kRefillFirst = false;
  // long rows: each consumer warp leaves one partial (the sum of its lanes')
  // in its lane 0's slot and the producer adds kConsumerWarps values; else
  // every thread leaves its own partial and the producer adds kConsumers
  static constexpr bool kWarpRowSums = false;
  static constexpr int kIntQuantity = -1;   // row quantity summed as an integer (none)
  // chunk the matrices flat (no per-row sums: prior, backward, compress)
  static constexpr bool kFlat = false;
  // staged outputs: buffers per stage (chunk n of a stage's ring writes
  // buffer (n / kStages) % kOutBuffers), kOutBufBytes apart
  static constexpr int kOutBuffers = 1;
  static constexpr uint32_t kOutBufBytes = 0;
  // > 0: the producer sleeps this long between tests of a stage's "empty"
  // barrier instead of polling with the suspend hint
  static constexpr uint32_t kProducerNapNs = 0;
};

template <int GPT>
struct PriorOp : OpBase<GPT, 4> {
  static constexpr bool kFlat = true;
  static constexpr bool kTable = false, kStaged = true, kWarpWide = false;
  static constexpr bool kOutOverlapsInput = false;   // W in, logits out: separate regions
  // two output buffers per stage: the consumers write one while the bulk
  // store of the stage's previous chunk still reads the other (there is no
  // Gumbel table, so the shared memory holds them)
  static constexpr int kOutBuffers = 2;
  static constexpr uint32_t kOutBufBytes = kChunkGroups * 24;
  static constexpr uint32_t kOutOffset = kChunkGroups * 8;
  static constexpr uint32_t kStageBytes = kOutOffset + kOutBuffers * kOutBufBytes;
  static constexpr uint32_t kOutBytesPerGroup = 24;

  __device__ static void issue(const MatDesc& d, const Chunk& c, uint8_t* st, uint64_t* bar) {
    const uint32_t wb = static_cast<uint32_t>(c.ng) * 8;
    mbar_expect_tx(bar, wb);
    bulk_load(st, static_cast<const uint8_t*>(d.W) + c.g0 * 8, wb, bar);
  }

  __device__ static void consume(const StreamParams& p, const MatDesc&, const Chunk& c,
                                 uint8_t* st, int t, const float*, float*) {
    uint32_t w[2 * GPT];
    load_w<GPT>(st, t, w);
    float out[6 * GPT];
    const float s = p.s.scale;
#pragma unroll
    for (int g = 0; g < GPT; ++g) {
      const float a0 = fabsf(bf16_lo(w[2 * g])), a1 = fabsf(bf16_hi(w[2 * g]));
      const float a2 = fabsf(bf16_lo(w[2 * g + 1])), a3 = fabsf(bf16_hi(w[2 * g + 1]));
      float* o = out + 6 * g;
      o[0] = __fmul_rn(s, __fadd_rn(a0, a1));
      o[1] = __fmul_rn(s, __fadd_rn(a0, a2));
      o[2] = __fmul_rn(s, __fadd_rn(a0, a3));
      o[3] = __fmul_rn(s, __fadd_rn(a1, a2));
      o[4] = __fmul_rn(s, __fadd_rn(a1, a3));
      o[5] = __fmul_rn(s, __fadd_rn(a2, a3));
    }
    store_l<GPT>(st + kOutOffset + c.obuf * kOutBufBytes, t, out);
  }
};

template <bool kProbs, int GPT>
struct FwdOp : OpBase<GPT, 4> {
  static constexpr bool kTable = true, kStaged = false, kWarpWide = false;
  static constexpr bool kOutOverlapsInput = false;
  static constexpr bool kRefillFirst = true;
  // forward 393.8 -> 380.8 us; the diagnostics measured slower with it
  static constexpr bool kWarpRowSums = true;
  // row sum of squares; each thread's partial in a region of its own after
  // the logits, so the refill can land while the producer reduces them
  static constexpr int kRowQuantities = 1;
  static constexpr uint32_t kPartOffset = kChunkGroups * (8 + 24);
  static constexpr uint32_t kPartStride = 4;
  __device__ static bool want_row(const MatDesc& d, int) { return d.out1 != nullptr; }
  __device__ static void write_row(const MatDesc& d, int64_t row, int, float v) {
    static_cast<float*>(d.out1)[row] = v;
  }
  static constexpr uint32_t kStageBytes = kPartOffset + (kChunkGroups / GPT) * kPartStride;
  static constexpr uint32_t kOutOffset = 0;
  static constexpr uint32_t kOutBytesPerGroup = 0;

  __device__ static void issue(const MatDesc& d, const Chunk& c, uint8_t* st, uint64_t* bar) {
    const uint32_t wb = static_cast<uint32_t>(c.ng) * 8, lb = static_cast<uint32_t>(c.ng) * 24;
    mbar_expect_tx(bar, wb + lb);
    bulk_load(st, static_cast<const uint8_t*>(d.W) + c.g0 * 8, wb, bar);
    bulk_load(st + kChunkGroups * 8, static_cast<const uint8_t*>(d.L) + c.g0 * 24, lb, bar);
  }

  __device__ static void group(const StreamParams& p, const float* tab, uint64_t gidx,
                               uint32_t tensor_id, const float L[kCand], uint32_t w01,
                               uint32_t w23, uint32_t& o01, uint32_t& o23, float& acc,
                               float prob[kCand]) {
    float g[kCand], e[kCand], inv, num[4], M[4];
    gumbel6(group_words(gidx, p.s.step, tensor_id, p.s.keys), tab, g);
    softmax6(L, g, p.s.kappa, p.s.rho, e, inv, num);
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
      for (int c = 0; c < kCand; ++c) prob[c] = e[c] * inv;
    }
  }

  __device__ static void consume(const StreamParams& p, const MatDesc& d, const Chunk& c,
                                 uint8_t* st, int t, const float* tab, float* acc) {
    uint32_t w[2 * GPT], o[2 * GPT];
    float L[6 * GPT], pr[6 * GPT];
    load_w<GPT>(st, t, w);
    load_l<GPT>(st + kChunkGroups * 8, t, L);
    const uint64_t g0 = static_cast<uint64_t>(c.g0) + static_cast<uint64_t>(GPT * t);
#pragma unroll
    for (int g = 0; g < GPT; ++g)
      group(p, tab, g0 + g, d.tensor_id, L + 6 * g, w[2 * g], w[2 * g + 1], o[2 * g],
            o[2 * g + 1], acc[0], pr + 6 * g);
    const int64_t unit = c.g0 / GPT + t;   // this thread's GPT-group unit
    store_w_global<GPT>(d.out0, unit, o);
    if (kProbs && d.out2 != nullptr) store_l<GPT>(d.out2, unit, pr);
  }
};

template <bool kReg, int GPT>
struct BwdOp : OpBase<GPT, 4> {
  static constexpr bool kFlat = true;
  static constexpr bool kTable = true, kStaged = true, kWarpWide = false;
  static constexpr bool kOutOverlapsInput = true;    // dlogits overwrite the logits
  // 482 -> 476 us on the LLaMA-2-7B block; the forward, prior, compress and
  // diagnostics measured 0.3-2% slower with a napping producer
  static constexpr uint32_t kProducerNapNs = 64;
  static constexpr uint32_t kStageBytes = kChunkGroups * (8 + 8 + 24);
  static constexpr uint32_t kOutOffset = kChunkGroups * 16;
  static constexpr uint32_t kOutBytesPerGroup = 24;

  __device__ static void issue(const MatDesc& d, const Chunk& c, uint8_t* st, uint64_t* bar) {
    const uint32_t wb = static_cast<uint32_t>(c.ng) * 8, lb = static_cast<uint32_t>(c.ng) * 24;
    mbar_expect_tx(bar, 2 * wb + lb);
    bulk_load(st, static_cast<const uint8_t*>(d.W) + c.g0 * 8, wb, bar);
    bulk_load(st + kChunkGroups * 8, static_cast<const uint8_t*>(d.G) + c.g0 * 8, wb, bar);
    bulk_load(st + kChunkGroups * 16, static_cast<const uint8_t*>(d.L) + c.g0 * 24, lb, bar);
  }

  // dlogits of one group; also leaves the scaled and the noisy logits
  // fl32(kappa L) and z in y and z (for the diagnostics)
  __device__ static void group(const StreamParams& p, const float* tab, uint64_t gidx,
                               uint32_t tensor_id, const float L[kCand], uint32_t w01,
                               uint32_t w23, uint32_t g01, uint32_t g23, float out[kCand],
                               float y[kCand], float z[kCand]) {
    float g[kCand], e[kCand], inv, num[4];
    gumbel6(group_words(gidx, p.s.step, tensor_id, p.s.keys), tab, g);
    noisy_logits6(L, g, p.s.kappa, p.s.rho, y, z);
    softmax6_of_z(z, e, inv, num);
    const float w[4] = {bf16_lo(w01), bf16_hi(w01), bf16_lo(w23), bf16_hi(w23)};
    float t[4] = {bf16_lo(g01), bf16_hi(g01), bf16_lo(g23), bf16_hi(g23)};
    if (kReg) {
      float M[4];
      soft_mask4(num, inv, M);
#pragma unroll
      for (int j = 0; j < 4; ++j) t[j] = __fmaf_rn(p.s.two_reg, __fmul_rn(w[j], M[j]), t[j]);
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
    for (int c = 0; c < kCand; ++c) out[c] = (p.s.dz_dlogit * pr[c]) * (dp[c] - r);
  }

  __device__ static void consume(const StreamParams& p, const MatDesc& d, const Chunk& c,
                                 uint8_t* st, int t, const float* tab, float*) {
    uint32_t w[2 * GPT], gr[2 * GPT];
    float L[6 * GPT], dl[6 * GPT];
    load_w<GPT>(st, t, w);
    load_w<GPT>(st + kChunkGroups * 8, t, gr);
    load_l<GPT>(st + kChunkGroups * 16, t, L);
    const uint64_t g0 = static_cast<uint64_t>(c.g0) + static_cast<uint64_t>(GPT * t);
#pragma unroll
    for (int g = 0; g < GPT; ++g) {
      float y[kCand], z[kCand];
      group(p, tab, g0 + g, d.tensor_id, L + 6 * g, w[2 * g], w[2 * g + 1], gr[2 * g],
            gr[2 * g + 1], dl + 6 * g, y, z);
    }
    store_l<GPT>(st + kChunkGroups * 16, t, dl);   // dlogits over this thread's own logits
  }
};

// Candidate c's metadata code i | j << 2 (one nibble per candidate) and the
// byte selector that gathers its kept pair (i, j) out of the group's 8 bytes
// (16 bits per candidate; byte k of the result takes source byte nibble k):
// c0 (0,1) c1 (0,2) c2 (0,3) c3 (1,2) c4 (1,3) c5 (2,3).
constexpr uint32_t kCode = 0xED9C84u;
constexpr uint64_t kGather03 = 0x5432761054103210ull;   // c0 .. c3
constexpr uint32_t kGather45 = 0x76547632u;             // c4, c5

// Hard-mask candidate: the first maximum of the raw logits.  fmaxf ignores a
// NaN operand, so m is the largest non-NaN logit (NaN only if all six are);
// the first c with L_c == m is the lowest index among the maxima (-0 == +0);
// when every logit is NaN no comparison holds and candidate 0 is chosen.
__device__ __forceinline__ int first_argmax6(const float L[kCand]) {
  const float m = fmaxf(fmaxf(fmaxf(L[0], L[1]), fmaxf(L[2], L[3])), fmaxf(L[4], L[5]));
  uint32_t hit = 0;
#pragma unroll
  for (int c = 0; c < kCand; ++c) hit |= static_cast<uint32_t>(L[c] == m) << c;
  return hit ? __ffs(hit) - 1 : 0;
}

__device__ __forceinline__ uint32_t gather_selector(int c) {
  return c < 4 ? static_cast<uint32_t>(kGather03 >> (16 * c)) & 0xFFFFu
               : (kGather45 >> (16 * (c - 4))) & 0xFFFFu;
}

template <int GPT>
struct CompressOp : OpBase<GPT, 4> {
  static constexpr bool kFlat = true;
  static constexpr bool kTable = false, kStaged = false, kWarpWide = true;
  static constexpr bool kOutOverlapsInput = false;
  static constexpr uint32_t kStageBytes = kChunkGroups * (8 + 24);
  static constexpr uint32_t kOutOffset = 0;
  static constexpr uint32_t kOutBytesPerGroup = 0;

  __device__ static void issue(const MatDesc& d, const Chunk& c, uint8_t* st, uint64_t* bar) {
    FwdOp<false, GPT>::issue(d, c, st, bar);
  }

  __device__ static void consume(const StreamParams&, const MatDesc& k, const Chunk& c,
                                 uint8_t* st, int t, const float*, float*) {
    // Every lane comes here.  Chunks hold a multiple of 8 groups, so the
    // 8/GPT lanes that share one 32-bit code word are all active or all not.
    constexpr int kLanesPerWord = 8 / GPT;
    const int64_t unit = c.g0 / GPT + t;
    const bool active = GPT * t < c.ng;
    uint32_t codes = 0;
    if (active) {
      uint32_t w[2 * GPT], v[GPT], cand[GPT];
      float L[6 * GPT];
      load_w<GPT>(st, t, w);
      load_l<GPT>(st + kChunkGroups * 8, t, L);
#pragma unroll
      for (int g = 0; g < GPT; ++g) {
        const int c = first_argmax6(L + 6 * g);
        v[g] = __byte_perm(w[2 * g], w[2 * g + 1], gather_selector(c));
        codes |= ((kCode >> (4 * c)) & 0xFu) << (4 * g);
        cand[g] = static_cast<uint32_t>(c);
      }
      if constexpr (GPT == 2) {
        __stcs(static_cast<uint2*>(k.out0) + unit, make_uint2(v[0], v[1]));
        if (k.out2 != nullptr)
          static_cast<uint16_t*>(k.out2)[unit] = static_cast<uint16_t>(cand[0] | (cand[1] << 8));
      } else {
        __stcs(static_cast<uint32_t*>(k.out0) + unit, v[0]);
        if (k.out2 != nullptr) static_cast<uint8_t*>(k.out2)[unit] = static_cast<uint8_t>(cand[0]);
      }
    }
    const int lane = t & 31;
    uint32_t word = codes << (4 * GPT * (lane % kLanesPerWord));
#pragma unroll
    for (int o = 1; o < kLanesPerWord; o <<= 1) word |= __shfl_down_sync(0xFFFFFFFFu, word, o);
    if (active && lane % kLanesPerWord == 0)
      __stcs(static_cast<uint32_t*>(k.out1) + unit / kLanesPerWord, word);
  }
};

// The previous step's draws of a chunk (one byte per group) travel with the
// chunk's other inputs as one more bulk copy when the copy's start and size
// are 16-byte multiples (every chunk of rows whose length is a multiple of
// 64 weights); otherwise each consumer thread loads its two bytes directly.
__device__ __forceinline__ bool prev_staged(const MatDesc& d, const Chunk& c) {
  return d.G != nullptr && ((c.g0 | c.ng) & 15) == 0;
}

__device__ __forceinline__ void issue_prev(const MatDesc& d, const Chunk& c, uint8_t* dst,
                                           uint64_t* bar) {
  if (prev_staged(d, c)) {
    mbar_expect_tx(bar, static_cast<uint32_t>(c.ng));
    bulk_load(dst, static_cast<const uint8_t*>(d.G) + c.g0, static_cast<uint32_t>(c.ng), bar);
  }
}

// This thread's previous draws (two bytes: groups 2t, 2t + 1).
__device__ __forceinline__ uint32_t load_prev2(const MatDesc& d, const Chunk& c,
                                               const uint8_t* staged, int t) {
  if (d.G == nullptr) return 0u;
  if (prev_staged(d, c)) return *reinterpret_cast<const uint16_t*>(staged + 2 * t);
  return static_cast<const uint16_t*>(d.G)[c.g0 / 2 + t];
}

// Convergence diagnostics ("MaskLLM" project page, Fig. 5): per step, the
// candidate drawn for every group (the first maximum of the noisy logits z,
// the mask the soft mask tends to as tau -> 0), the L1 distance of the drawn
// masks to the previous step's draws, and the maximum probability of the
// categorical distribution softmax(fl32(kappa * L)) the draw samples from.
// Candidate c's kept positions as a 4-bit mask (bit j = position j), one
// nibble per candidate: c0 0011, c1 0101, c2 1001, c3 0110, c4 1010, c5 1100.
constexpr uint32_t kKeepBits = 0xCA6953u;

template <int GPT>
struct StatsOp : OpBase<GPT, 4> {
  static constexpr bool kTable = true, kStaged = false, kWarpWide = false;
  static constexpr bool kOutOverlapsInput = false;
  static constexpr bool kRefillFirst = true;   // partials after the logits
  static constexpr uint32_t kOutOffset = 0;
  static constexpr uint32_t kOutBytesPerGroup = 0;
  // logits, per-thread partials (L1 distance, max probability), then the
  // previous draws (one byte per group)
  static constexpr int kRowQuantities = 2;
  static constexpr bool kWarpRowSums = true;
  static constexpr int kIntQuantity = 0;   // the L1 distance is an integer count
  static constexpr uint32_t kPartOffset = kChunkGroups * 24;
  static constexpr uint32_t kPartStride = 8;
  static constexpr uint32_t kPrevOffset = kPartOffset + (kChunkGroups / GPT) * kPartStride;
  static constexpr uint32_t kStageBytes = kPrevOffset + kChunkGroups;
  static_assert(kPrevOffset % 16 == 0, "the previous draws' copy starts on a 16-byte boundary");

  __device__ static bool want_row(const MatDesc& d, int q) {
    return q == 0 ? (d.out1 != nullptr && d.G != nullptr) : d.out2 != nullptr;
  }
  __device__ static void write_row(const MatDesc& d, int64_t row, int q, float v) {
    if (q == 0)
      static_cast<uint32_t*>(d.out1)[row] = static_cast<uint32_t>(v);   // exact below 2^24
    else
      static_cast<float*>(d.out2)[row] = v;
  }

  __device__ static void issue(const MatDesc& d, const Chunk& c, uint8_t* st, uint64_t* bar) {
    const uint32_t lb = static_cast<uint32_t>(c.ng) * 24;
    mbar_expect_tx(bar, lb);
    bulk_load(st, static_cast<const uint8_t*>(d.L) + c.g0 * 24, lb, bar);
    issue_prev(d, c, st + kPrevOffset, bar);
  }

  __device__ static void consume(const StreamParams& p, const MatDesc& d, const Chunk& c,
                                 uint8_t* st, int t, const float* tab, float* acc) {
    static_assert(GPT == 2, "draws are stored as one 16-bit pair per thread");
    float L[6 * GPT];
    load_l<GPT>(st, t, L);
    const int64_t unit = c.g0 / GPT + t;
    const uint32_t prev = load_prev2(d, c, st + kPrevOffset, t);
    uint32_t drawn = 0;
    const uint64_t g0 = static_cast<uint64_t>(c.g0) + static_cast<uint64_t>(GPT * t);
#pragma unroll
    for (int k = 0; k < GPT; ++k) {
      const float* Lk = L + 6 * k;
      float g[kCand], z[kCand], y[kCand];
      gumbel6(group_words(g0 + k, p.s.step, d.tensor_id, p.s.keys), tab, g);
#pragma unroll
      for (int c6 = 0; c6 < kCand; ++c6) {
        y[c6] = __fmul_rn(p.s.kappa, Lk[c6]);
        z[c6] = __fmul_rn(__fadd_rn(y[c6], g[c6]), p.s.rho);
      }
      const int s = first_argmax6(z);
      drawn |= static_cast<uint32_t>(s) << (8 * k);
      if (d.G != nullptr) {
        const uint32_t q = (prev >> (8 * k)) & 7u;   // entries 6, 7 count as empty masks
        acc[0] += static_cast<float>(__popc(((kKeepBits >> (4 * s)) ^ (kKeepBits >> (4 * q))) & 0xFu));
      }
      const float m = fmaxf(fmaxf(fmaxf(y[0], y[1]), fmaxf(y[2], y[3])), fmaxf(y[4], y[5]));
      float sum = 0.f;
#pragma unroll
      for (int c6 = 0; c6 < kCand; ++c6) sum += ex2_approx((y[c6] - m) * kLog2e);
      acc[1] += rcp_approx(sum);   // the largest term is 2^0 = 1
    }
    if (d.out0 != nullptr) static_cast<uint16_t*>(d.out0)[unit] = static_cast<uint16_t>(drawn);
  }
};

// The forward with the convergence diagnostics in the same pass (the
// optional outputs of the "MaskLLM" Fig. 5 quantities): the noisy logits z
// the forward forms anyway give the draw (their first maximum), and the
// scaled logits fl32(kappa * L) it forms on the way give the distribution's
// largest probability.  W' is computed exactly as in FwdOp, the draws and
// the L1 distances exactly as in StatsOp, and the row sums are added in
// their order too (each thread's groups in turn, warp sums, the producer
// adding the 16 warp sums).  Row quantities: 0 row_sq, 1 L1 distance, 2
// max-probability sum.
template <int GPT>
struct FwdStatsOp : OpBase<GPT, 4> {
  static constexpr bool kTable = true, kStaged = false, kWarpWide = false;
  static constexpr bool kOutOverlapsInput = false;
  static constexpr int kRowQuantities = 3;
  // warp sums in a region of their own after the logits, the refill issued
  // before the producer adds them: 584 -> 536 us on the LLaMA-2-7B block
  // (rows of 1024 groups end a row every chunk), a Nemotron-4 layer 1012 ->
  // 1039 us (a row end every other chunk); per-thread partials summed by the
  // producer after its refill: 613 and 980 us
  static constexpr bool kWarpRowSums = true;
  static constexpr int kIntQuantity = 1;   // the L1 distance is an integer count
  static constexpr bool kRefillFirst = true;
  static constexpr uint32_t kPartOffset = kChunkGroups * (8 + 24);
  static constexpr uint32_t kPartStride = 12;
  __device__ static bool want_row(const MatDesc& d, int q) {
    return q == 0 ? d.out1 != nullptr : (q == 1 ? (d.out3 != nullptr && d.G != nullptr)
                                                 : d.out4 != nullptr);
  }
  __device__ static void write_row(const MatDesc& d, int64_t row, int q, float v) {
    if (q == 0)
      static_cast<float*>(d.out1)[row] = v;
    else if (q == 1)
      static_cast<uint32_t*>(d.out3)[row] = static_cast<uint32_t>(v);   // exact below 2^24
    else
      static_cast<float*>(d.out4)[row] = v;
  }
  static constexpr uint32_t kStageBytes = kPartOffset + (kChunkGroups / GPT) * kPartStride;
  static constexpr uint32_t kOutOffset = 0;
  static constexpr uint32_t kOutBytesPerGroup = 0;

  __device__ static void issue(const MatDesc& d, const Chunk& c, uint8_t* st, uint64_t* bar) {
    FwdOp<false, GPT>::issue(d, c, st, bar);
  }

  __device__ static void consume(const StreamParams& p, const MatDesc& d, const Chunk& c,
                                 uint8_t* st, int t, const float* tab, float* acc) {
    static_assert(GPT == 2, "draws are stored as one 16-bit pair per thread");
    uint32_t w[2 * GPT], o[2 * GPT];
    float L[6 * GPT];
    load_w<GPT>(st, t, w);
    load_l<GPT>(st + kChunkGroups * 8, t, L);
    const int64_t unit = c.g0 / GPT + t;
    const uint32_t prev = d.G != nullptr ? static_cast<const uint16_t*>(d.G)[unit] : 0u;
    const uint64_t g0 = static_cast<uint64_t>(c.g0) + static_cast<uint64_t>(GPT * t);
    uint32_t drawn = 0;
#pragma unroll
    for (int k = 0; k < GPT; ++k) {
      const float* Lk = L + 6 * k;
      float g[kCand], y[kCand], z[kCand], e[kCand], inv, num[4], M[4];
      gumbel6(group_words(g0 + k, p.s.step, d.tensor_id, p.s.keys), tab, g);
      noisy_logits6(Lk, g, p.s.kappa, p.s.rho, y, z);
      softmax6_of_z(z, e, inv, num);
      soft_mask4(num, inv, M);
      const uint32_t w01 = w[2 * k], w23 = w[2 * k + 1];
      const float x0 = __fmul_rn(bf16_lo(w01), M[0]);
      const float x1 = __fmul_rn(bf16_hi(w01), M[1]);
      const float x2 = __fmul_rn(bf16_lo(w23), M[2]);
      const float x3 = __fmul_rn(bf16_hi(w23), M[3]);
      o[2 * k] = pack_bf16x2_rn(x0, x1);
      o[2 * k + 1] = pack_bf16x2_rn(x2, x3);
      acc[0] = __fmaf_rn(x0, x0, acc[0]);
      acc[0] = __fmaf_rn(x1, x1, acc[0]);
      acc[0] = __fmaf_rn(x2, x2, acc[0]);
      acc[0] = __fmaf_rn(x3, x3, acc[0]);
      // diagnostics
      const int s = first_argmax6(z);
      drawn |= static_cast<uint32_t>(s) << (8 * k);
      const float my = fmaxf(fmaxf(fmaxf(y[0], y[1]), fmaxf(y[2], y[3])), fmaxf(y[4], y[5]));
      float sum = 0.f;
#pragma unroll
      for (int c6 = 0; c6 < kCand; ++c6) sum += ex2_approx((y[c6] - my) * kLog2e);
      acc[2] += rcp_approx(sum);   // the largest term is 2^0 = 1
    }
    // the previous draws are used last, so their load has the most work to
    // hide behind (integer counts: the order of the additions is immaterial)
    if (d.G != nullptr) {
#pragma unroll
      for (int k = 0; k < GPT; ++k) {
        const uint32_t s = (drawn >> (8 * k)) & 0xFFu;
        const uint32_t q = (prev >> (8 * k)) & 7u;   // entries 6, 7 count as empty masks
        acc[1] += static_cast<float>(
            __popc(((kKeepBits >> (4 * s)) ^ (kKeepBits >> (4 * q))) & 0xFu));
      }
    }
    store_w_global<GPT>(d.out0, unit, o);
    if (d.out2 != nullptr) static_cast<uint16_t*>(d.out2)[unit] = static_cast<uint16_t>(drawn);
  }
};

// The backward with the convergence diagnostics in the same pass (the
// "MaskLLM" Fig. 5 quantities, as FwdStatsOp gives them with the forward):
// the noisy logits z the backward regenerates give the draw, the scaled
// logits fl32(kappa * L) the distribution's largest probability.  dlogits
// are computed exactly as in BwdOp; the draws, the L1 distances and the
// max-probability row sums exactly as in StatsOp, added in its order.  The
// backward's compute and its copies are balanced, so the diagnostics' ~50
// instructions per group cost time (LLaMA-2-7B block: 648 against 475 us),
// less than a separate diagnostics pass (438 us).  Row-chunked (the row
// sums), the previous draws read from the parameter block's prev[]
// (nullable).
// Outputs: out0 dlogits (staged over the logits, bulk-stored), out1 draws,
// out2 L1 distance per row (u32, needs the previous draws), out3
// max-probability sum per row.  Row quantities: 0 L1 distance, 1
// max-probability sum.
template <bool kReg, int GPT>
struct BwdStatsOp : OpBase<GPT, 4> {
  static constexpr bool kTable = true, kStaged = true, kWarpWide = false;
  static constexpr bool kOutOverlapsInput = true;    // dlogits overwrite the logits
  static constexpr uint32_t kProducerNapNs = 64;
  static constexpr int kRowQuantities = 2;
  static constexpr bool kWarpRowSums = true;
  static constexpr int kIntQuantity = 0;   // the L1 distance is an integer count
  // row partials (a warp's sum in its lane 0's slot; short rows: one per
  // thread) in each thread's own W slot, consumed before it writes there:
  // the stage holds nothing more than BwdOp's.  The producer adds them up
  // before it refills the stage, and the consumers' proxy fence (staged
  // outputs) orders these writes before the refill's copies.
  static constexpr uint32_t kPartOffset = 0;
  static constexpr uint32_t kPartStride = 8 * GPT;
  static_assert(8 * GPT >= 8, "two row partials fit the thread's W slot");
  static constexpr uint32_t kStageBytes = kChunkGroups * (8 + 8 + 24);
  static constexpr uint32_t kOutOffset = kChunkGroups * 16;
  static constexpr uint32_t kOutBytesPerGroup = 24;

  // an L1 output implies previous draws (the host checks)
  __device__ static bool want_row(const MatDesc& d, int q) {
    return q == 0 ? d.out2 != nullptr : d.out3 != nullptr;
  }
  __device__ static void write_row(const MatDesc& d, int64_t row, int q, float v) {
    if (q == 0)
      static_cast<uint32_t*>(d.out2)[row] = static_cast<uint32_t>(v);   // exact below 2^24
    else
      static_cast<float*>(d.out3)[row] = v;
  }

  __device__ static void issue(const MatDesc& d, const Chunk& c, uint8_t* st, uint64_t* bar) {
    BwdOp<kReg, GPT>::issue(d, c, st, bar);
  }

  __device__ static void consume(const StreamParams& p, const MatDesc& d, const Chunk& c,
                                 uint8_t* st, int t, const float* tab, float* acc) {
    static_assert(GPT == 2, "draws are stored as one 16-bit pair per thread");
    uint32_t w[2 * GPT], gr[2 * GPT];
    float L[6 * GPT], dl[6 * GPT];
    load_w<GPT>(st, t, w);
    load_w<GPT>(st + kChunkGroups * 8, t, gr);
    load_l<GPT>(st + kChunkGroups * 16, t, L);
    const int64_t unit = c.g0 / GPT + t;
    const uint16_t* prevp = static_cast<const uint16_t*>(p.prev[c.mat]);
    const uint32_t prev = prevp != nullptr ? prevp[unit] : 0u;
    const uint64_t g0 = static_cast<uint64_t>(c.g0) + static_cast<uint64_t>(GPT * t);
    uint32_t drawn = 0;
#pragma unroll
    for (int k = 0; k < GPT; ++k) {
      float y[kCand], z[kCand];
      BwdOp<kReg, GPT>::group(p, tab, g0 + k, d.tensor_id, L + 6 * k, w[2 * k], w[2 * k + 1],
                              gr[2 * k], gr[2 * k + 1], dl + 6 * k, y, z);
      const int s = first_argmax6(z);
      drawn |= static_cast<uint32_t>(s) << (8 * k);
      if (prevp != nullptr) {
        const uint32_t q = (prev >> (8 * k)) & 7u;   // entries 6, 7 count as empty masks
        acc[0] += static_cast<float>(__popc(((kKeepBits >> (4 * s)) ^ (kKeepBits >> (4 * q))) & 0xFu));
      }
      const float m = fmaxf(fmaxf(fmaxf(y[0], y[1]), fmaxf(y[2], y[3])), fmaxf(y[4], y[5]));
      float sum = 0.f;
#pragma unroll
      for (int c6 = 0; c6 < kCand; ++c6) sum += ex2_approx((y[c6] - m) * kLog2e);
      acc[1] += rcp_approx(sum);   // the largest term is 2^0 = 1
    }
    store_l<GPT>(st + kChunkGroups * 16, t, dl);   // dlogits over this thread's own logits
    if (d.out1 != nullptr) static_cast<uint16_t*>(d.out1)[unit] = static_cast<uint16_t>(drawn);
  }
};

// ---------------------------------------------------------------------------
// The kernel.
// ---------------------------------------------------------------------------

template <class Op>
struct Layout {
  static constexpr uint32_t kTableBytes = Op::kTable ? kTableSize * 4 : 0;
  static constexpr uint32_t kStageOff = kTableBytes;
  static constexpr uint32_t kBarOff = kStageOff + Op::kStages * Op::kStageBytes;
  static constexpr uint32_t kChunkOff = kBarOff + 2 * Op::kStages * 8;
  static constexpr uint32_t kFlagOff = kChunkOff + Op::kStages * sizeof(Chunk);
  static constexpr uint32_t kBytes = kFlagOff + 16;

  // Every shared-memory region a consumer writes lies inside its stage: the
  // row partials of every consumer thread (short rows use one slot per
  // thread), the staged output in every output buffer, and (as each op
  // states beside its layout) the inputs.
  static_assert(Op::kRowQuantities == 0 ||
                    (4 * Op::kRowQuantities <= Op::kPartStride &&
                     Op::kPartOffset + Op::kConsumers * Op::kPartStride <= Op::kStageBytes),
                "row partials of every consumer lie inside the stage");
  static_assert(!Op::kStaged || Op::kOutOffset + (Op::kOutBuffers - 1) * Op::kOutBufBytes +
                                        kChunkGroups * Op::kOutBytesPerGroup <=
                                    Op::kStageBytes,
                "staged outputs lie inside the stage");
  static_assert(Op::kStageBytes % 16 == 0, "stages start on 16-byte boundaries");
};

// The producer's wait for the consumers to release a stage.
template <class Op>
__device__ __forceinline__ bool wait_empty(uint64_t* bar, uint32_t parity, uint64_t limit_ns,
                                           volatile int* abort_flag) {
  if (Op::kProducerNapNs > 0)
    return mbar_wait_napping(bar, parity, limit_ns, abort_flag, Op::kProducerNapNs);
  return mbar_wait_bounded(bar, parity, limit_ns, abort_flag);
}

// Producer warp: refills the stage ring, finishes retired chunks.
template <class Op>
__device__ void producer(const StreamParams& p, uint8_t* smem, int64_t u0, int64_t u1) {
  using Lay = Layout<Op>;
  constexpr int S = Op::kStages;
  const int lane = threadIdx.x & 31;
  uint8_t* stages = smem + Lay::kStageOff;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Lay::kBarOff);
  uint64_t* empty = full + S;
  Chunk* held = reinterpret_cast<Chunk*>(smem + Lay::kChunkOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Lay::kFlagOff);

  // Finish the chunk that occupied stage s: row sums and staged stores.
  auto retire = [&](const Chunk c, int s) {
    const MatDesc& d = p.mats[c.mat];
    const uint8_t* st = stages + s * Op::kStageBytes;
    if (Op::kRowQuantities > 0 && c.nrows > 0) {
#pragma unroll
      for (int q = 0; q < Op::kRowQuantities; ++q) {
        if (!Op::want_row(d, q)) continue;
        auto part = [&](int k) {
          return *reinterpret_cast<const float*>(st + Op::kPartOffset + k * Op::kPartStride +
                                                 4 * q);
        };
        if (d.cpr > 0 && Op::kWarpRowSums) {
          // one partial per consumer warp (each already its warp's sum, in
          // the slot of the warp's lane 0)
          static_assert(Op::kConsumerWarps <= 32, "one warp sum per lane");
          float v = lane < Op::kConsumerWarps ? part(32 * lane) : 0.f;
          v = warp_sum(v);
          if (lane == 0) Op::write_row(d, c.row0, q, v);
        } else if (d.cpr > 0) {
          // the same order as a lane-strided loop (lane, lane + 32, ...),
          // with every load issued up front
          float v = 0.f;
#pragma unroll
          for (int i = 0; i < Op::kConsumers / 32; ++i) v += part(lane + 32 * i);
          v = warp_sum(v);
          if (lane == 0) Op::write_row(d, c.row0, q, v);
        } else {
          const int tpr = d.gpr / Op::kGPT;   // threads per short row
          for (int r = 0; r < c.nrows; ++r) {
            float v = 0.f;
            for (int k = lane; k < tpr; k += 32) v += part(r * tpr + k);
            v = warp_sum(v);
            if (lane == 0) Op::write_row(d, c.row0 + r, q, v);
          }
        }
      }
    }
    if (Op::kStaged && lane == 0) {
      bulk_store(static_cast<uint8_t*>(d.out0) + c.g0 * Op::kOutBytesPerGroup,
                 st + Op::kOutOffset + c.obuf * Op::kOutBufBytes,
                 static_cast<uint32_t>(c.ng) * Op::kOutBytesPerGroup);
      bulk_commit();
    }
  };

  ChunkIter<Op::kFlat> it;
  it.init(&p, u0, u1);
  Chunk c;
  int64_t n = 0;
  bool ok = true;
  Chunk old;
  while (it.next(c)) {
    const int s = static_cast<int>(n % S);
    if (n >= S) {
      const bool got = wait_empty<Op>(&empty[s], static_cast<uint32_t>((n / S - 1) & 1), p.wait_ns,
                                      abort_flag);
      if (!__all_sync(0xFFFFFFFFu, got)) {
        if (lane == 0) raise_abort(abort_flag, 2u);
        ok = false;
        break;
      }
      old = held[s];
      // every lane has the old record before lane 0 replaces it (otherwise
      // the retirement and its barrier below come first)
      if (Op::kRefillFirst) __syncwarp();
      if (!Op::kRefillFirst) {
        retire(old, s);
        __syncwarp();
      }
    }
    if (lane == 0) {
      c.obuf = static_cast<int32_t>((n / S) % Op::kOutBuffers);
      held[s] = c;
      // a staged store may still be reading this stage's output region:
      // wait before the refill if the copies land there, after it if not
      if (Op::kStaged && Op::kOutOverlapsInput) bulk_wait_reads();
      if (!p.withhold_loads)
        Op::issue(p.mats[c.mat], c, stages + s * Op::kStageBytes, &full[s]);
      else
        mbar_expect_tx(&full[s], 16);   // test hook: bytes that never come
    }
    if (Op::kRefillFirst && n >= S) {
      retire(old, s);   // the copies above land elsewhere in the stage
      __syncwarp();
    }
    if (lane == 0) {
      // the store that last read the output buffer this chunk will write --
      // the stage's chunk kOutBuffers turns ago -- has at most
      // S (kOutBuffers - 1) stores committed after it
      if (Op::kStaged && !Op::kOutOverlapsInput)
        bulk_wait_reads_but<S * (Op::kOutBuffers - 1)>();
      mbar_arrive(&full[s]);   // with the copies' bytes, completes the phase
    }
    __syncwarp();
    ++n;
  }
  if (ok) {
    // drain: finish the last chunks as the consumers release them
    for (int64_t k = n > S ? n - S : 0; k < n; ++k) {
      const int s = static_cast<int>(k % S);
      const bool got = wait_empty<Op>(&empty[s], static_cast<uint32_t>((k / S) & 1), p.wait_ns,
                                      abort_flag);
      if (!__all_sync(0xFFFFFFFFu, got)) {
        if (lane == 0) raise_abort(abort_flag, 2u);
        ok = false;
        break;
      }
      retire(held[s], s);
      __syncwarp();
    }
  }
  if (!ok && !p.withhold_loads) {
    // aborted: wait (bounded) for every copy still landing in shared memory
    for (int64_t k = n > S ? n - S : 0; k < n; ++k) {
      const int s = static_cast<int>(k % S);
      int never = 0;
      const bool landed = mbar_wait_bounded(&full[s], static_cast<uint32_t>((k / S) & 1),
                                            p.drain_ns, &never);
      if (!landed && lane == 0) atomicOr(&g_stream_error_word, 4u);
    }
  }
  if (Op::kStaged && lane == 0) bulk_wait_all();
}

// Consumer warps: thread t owns GPT groups of every chunk.  The chunk in a
// stage is the one the producer recorded there (held[s], written before its
// arrival on full[s]); the consumers only count their chunks.
template <class Op>
__device__ void consumer(const StreamParams& p, uint8_t* smem, int64_t u0, int64_t u1) {
  using Lay = Layout<Op>;
  constexpr int S = Op::kStages;
  const int t = threadIdx.x - 32;
  const int lane = threadIdx.x & 31;
  uint8_t* stages = smem + Lay::kStageOff;
  const float* tab = reinterpret_cast<const float*>(smem);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Lay::kBarOff);
  uint64_t* empty = full + S;
  const Chunk* held = reinterpret_cast<const Chunk*>(smem + Lay::kChunkOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Lay::kFlagOff);

  const int64_t nchunks = chunk_index(p, u1) - chunk_index(p, u0);
  float acc[3] = {0.f, 0.f, 0.f};   // per-row quantities of this thread
  for (int64_t n = 0; n < nchunks; ++n) {
    const int s = static_cast<int>(n % S);
    const bool got = mbar_wait_bounded(&full[s], static_cast<uint32_t>((n / S) & 1), p.wait_ns,
                                       abort_flag);
    if (!__all_sync(0xFFFFFFFFu, got)) {
      if (lane == 0) raise_abort(abort_flag, 1u);
      break;
    }
    const Chunk c = held[s];
    const MatDesc& d = p.mats[c.mat];
    uint8_t* st = stages + s * Op::kStageBytes;
    if (Op::kWarpWide)
      Op::consume(p, d, c, st, t, tab, acc);   // every lane, active or not
    else if (Op::kGPT * t < c.ng)
      Op::consume(p, d, c, st, t, tab, acc);
    if (Op::kRowQuantities > 0) {
      if (Op::kWarpRowSums && d.cpr > 0) {
        if (c.nrows > 0) {
          // the row ends in this chunk: each warp leaves the sum of its
          // lanes' partials in its lane 0's slot (a slot that thread has
          // consumed itself), so the producer adds only kConsumerWarps values
          float* part =
              reinterpret_cast<float*>(st + Op::kPartOffset + (t & ~31) * Op::kPartStride);
#pragma unroll
          for (int q = 0; q < Op::kRowQuantities; ++q) {
            // an integer count below 2^24 is exact in fp32 and sums in one
            // warp-reduce instruction
            const float v = q == Op::kIntQuantity
                                ? static_cast<float>(__reduce_add_sync(
                                      0xFFFFFFFFu, static_cast<uint32_t>(acc[q])))
                                : warp_sum(acc[q]);
            if (lane == 0) part[q] = v;
            acc[q] = 0.f;
          }
        }
      } else if (d.cpr == 0 || c.nrows > 0) {
        // the row ends in this chunk (long rows), or each thread's groups
        // lie in one short row of this chunk: each thread's own partial
        float* part = reinterpret_cast<float*>(st + Op::kPartOffset + t * Op::kPartStride);
#pragma unroll
        for (int q = 0; q < Op::kRowQuantities; ++q) {
          part[q] = acc[q];
          acc[q] = 0.f;
        }
      }
    }
    if (Op::kStaged) fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
}

template <class Op>
__global__ void __launch_bounds__(Op::kThreads, 1)
    stream_kernel(const __grid_constant__ StreamParams p) {
  using Lay = Layout<Op>;
  extern __shared__ __align__(128) uint8_t smem[];
  if (Op::kTable) {
    const float4* src = reinterpret_cast<const float4*>(g_gumbel_table_s);
    float4* dst = reinterpret_cast<float4*>(smem);
    for (int i = threadIdx.x; i < kTableSize / 4; i += Op::kThreads) dst[i] = src[i];
  }
  if (threadIdx.x == 0) {
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kBarOff);
    for (int s = 0; s < Op::kStages; ++s) {
      mbar_init(&bars[s], 1);                                  // full: producer's expect_tx
      mbar_init(&bars[Op::kStages + s], Op::kConsumerWarps);   // empty: one per consumer warp
    }
    *reinterpret_cast<volatile int*>(smem + Lay::kFlagOff) = 0;
    fence_barrier_init();
  }
  __syncthreads();
  const int64_t u0 = cta_first_unit(p, blockIdx.x, gridDim.x);
  const int64_t u1 = cta_first_unit(p, blockIdx.x + 1, gridDim.x);
  if (threadIdx.x < 32)
    producer<Op>(p, smem, u0, u1);
  else
    consumer<Op>(p, smem, u0, u1);
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------

// Host settings, written by the exported setters from any thread and read
// by every launch.
std::atomic<uint64_t> g_wait_ns{2000000000ull};   // 2 s
std::atomic<int> g_withhold_loads{0};

// Chunking of each matrix.  Ops with per-row sums (forward, diagnostics)
// chunk row by row: a long row is split into chunks, short rows are packed
// whole, so every row ends inside one chunk range and one CTA.  The other
// ops (prior, backward, hard-compress) treat the matrix as one flat array of
// groups (row-major, no padding): chunks of kChunkGroups groups with a
// ragged last chunk, described as "rows" of one chunk each -- every chunk
// full, and the CTAs' shares equal to within one chunk whatever the row
// length.
void describe(StreamParams& p, const StreamMatrix* mats, int n, bool flat) {
  p.nmats = n;
  p.flat = flat ? 1 : 0;
  int64_t units = 0, chunks = 0;
  for (int i = 0; i < n; ++i) {
    MatDesc& d = p.mats[i];
    const StreamMatrix& m = mats[i];
    d.W = m.W;
    d.L = m.L;
    d.G = m.G;
    d.out0 = m.out0;
    d.out1 = m.out1;
    d.out2 = m.out2;
    d.out3 = m.out3;
    d.out4 = m.out4;
    d.rows = m.rows;
    d.gpr = static_cast<int32_t>(m.cols / 4);
    d.tensor_id = m.tensor_id;
    p.prev[i] = m.P;
    if (flat) {
      const int64_t groups = m.rows * (m.cols / 4);
      d.gpr = kChunkGroups;
      d.rows = (groups + kChunkGroups - 1) / kChunkGroups;
      d.cpr = 1;
      d.rpc = static_cast<int32_t>(groups - (d.rows - 1) * kChunkGroups);
    } else if (d.gpr >= kChunkGroups) {
      d.cpr = (d.gpr + kChunkGroups - 1) / kChunkGroups;
      d.rpc = 0;
    } else {
      d.cpr = 0;
      d.rpc = kChunkGroups / d.gpr;
    }
    d.unit_begin = units;
    d.chunk_begin = chunks;
    const int64_t u = d.cpr > 0 ? d.rows : (d.rows + d.rpc - 1) / d.rpc;
    units += u;
    chunks += d.cpr > 0 ? u * d.cpr : u;
  }
  p.total_units = units;
  p.total_chunks = chunks;
  const uint64_t wait_ns = g_wait_ns.load(std::memory_order_relaxed);
  p.wait_ns = wait_ns;
  p.drain_ns = wait_ns > 1000000000ull ? wait_ns : 1000000000ull;
  p.withhold_loads = g_withhold_loads.load(std::memory_order_relaxed);
}

template <class Op>
cudaError_t launch(const Device& dev, const StreamParams& p, cudaStream_t s) {
  if (p.flat != (Op::kFlat ? 1 : 0)) return cudaErrorInvalidValue;   // chunking mismatch
  const uint32_t bytes = Layout<Op>::kBytes;
  cudaError_t e = cudaFuncSetAttribute(stream_kernel<Op>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  const int64_t grid = p.total_units < dev.num_sms ? p.total_units : dev.num_sms;
  stream_kernel<Op><<<static_cast<int>(grid), Op::kThreads, bytes, s>>>(p);
  return cudaGetLastError();
}

Scalars scalars(float tau, float kappa, RngArgs rng, float reg, float scale) {
  Scalars sc;
  sc.kappa = kappa;
  sc.rho = static_cast<float>(1.0 / static_cast<double>(tau));
  sc.dz_dlogit = static_cast<float>(static_cast<double>(kappa) * static_cast<double>(sc.rho));
  sc.two_reg = 2.0f * reg;
  sc.scale = scale;
  sc.step = rng.step;
  sc.keys = make_round_keys(rng.seed);
  return sc;
}

}  // namespace

constexpr int kGPT = 2;   // groups per consumer thread (16 consumer warps)
static_assert(Layout<FwdOp<true, kGPT>>::kBytes <= 232448, "forward shared memory");
static_assert(Layout<BwdOp<true, kGPT>>::kBytes <= 232448, "backward shared memory");
static_assert(Layout<PriorOp<kGPT>>::kBytes <= 232448, "prior shared memory");
static_assert(Layout<CompressOp<kGPT>>::kBytes <= 232448, "compress shared memory");
static_assert(Layout<StatsOp<kGPT>>::kBytes <= 232448, "stats shared memory");
static_assert(Layout<FwdStatsOp<kGPT>>::kBytes <= 232448, "forward + stats shared memory");
static_assert(Layout<BwdStatsOp<true, kGPT>>::kBytes <= 232448, "backward + stats shared memory");
static_assert(sizeof(StreamParams) <= 4000, "kernel parameters");

cudaError_t stream_prior_init(const Device& d, const StreamMatrix* m, int n, float scale,
                              cudaStream_t s) {
  StreamParams p;
  describe(p, m, n, true);
  p.s = scalars(1.0f, 0.0f, {0, 0, 0}, 0.0f, scale);
  return launch<PriorOp<kGPT>>(d, p, s);
}

cudaError_t stream_forward(const Device& d, const StreamMatrix* m, int n, float tau, float kappa,
                           RngArgs rng, bool probs, cudaStream_t s) {
  StreamParams p;
  describe(p, m, n, false);
  p.s = scalars(tau, kappa, rng, 0.0f, 0.0f);
  return probs ? launch<FwdOp<true, kGPT>>(d, p, s) : launch<FwdOp<false, kGPT>>(d, p, s);
}

cudaError_t stream_backward(const Device& d, const StreamMatrix* m, int n, float tau, float kappa,
                            RngArgs rng, float reg_coeff, cudaStream_t s) {
  StreamParams p;
  describe(p, m, n, true);
  p.s = scalars(tau, kappa, rng, reg_coeff, 0.0f);
  return reg_coeff != 0.0f ? launch<BwdOp<true, kGPT>>(d, p, s)
                           : launch<BwdOp<false, kGPT>>(d, p, s);
}

cudaError_t stream_hard_compress(const Device& d, const StreamMatrix* m, int n, cudaStream_t s) {
  StreamParams p;
  describe(p, m, n, true);
  p.s = scalars(1.0f, 0.0f, {0, 0, 0}, 0.0f, 0.0f);
  return launch<CompressOp<kGPT>>(d, p, s);
}

cudaError_t stream_mask_stats(const Device& d, const StreamMatrix* m, int n, float tau, float kappa,
                              RngArgs rng, cudaStream_t s) {
  StreamParams p;
  describe(p, m, n, false);
  p.s = scalars(tau, kappa, rng, 0.0f, 0.0f);
  return launch<StatsOp<kGPT>>(d, p, s);
}

cudaError_t stream_forward_stats(const Device& d, const StreamMatrix* m, int n, float tau,
                                 float kappa, RngArgs rng, cudaStream_t s) {
  StreamParams p;
  describe(p, m, n, false);
  p.s = scalars(tau, kappa, rng, 0.0f, 0.0f);
  return launch<FwdStatsOp<kGPT>>(d, p, s);
}

cudaError_t stream_backward_stats(const Device& d, const StreamMatrix* m, int n, float tau,
                                  float kappa, RngArgs rng, float reg_coeff, cudaStream_t s) {
  StreamParams p;
  describe(p, m, n, false);
  p.s = scalars(tau, kappa, rng, reg_coeff, 0.0f);
  return reg_coeff != 0.0f ? launch<BwdStatsOp<true, kGPT>>(d, p, s)
                           : launch<BwdStatsOp<false, kGPT>>(d, p, s);
}

void stream_set_wait_ns(uint64_t ns) { g_wait_ns.store(ns, std::memory_order_relaxed); }
uint64_t stream_wait_ns() { return g_wait_ns.load(std::memory_order_relaxed); }
void stream_set_withhold_loads(int on) {
  g_withhold_loads.store(on, std::memory_order_relaxed);
}

cudaError_t read_and_clear_stream_error(cudaStream_t s, uint32_t* value) {
  uint32_t zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(value, g_stream_error_word, sizeof(uint32_t), 0,
                                            cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return e;
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return e;
  if (*value != 0) {
    e = cudaMemcpyToSymbolAsync(g_stream_error_word, &zero, sizeof(uint32_t), 0,
                                cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(s);
  }
  return e;
}

}  // namespace maskllm
