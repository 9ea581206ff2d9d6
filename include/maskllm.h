/*
 * maskllm.h -- C ABI of libmaskllm: MaskLLM's differentiable 2:4 mask layer
 * on NVIDIA GB300 (sm_103a).
 *
 * The method.  "MaskLLM: Learnable Semi-Structured Sparsity for Large Language
 * Models" (project page), Fig. 3: every group of M = 4 consecutive weights of
 * a frozen matrix carries a learnable categorical distribution over the
 * candidate 2:4 masks; a mask is drawn with the Gumbel softmax and the
 * candidates are averaged with its weights, all differentiably.  Fig. 5: the
 * logits are scaled by kappa, which sets the randomness of the draw.  Table 2:
 * prior masks initialise the logits.  Table 3: a weight regulariser helps.
 * "Accelerating Sparse Deep Neural Networks" (Mishra et al.), Sec. 3.1: a 2:4
 * matrix is stored as the two kept values of each group of four plus 2 bits of
 * position metadata per kept value; Sec. 4.1: magnitude pruning keeps the two
 * largest of four.
 *
 * Notation used below.
 *   W        frozen weights, bf16, [rows, cols] row-major (bf16 values travel
 *            as their uint16_t bit patterns).  cols % 32 == 0.
 *   group    k-th group of row r = W[r, 4k .. 4k+3]; its index within the
 *            matrix is  gidx = r * (cols/4) + k.
 *   candidates  the six kept index pairs in lexicographic order
 *            c0 (0,1)  c1 (0,2)  c2 (0,3)  c3 (1,2)  c4 (1,3)  c5 (2,3).
 *   logits   L, fp32, [rows, cols/4, 6] row-major (24 bytes per group).
 *   noise    g_c, Gumbel(0,1) quantised to 2^14 cells: the four words
 *            Philox4x32-10(key = (seed lo, seed hi),
 *                           counter = (gidx lo, gidx hi, step, tensor_id));
 *            candidate c takes 16-bit half (c & 1) of word (c >> 1) (low half
 *            for even c), cell = its top 14 bits, g_c = fl32(-ln(-ln((cell +
 *            0.5) / 2^14))).  Word 3 is unused.  The noise is a pure function
 *            of (rng, gidx), so the forward and the backward of one step draw
 *            the same noise; it is never stored.
 *   z_c      = fl32(fl32(fl32(kappa * L_c) + g_c) * rho), rho = fl32(1/tau).
 *   p        = softmax(z);  M_j = sum over candidates c keeping j of p_c.
 *
 * Conventions shared by every call.
 *   - Every pointer is a DEVICE pointer owned by the caller, 16-byte aligned.
 *     The library never allocates, frees or keeps device memory of the
 *     caller.  Inputs are read only; outputs are overwritten, never
 *     accumulated into.  An output may not overlap any input or another
 *     output.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream) and returns after the launch; nothing
 *     synchronises.
 *   - Arguments are validated on the host before anything is launched; a
 *     failed check returns its error and launches nothing.  After the launch
 *     cudaGetLastError() is checked; a launch failure returns
 *     MASKLLM_ERR_CUDA (maskllm_last_cuda_error() gives the CUDA message).
 *   - Shapes: rows >= 1, cols >= 32, cols % 32 == 0, rows * cols < 2^46.
 *     (The multiple of 32 follows the page's rule that pruned GEMM
 *     dimensions are multiples of 16/32, and makes the 32-bit metadata words
 *     of a row whole.)
 */
#ifndef MASKLLM_H_
#define MASKLLM_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t (both are `struct CUstream_st *`). */
typedef struct CUstream_st* maskllm_stream_t;

typedef enum {
  MASKLLM_OK = 0,
  MASKLLM_ERR_INVALID_ARG = 1, /* null pointer, non-finite or out-of-range scalar */
  MASKLLM_ERR_SHAPE = 2,       /* rows/cols outside the rules above */
  MASKLLM_ERR_ALIGNMENT = 3,   /* a pointer not 16-byte aligned */
  MASKLLM_ERR_ALIAS = 4,       /* an output overlaps an input or another output */
  MASKLLM_ERR_CUDA = 5,        /* the CUDA runtime reported an error */
  MASKLLM_ERR_TIMEOUT = 6      /* a bounded device-side wait gave up */
} maskllm_status;

/* Stateless RNG coordinates of one draw.  seed selects the key; step and
 * tensor_id the counter's high words (one noise stream per training step and
 * per weight matrix). */
typedef struct {
  uint64_t seed;
  uint32_t step;
  uint32_t tensor_id;
} maskllm_rng;

/* Magnitude prior (MaskLLM Table 2: prior masks initialise the logits;
 * Mishra et al. Sec. 4.1: magnitude pruning).
 *   logits_out[r, k, c] = fl32(scale * fl32(|w_i| + |w_j|)), (i, j) = pair c
 * so the argmax candidate keeps the two largest magnitudes of the group.
 *   W           in   bf16 [rows, cols]
 *   scale       in   finite
 *   logits_out  out  fp32 [rows, cols/4, 6]
 * Moves 8 bytes per weight. */
maskllm_status maskllm_prior_init(const uint16_t* W, int64_t rows, int64_t cols, float scale,
                                  float* logits_out, maskllm_stream_t stream);

/* Forward of the differentiable mask (MaskLLM Fig. 3, Fig. 5, Table 3):
 *   x_j = fl32(w_j * M_j),  W_out_j = bf16 round-to-nearest-even of x_j,
 *   row_sq_out[r] = sum over the row of x_j^2 (the weight regulariser's
 *                   per-row value; deterministic for a given shape).
 *   W           in   bf16 [rows, cols]
 *   logits      in   fp32 [rows, cols/4, 6]
 *   tau         in   > 0, finite (Gumbel-softmax temperature)
 *   kappa       in   finite (logit scale)
 *   rng         in   noise coordinates (see the notation above)
 *   W_out       out  bf16 [rows, cols]
 *   row_sq_out  out  fp32 [rows], or NULL to skip
 *   probs_out   out  fp32 [rows, cols/4, 6] = p, or NULL (debug output;
 *                    adds 24 bytes per group of traffic)
 * Moves 10 bytes per weight (W 2, logits 6, W_out 2). */
maskllm_status maskllm_forward(const uint16_t* W, const float* logits, int64_t rows,
                               int64_t cols, float tau, float kappa, maskllm_rng rng,
                               uint16_t* W_out, float* row_sq_out, float* probs_out,
                               maskllm_stream_t stream);

/* Backward of the mask (MaskLLM Fig. 3: every step is differentiable).  The
 * loss seen by the layer is  l = <G, W_out> + reg_coeff * sum x^2  with the
 * bf16 rounding of W_out passed straight through and the noise held fixed:
 *   t_j = G_j + 2 reg_coeff x_j,  h_j = t_j w_j,  dp_c = h_i + h_j,
 *   r = sum_c p_c dp_c,  dlogits_c = (kappa * rho) p_c (dp_c - r).
 * Must be called with the same rng, tau and kappa as the forward it
 * differentiates (it redraws the same noise).
 *   W           in   bf16 [rows, cols]
 *   logits      in   fp32 [rows, cols/4, 6]
 *   grad_W_out  in   bf16 [rows, cols] = dl/dW_out
 *   reg_coeff   in   finite (0 disables the regulariser term exactly)
 *   dlogits_out out  fp32 [rows, cols/4, 6] (overwritten)
 * Moves 16 bytes per weight (W 2, logits 6, grad 2, dlogits 6). */
maskllm_status maskllm_backward(const uint16_t* W, const float* logits,
                                const uint16_t* grad_W_out, int64_t rows, int64_t cols,
                                float tau, float kappa, maskllm_rng rng, float reg_coeff,
                                float* dlogits_out, maskllm_stream_t stream);

/* Hard mask and 2:4 compression (MaskLLM: the learned distribution's most
 * likely candidate is the deployed mask; Mishra et al. Sec. 3.1 storage).
 *   c* = argmax_c logits[r, k, c] over the raw logits (no noise, no kappa or
 *        tau), lowest index on ties; a NaN logit never wins; six NaNs give 0.
 *   values_out[r, 2k], values_out[r, 2k+1] = w_i, w_j for (i, j) = pair c*
 *   meta_out[r, k/8] bits 4(k%8) .. 4(k%8)+3 = i | j << 2
 *   W           in   bf16 [rows, cols]
 *   logits      in   fp32 [rows, cols/4, 6]
 *   values_out  out  bf16 [rows, cols/2]
 *   meta_out    out  uint32 [rows, cols/32]
 *   idx_out     out  uint8 [rows, cols/4] = c*, or NULL to skip
 * Moves 9.125 bytes per weight (W 2, logits 6, values 1, meta 0.125). */
maskllm_status maskllm_hard_compress(const uint16_t* W, const float* logits, int64_t rows,
                                     int64_t cols, uint16_t* values_out, uint32_t* meta_out,
                                     uint8_t* idx_out, maskllm_stream_t stream);

/* Inverse of the storage above: W_out = the kept values in place, +0 (0x0000)
 * at the two dropped positions of every group.
 *   values  in   bf16 [rows, cols/2]
 *   meta    in   uint32 [rows, cols/32]; every 4-bit code must have i < j
 *   W_out   out  bf16 [rows, cols] */
maskllm_status maskllm_decompress(const uint16_t* values, const uint32_t* meta, int64_t rows,
                                  int64_t cols, uint16_t* W_out, maskllm_stream_t stream);

/* The four Philox4x32-10 noise words of groups [group_begin, group_begin + n)
 * (see the notation above), for checking the noise stream.
 *   group_begin >= 0, n >= 1
 *   out4  out  uint32 [n, 4] */
maskllm_status maskllm_noise_words(maskllm_rng rng, int64_t group_begin, int64_t n,
                                   uint32_t* out4, maskllm_stream_t stream);

/* Logits that start from a given mask (MaskLLM Table 2: learned masks are
 * initialised from a prior mask and refined; masks transfer across tasks).
 * For every group, logits_out = high on the candidate its 4-bit code names
 * and low on the other five; a code that names no candidate (anything but
 * 0x4 0x8 0xC 0x9 0xD 0xE) gives low on all six.
 *   meta        in   uint32 [rows, cols/32], the layout maskllm_hard_compress writes
 *   high, low   in   finite
 *   logits_out  out  fp32 [rows, cols/4, 6]
 * Moves 6.125 bytes per weight. */
maskllm_status maskllm_prior_from_mask(const uint32_t* meta, int64_t rows, int64_t cols,
                                       float high, float low, float* logits_out,
                                       maskllm_stream_t stream);

/* Convergence diagnostics of one step (MaskLLM Fig. 5: (a) the L1 distance of
 * sampled masks between adjacent training steps, (b) the maximum probability
 * of the mask distribution, both governed by kappa).
 *   draw        the candidate sampled for each group at this step: the first
 *               maximum of z (see the notation above) -- the candidate the
 *               soft mask of maskllm_forward tends to as tau -> 0
 *   l1          per row, sum over groups of the L1 distance (0, 2 or 4)
 *               between this step's drawn mask and the mask of prev_idx
 *   maxprob     per row, sum over groups of max_c softmax(fl32(kappa * L))_c,
 *               the categorical distribution the draw samples from (divide by
 *               cols/4 for the row mean)
 *   logits          in   fp32 [rows, cols/4, 6]
 *   prev_idx        in   uint8 [rows, cols/4], the previous step's draws
 *                        (entries 0..5), or NULL when there is none
 *   tau, kappa, rng in   as for maskllm_forward (same noise as the forward of
 *                        this step)
 *   idx_out         out  uint8 [rows, cols/4] = the draws, or NULL
 *   l1_row_out      out  uint32 [rows], or NULL; requires prev_idx
 *   maxprob_row_out out  fp32 [rows], or NULL
 * cols <= 2^24 (the per-row L1 is summed exactly in fp32).  Moves 6.25-6.5
 * bytes per weight. */
maskllm_status maskllm_mask_stats(const float* logits, const uint8_t* prev_idx, int64_t rows,
                                  int64_t cols, float tau, float kappa, maskllm_rng rng,
                                  uint8_t* idx_out, uint32_t* l1_row_out,
                                  float* maxprob_row_out, maskllm_stream_t stream);

/* ---- Channel permutation before pruning ---------------------------------
 * "Accelerating Sparse Deep Neural Networks", Sec. 4.1 (Fig. 5): permuting
 * the input channels (columns) of W before 2:4 magnitude pruning raises the
 * magnitude that pruning keeps; the layer producing those channels permutes
 * its output rows alike, so the network computes the same function.
 * "Channel Permutations for N:M Sparsity" (abstract): a quality metric judges
 * permutations and a search finds good ones.
 *
 *   perm      int32 [cols], a permutation of 0..cols-1: slot i of the
 *             permuted matrix holds channel perm[i], W_perm[r, i] =
 *             W[r, perm[i]].
 *   q(w)      = floor(|w| * 2^shift), shift = 31 - ceil(log2 rows) -
 *             floor(log2 max|w|) (0 for an all-zero W): fixed-point
 *             magnitudes whose sum over any column is below 2^32.
 *   metric    = sum over rows and groups of W_perm of the two largest q of
 *             the group (the magnitude 2:4 magnitude pruning keeps, exact).
 *   gain(a,b) = metric after exchanging the channels of slots a and b minus
 *             the metric before; 0 for two slots of one group.
 *   search    = steepest ascent: apply the swap of largest gain (ties: the
 *             smallest a, then the smallest b, a < b) while some gain is
 *             positive, at most max_swaps times.  (The pages mention further
 *             devices for leaving local optima without describing them; they
 *             are not implemented.)
 * All comparisons are on exact integers, so results do not depend on the
 * order of any addition.  Shapes: the rules above, plus cols <= 32768 and
 * rows <= 2^24. */

/* shift_out (device int32 [1]) = the fixed-point shift of W, or INT32_MIN
 * when W holds an infinity or NaN. */
maskllm_status maskllm_perm_shift(const uint16_t* W, int64_t rows, int64_t cols,
                                  int32_t* shift_out, maskllm_stream_t stream);

/* metric_out (device uint64 [1]) = the fixed-point metric of perm, with the
 * shift read from the device int32 *shift (normally maskllm_perm_shift's
 * output).  An entry of perm outside [0, cols) reads as a zero weight and
 * makes the next maskllm_device_status() return MASKLLM_ERR_INVALID_ARG. */
maskllm_status maskllm_perm_metric(const uint16_t* W, int64_t rows, int64_t cols,
                                   const int32_t* perm, const int32_t* shift,
                                   uint64_t* metric_out, maskllm_stream_t stream);

/* W_out[r, i] = W[r, perm[i]] (bf16 [rows, cols]); out-of-range entries as for
 * maskllm_perm_metric (the element is written as +0). */
maskllm_status maskllm_permute_columns(const uint16_t* W, int64_t rows, int64_t cols,
                                       const int32_t* perm, uint16_t* W_out,
                                       maskllm_stream_t stream);

/* Device scratch the two calls below need, in bytes (0 for a shape outside
 * the rules): a [cols, cols] and two [rows, cols] uint32 tables, 8 bytes
 * per 32 x 32 tile of the first's upper triangle, and a few hundred bytes of
 * control.  The caller owns it; it holds nothing between
 * calls. */
int64_t maskllm_perm_workspace_bytes(int64_t rows, int64_t cols);

/* gains_out (device int64 [cols, cols], symmetric) = gain(a, b) of every pair
 * of slots under perm.  info_out (device int32 [1]) = 0, or -1 when perm is
 * not a permutation of 0..cols-1, or -2 when W holds an infinity or NaN (then
 * gains_out is not written).  shift_out (device int32 [1], nullable) = the
 * shift used. */
maskllm_status maskllm_perm_swap_gains(const uint16_t* W, int64_t rows, int64_t cols,
                                       const int32_t* perm, void* workspace,
                                       int64_t workspace_bytes, int64_t* gains_out,
                                       int32_t* info_out, int32_t* shift_out,
                                       maskllm_stream_t stream);

/* The search, from the permutation in perm (device int32 [cols], updated in
 * place).  Swap s is logged in swaps_out[2s], swaps_out[2s+1] (the slots a <
 * b; device int32 [max_swaps, 2], nullable) and gains_out[s] (device int64
 * [max_swaps], nullable).  n_swaps_out (device int32 [1]) = the number of
 * swaps applied, or -1 / -2 as info_out above (then perm is unchanged).
 * shift_out as above.  max_swaps >= 0 steps are enqueued without any
 * synchronisation; once no swap gains, the remaining steps return at once
 * (a few microseconds each). */
maskllm_status maskllm_perm_search(const uint16_t* W, int64_t rows, int64_t cols, int32_t* perm,
                                   int32_t max_swaps, void* workspace, int64_t workspace_bytes,
                                   int32_t* swaps_out, int64_t* gains_out,
                                   int32_t* n_swaps_out, int32_t* shift_out,
                                   maskllm_stream_t stream);

/* ---- 2:4 sparse x dense product ------------------------------------------
 * "Accelerating Sparse Deep Neural Networks", Sec. 3.2: the sparse tensor
 * core multiplies a 2:4 sparse first operand by a dense second operand into
 * a dense result, skipping the zeros (twice the math rate of the dense
 * product); Sec. 3.1: the sparse operand is stored as its kept values plus
 * 2-bit positions.
 *
 *   C[m, n] = sum over k of A[m, k] * B[n, k]      (C = A B^T)
 *
 *   values  in   bf16 [M, K/2] and
 *   meta    in   u32 [M, K/32]: A in the layout maskllm_hard_compress writes
 *                (group g of row m keeps values[m, 2g], values[m, 2g+1] at
 *                positions i < j given by the 4-bit code i | j << 2 at bits
 *                4(g % 8) of meta[m, g / 8]); codes must name two distinct
 *                positions (the six candidates)
 *   B       in   bf16 [N, K] row-major (for a linear layer: the N input rows)
 *   C       out  fp32 [M, N] row-major
 * Products are exact in fp32; they are summed in fp32 on the tensor cores in
 * an order of their own.  M, N >= 1, K >= 32, K % 32 == 0, M, N < 2^31,
 * K < 2^31, N <= 65535 * 256.  C is written by bulk tensor stores when
 * N % 4 == 0 and row by row otherwise.  A bounded wait that gives up makes the next
 * maskllm_device_status() return MASKLLM_ERR_TIMEOUT; MASKLLM_ERR_CUDA if the
 * driver cannot describe the operands to the copy engine. */
maskllm_status maskllm_spmm(const uint16_t* values, const uint32_t* meta, int64_t M, int64_t K,
                            const uint16_t* B, int64_t N, float* C, maskllm_stream_t stream);

/* ---- Permutation search without caller memory ---------------------------
 * Not part of the method: the papers have no counterpart.  Some callers
 * cannot hand the library device memory: code that must not call
 * cudaMalloc (or any allocator) at the point where it runs the search, for
 * example a runtime that has reserved all device memory up front for its own
 * pool, or a host program with no allocator of device memory of its own.
 * For them, maskllm_perm_search_static runs maskllm_perm_search with its
 * scratch in an array that the library itself holds in device memory:
 * MASKLLM_PERM_SEARCH_STATIC_BYTES bytes, held by every GPU that loads the
 * library until the process exits.  It allocates nothing and frees nothing.
 *
 * Arguments, results and outcome codes are those of maskllm_perm_search
 * without workspace and workspace_bytes.  A shape whose
 * maskllm_perm_workspace_bytes() exceeds MASKLLM_PERM_SEARCH_STATIC_BYTES
 * (for example cols = 1024 with rows above 3583, or cols = 2048 with rows
 * above 1022) returns MASKLLM_ERR_SHAPE and launches nothing.
 *
 * Every call looks up the array's device address on the current device
 * afresh, so a cudaDeviceReset or a re-created context between calls is
 * safe.  The first call on a device may load the library's device code;
 * make it before any stream capture begins: a first call made while
 * `stream` is capturing returns MASKLLM_ERR_INVALID_ARG and launches
 * nothing.  Every call on a device shares the one array: each call zeroes what
 * must start at zero and overwrites the rest, so nothing carries over from
 * the previous call, but calls that overlap on the GPU (other streams, other
 * host threads) race on the array and give wrong results.  Issue them in
 * order, on one stream or with synchronisation between them. */
#define MASKLLM_PERM_SEARCH_STATIC_BYTES (32LL * 1024 * 1024)

maskllm_status maskllm_perm_search_static(const uint16_t* W, int64_t rows, int64_t cols,
                                          int32_t* perm, int32_t max_swaps, int32_t* swaps_out,
                                          int64_t* gains_out, int32_t* n_swaps_out,
                                          int32_t* shift_out, maskllm_stream_t stream);

/* The forward and the convergence diagnostics of one step in a single pass
 * (MaskLLM Fig. 5; the optional outputs of maskllm_forward): every output
 * is bit-identical to that of maskllm_forward (W_out, row_sq_out) or
 * maskllm_mask_stats (idx_out, l1_row_out, maxprob_row_out) for the same
 * step: the row sums are added in the same order.  The noisy logits z the
 * forward forms give the draws, so the
 * diagnostics cost no second pass over the logits: 2 bytes of traffic per
 * group (0.5 per weight) more than the forward (the draws out, the previous
 * draws in).
 *   W, logits, W_out, row_sq_out   as maskllm_forward (row_sq_out nullable)
 *   prev_idx, idx_out, l1_row_out, maxprob_row_out   as maskllm_mask_stats
 *                                  (all nullable; l1_row_out needs prev_idx)
 * cols <= 2^24. */
maskllm_status maskllm_forward_stats(const uint16_t* W, const float* logits,
                                     const uint8_t* prev_idx, int64_t rows, int64_t cols,
                                     float tau, float kappa, maskllm_rng rng, uint16_t* W_out,
                                     float* row_sq_out, uint8_t* idx_out, uint32_t* l1_row_out,
                                     float* maxprob_row_out, maskllm_stream_t stream);

/* The backward and the convergence diagnostics of one step in a single pass
 * (MaskLLM Fig. 5; the same quantities as maskllm_forward_stats, for a
 * caller that wants them from the backward): every output is bit-identical
 * to that of maskllm_backward (dlogits_out) or maskllm_mask_stats (idx_out,
 * l1_row_out, maxprob_row_out) for the same step.  The backward regenerates
 * the step's noisy logits z, which give the draws, so the diagnostics need
 * no second pass over the logits: 2 bytes of traffic per group (0.5 per
 * weight) more than the backward, and their arithmetic.
 *   W, logits, grad_W_out, reg_coeff, dlogits_out   as maskllm_backward
 *   prev_idx, idx_out, l1_row_out, maxprob_row_out   as maskllm_mask_stats
 *                                  (all nullable; l1_row_out needs prev_idx)
 * cols <= 2^24. */
maskllm_status maskllm_backward_stats(const uint16_t* W, const float* logits,
                                      const uint16_t* grad_W_out, const uint8_t* prev_idx,
                                      int64_t rows, int64_t cols, float tau, float kappa,
                                      maskllm_rng rng, float reg_coeff, float* dlogits_out,
                                      uint8_t* idx_out, uint32_t* l1_row_out,
                                      float* maxprob_row_out, maskllm_stream_t stream);

/* ---- Batched calls ------------------------------------------------------
 * One launch processes up to MASKLLM_MAX_BATCH matrices (for example the
 * seven linears of a transformer block); longer lists are split into several
 * launches.  The work of the whole batch is spread over the GPU as one
 * stream of row chunks, so small matrices do not each pay a launch and a
 * pipeline ramp.  Per-matrix results are identical to the single-matrix
 * calls.  Each matrix is described by a maskllm_matrix; a call reads only
 * the fields of its own operation (the others are ignored), and every rule
 * of the single-matrix call applies to each matrix.  Outputs may not overlap
 * any input or output of any matrix in the batch. */
#define MASKLLM_MAX_BATCH 16

typedef struct {
  const uint16_t* W;          /* bf16 [rows, cols] (all operations but prior_from_mask) */
  const float* logits;        /* fp32 [rows, cols/4, 6] (forward, backward, compress) */
  const uint16_t* grad_W_out; /* bf16 [rows, cols] (backward) */
  int64_t rows;
  int64_t cols;
  uint32_t tensor_id;         /* noise counter word 3 (forward, backward) */
  float* logits_out;          /* prior_init output */
  uint16_t* W_out;            /* forward output */
  float* row_sq_out;          /* forward output, nullable */
  float* probs_out;           /* forward output, nullable */
  float* dlogits_out;         /* backward output */
  uint16_t* values_out;       /* hard_compress output */
  uint32_t* meta_out;         /* hard_compress output */
  uint8_t* idx_out;           /* hard_compress output, nullable */
  const uint32_t* meta;       /* prior_from_mask input: 4-bit codes u32 [rows, cols/32]
                                 (logits_out is its output; W is not read) */
  const uint8_t* prev_idx;    /* mask_stats, forward_stats, backward_stats input: the
                                 previous step's draws, u8 [rows, cols/4], nullable */
  uint32_t* l1_row_out;       /* diagnostics output, nullable (needs prev_idx) */
  float* maxprob_row_out;     /* diagnostics output, nullable */
} maskllm_matrix;

/* n >= 1 matrices; the noise of matrix i uses (seed, step, mats[i].tensor_id). */
maskllm_status maskllm_prior_init_batched(const maskllm_matrix* mats, int32_t n, float scale,
                                          maskllm_stream_t stream);
maskllm_status maskllm_forward_batched(const maskllm_matrix* mats, int32_t n, float tau,
                                       float kappa, uint64_t seed, uint32_t step,
                                       maskllm_stream_t stream);
maskllm_status maskllm_backward_batched(const maskllm_matrix* mats, int32_t n, float tau,
                                        float kappa, uint64_t seed, uint32_t step,
                                        float reg_coeff, maskllm_stream_t stream);
maskllm_status maskllm_hard_compress_batched(const maskllm_matrix* mats, int32_t n,
                                             maskllm_stream_t stream);
/* maskllm_prior_from_mask over a batch (MaskLLM Table 2): reads meta, writes
 * logits_out of every matrix; high and low as in the single call. */
maskllm_status maskllm_prior_from_mask_batched(const maskllm_matrix* mats, int32_t n, float high,
                                               float low, maskllm_stream_t stream);
/* maskllm_mask_stats over a batch (MaskLLM Fig. 5): reads logits and
 * prev_idx, writes idx_out (the draws), l1_row_out and maxprob_row_out of
 * every matrix; W is not read (rows and cols still describe the matrix). */
maskllm_status maskllm_mask_stats_batched(const maskllm_matrix* mats, int32_t n, float tau,
                                          float kappa, uint64_t seed, uint32_t step,
                                          maskllm_stream_t stream);
/* maskllm_forward_stats over a batch: reads W, logits and prev_idx, writes
 * W_out, row_sq_out, idx_out (the draws), l1_row_out and maxprob_row_out. */
maskllm_status maskllm_forward_stats_batched(const maskllm_matrix* mats, int32_t n, float tau,
                                             float kappa, uint64_t seed, uint32_t step,
                                             maskllm_stream_t stream);
/* maskllm_backward_stats over a batch: reads W, logits, grad_W_out and
 * prev_idx, writes dlogits_out, idx_out (the draws), l1_row_out and
 * maxprob_row_out. */
maskllm_status maskllm_backward_stats_batched(const maskllm_matrix* mats, int32_t n, float tau,
                                              float kappa, uint64_t seed, uint32_t step,
                                              float reg_coeff, maskllm_stream_t stream);

/* ---- Failure detection -------------------------------------------------
 * The pipelined kernels wait on shared-memory barriers for their bulk copies.
 * Every such wait gives up after `nanoseconds` (default 2 s); the kernel then
 * sets the device error word (see maskllm_device_status), waits up to
 * max(nanoseconds, 1 s) for its own copies still in flight, and returns.
 * Applies to launches issued after the call (host-global setting). */
maskllm_status maskllm_set_wait_timeout(uint64_t nanoseconds);

/* Test hook for the timeout path: while enabled (nonzero), the pipelined
 * kernels issue no copies at all, so their consumers' waits run out and the
 * next maskllm_device_status() returns MASKLLM_ERR_TIMEOUT.  Results of
 * launches issued while enabled are invalid.  Host-global setting. */
maskllm_status maskllm_test_withhold_loads(int32_t enable);

/* Test hook for the sparse product (maskllm_spmm): a tile of C is 256 rows by
 * a width the library picks per call from 256, 224, 192, 160, 128 columns
 * against the number of tile waves.  n = 128..256, a multiple of 32, makes
 * every later call use width n; n = 0 restores the choice per call.  Results
 * are the same for every width (up to the fp32 summation order the tensor
 * cores use).  MASKLLM_ERR_INVALID_ARG for any other n.  Host-global
 * setting. */
maskllm_status maskllm_test_spmm_tile_n(int32_t n);

/* Waits for `stream`, then reads and clears the library's device error words
 * on the current device.  Returns MASKLLM_ERR_TIMEOUT if a bounded wait inside
 * a kernel gave up since the last call (its results are then invalid),
 * else MASKLLM_ERR_INVALID_ARG if a permutation entry was out of range,
 * MASKLLM_ERR_CUDA if the wait itself failed, MASKLLM_OK otherwise. */
maskllm_status maskllm_device_status(maskllm_stream_t stream);

/* Human-readable name of a status code (static storage). */
const char* maskllm_status_string(maskllm_status status);

/* The CUDA error message of the last MASKLLM_ERR_CUDA returned to this host
 * thread, or "" (thread-local static storage). */
const char* maskllm_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MASKLLM_H_ */
