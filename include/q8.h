/*
 * q8.h -- C ABI of libq8, the Q8_0 block-quantized decode product on one
 * NVIDIA GB300 (sm_103a).
 *
 * What is computed (sources are web pages, cited by title and section):
 *
 *   Q8_0 block: one fp16 scale d followed by 32 int8 quants q, 34 bytes
 *   ("Ember: packed Q8 decode", the row-contiguous source figure, which shows
 *   each row's block as a scale and then the quants q0..q31; and the
 *   packed-tile figure, whose 544-byte record holds exactly 16 blocks).  Byte 0..1: d, IEEE binary16, little-endian;
 *   bytes 2..33: q[0..31] as two's-complement int8.
 *
 *   Activations are quantized once per 32-wide block ("Ferro" README, "How
 *   the iGPU path is fast", item 1), and one quantization is shared by every
 *   projection that reads the same input (Ember, the paragraph on the runtime
 *   pass before the packed layout: Q/K/V share one, gate/up share one).  Rounding rule (the
 *   llama.cpp-style scheme the Ferro README names; the pages do not spell it
 *   out): d = amax / 127 in fp32, q_i = roundf(x_i * (1/d)) with ties away
 *   from zero and 1/d taken from the fp32 d, scale stored as binary16 rounded
 *   to nearest even; amax == 0 gives d = 0 and q = 0.
 *
 *   y[m][n] = sum over blocks b of  isum(n,m,b) * d_w[n][b] * d_a[m][b],
 *   isum = sum_{i<32} q_w[n][b][i] * q_a[m][b][i] computed exactly in int32
 *   (Ferro, item 1: int8 DP4A dot products over per-32-block activations).
 *
 *   Batch invariance (Ferro README, "Exactness, scheduling and operations",
 *   "Exactness contract": a decode row gets the same result whatever else is
 *   batched with it).  Each block term is rounded once in fp32 as
 *   t_b = float(isum) * (float(d_w) * float(d_a)), where the inner product of
 *   two binary16 values is exact in fp32, and the terms are summed in fp32 in
 *   one fixed order: the pairwise tree over the block index b, padded with
 *   zeros to the next power of two.  The result for (m, n) therefore depends
 *   only on row n of W, row m of the activations and K: it is bitwise the
 *   same for every M, every position of the row in the batch, every split of
 *   the work and every kernel path.
 *
 * Conventions for every call:
 *   - Pointers named W, A_blocks, x, y, workspace, src/dst are DEVICE
 *     pointers owned by the caller (allocated on the current device); the
 *     library never frees or retains them after the call returns.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls are asynchronous on that stream; a return of Q8_OK means
 *     the work was enqueued, not that it finished.
 *   - Arguments are checked on the host before anything is enqueued; on any
 *     error nothing is launched and the status says why.  Q8_ECUDA means a
 *     CUDA runtime call failed (cudaGetLastError is left set).
 *   - K must be a positive multiple of 32.  Row counts are positive.
 *   - The library owns no device memory and allocates none in these calls.
 *   - Only sm_103 devices are accepted (Q8_EDEVICE otherwise).
 *   - There is no CPU fallback.
 */
#ifndef Q8_H
#define Q8_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define Q8_API __attribute__((visibility("default")))
#else
#define Q8_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define Q8_QK 32            /* values per block                               */
#define Q8_BLOCK_BYTES 34   /* bytes per block: fp16 scale + 32 int8          */
#define Q8_MAX_M 4096       /* most activation rows per q8_gemm call          */
#define Q8_MAX_DOTS_M 64    /* most activation rows per q8_block_dots call    */
#define Q8_MAX_TILE_ROWS 128 /* packed layout: most output rows per tile       */
#define Q8_CHUNK_BLOCKS 8   /* packed layout: blocks per chunk                */
#define Q8_PREFILL_TILE_ROWS 128 /* prefill GEMM: weight rows and activation
                                    rows of one output tile                  */
#define Q8_PREFILL_SEGMENT 16 /* prefill GEMM: blocks per segment of its
                                 summation order (see q8_gemm_prefill)       */
#define Q8_MAX_PREFILL_K 65536 /* prefill GEMM: largest K                     */

/* Flags for the compute calls. */
#define Q8_FLAG_PDL 1u      /* launch as a programmatic dependent of the
                               previous work on the stream (see q8_gemm)     */
#define Q8_FLAG_TCGEN05 2u  /* q8_gemm / q8_fused_quant_gemm: block dots on
                               the tcgen05 tensor cores (see q8_gemm)        */

typedef enum q8_status {
    Q8_OK = 0,
    Q8_EINVAL = -1,      /* null pointer or bad flag                          */
    Q8_ESHAPE = -2,      /* K not a positive multiple of 32, M or N out of range */
    Q8_EALIGN = -3,      /* a pointer is not aligned as documented            */
    Q8_EDEVICE = -4,     /* current device is not sm_103                      */
    Q8_ECUDA = -5,       /* a CUDA runtime call failed                        */
    Q8_EWORKSPACE = -6,  /* workspace missing or smaller than required        */
    Q8_ETIMEOUT = -7,    /* (q8_device_error only) a device wait gave up      */
    Q8_ESCRATCH = -8     /* (q8_gemm_noalloc only) shape needs more scratch
                            than the built-in Q8_NOALLOC_SCRATCH_BYTES         */
} q8_status;

/* Human-readable name of a status code.  Static string, never NULL. */
Q8_API const char *q8_strerror(int status);

/* ABI version of this header/library pair: 1. */
Q8_API int q8_abi_version(void);

/* Bytes of `rows` rows of K/32 row-contiguous Q8_0 blocks: rows*(K/32)*34. */
Q8_API size_t q8_blocks_bytes(int64_t rows, int64_t K);

/* Bytes of the packed weight layout for an N x K matrix.  Equal to
 * q8_blocks_bytes(N, K): repacking moves bytes, it adds none (Ember's packed
 * tile is likewise exactly the size of the blocks it holds). */
Q8_API size_t q8_packed_bytes(int64_t N, int64_t K);

/* Rows per tile of the packed layout of an N-row matrix (16, 32, 64 or
 * 128; see q8_repack_weights).  Returns 0 for N <= 0. */
Q8_API int q8_packed_tile_rows(int64_t N);

/* Workspace bytes q8_gemm / q8_fused_quant_gemm need for this shape on the
 * current device: partial sums when the work is split along K, and from 16
 * rows per launch the activations staged once per call for every CTA; 0
 * when neither applies.  Returns 0 for invalid shapes. */
Q8_API size_t q8_workspace_bytes(int64_t N, int64_t K, int M);

/*
 * q8_quantize_act -- quantize fp32 activations to Q8_0 blocks.
 * (Ferro README, "How the iGPU path is fast", item 1; rounding rule above.)
 *
 *   x          [M][K] fp32, row-major, 4-byte aligned.
 *   M          rows, 1 <= M <= 2^31-1 (also used to quantize weight rows).
 *   K          positive multiple of 32.
 *   out_blocks [M][K/32] blocks of 34 bytes, row-contiguous; 2-byte aligned;
 *              q8_blocks_bytes(M, K) bytes.
 *   flags      0 or Q8_FLAG_PDL.
 * Bit-exact with the rule above for finite inputs; NaN/Inf inputs and scales
 * beyond the binary16 range (amax > 65504*127) are outside the contract.
 */
Q8_API int q8_quantize_act(const float *x, int64_t M, int64_t K, void *out_blocks,
                    unsigned flags, void *stream);

/*
 * Fused producers: the step before a GEMV, emitting its activation blocks
 * directly (Ferro README, "How the iGPU path is fast", item 3: the residual
 * add, the norm and the int8 quantization in one pass; SwiGLU emits the next
 * GEMM's int8 input).  The pages give no arithmetic for these steps; the
 * readings below are single-precision operations with one IEEE rounding
 * each (sqrt and division correctly rounded), so the output is bit-exact
 * and reproducible anywhere.  Both end in the rounding rule of
 * q8_quantize_act.
 */

/*
 * q8_residual_rmsnorm_quantize -- h = x + delta (or x when delta is NULL);
 * y = RMSNorm(h) * gamma as in the Llama family; out_blocks = q8_quantize_act(y).
 *
 *   s  = sum over k of h_k * h_k, added as the pairwise tree over k (leaves
 *        padded with zeros to the next power of two);
 *   ms = s / K;  r = 1 / sqrt(ms + eps);  y_k = (h_k * r) * gamma_k.
 *
 *   x, delta   [M][K] fp32, 16-byte aligned (delta may be NULL).
 *   gamma      [K] fp32, 16-byte aligned.
 *   eps        positive and finite (else Q8_EINVAL).
 *   M          rows, 1 <= M <= 2^31-1; K a positive multiple of 32,
 *              K <= Q8_MAX_NORM_K.
 *   h_out      optional [M][K] fp32 (16-byte aligned) receiving h, the new
 *              residual stream; it may be x or delta (in-place update).
 *   out_blocks [M][K/32] blocks, 2-byte aligned.
 *   flags      0 or Q8_FLAG_PDL.
 * One CTA per row.  Inputs whose squares overflow are outside the contract.
 */
#define Q8_MAX_NORM_K (1 << 24)
Q8_API int q8_residual_rmsnorm_quantize(const float *x, const float *delta, const float *gamma,
                                        float eps, int64_t M, int64_t K, float *h_out,
                                        void *out_blocks, unsigned flags, void *stream);

/*
 * q8_swiglu_quantize -- h = silu(gate) * up, out_blocks = q8_quantize_act(h).
 *
 *   gate_up    [M][2F] fp32, 16-byte aligned: gate in columns [0, F), up in
 *              [F, 2F) (the output of one GEMV over the concatenated gate
 *              and up weights).
 *   F          positive multiple of 32.
 *   out_blocks [M][F/32] blocks, 2-byte aligned.
 *   flags      0 or Q8_FLAG_PDL.
 * silu(g) = g / (1 + e^-g).  e^x is a fixed procedure (Cody and Waite's
 * reduction, then a Taylor polynomial), identical wherever it runs; fma is
 * a fused multiply-add (one rounding):
 *   x > 88: +inf;  x < -87: 0;  otherwise n = rint(x * L2E),
 *   r = fma(-n, LN2_LO, fma(-n, LN2_HI, x)),
 *   p = C7, then p = fma(p, r, c) for c = C6, C5, C4, C3, 1/2, 1, 1,
 *   e^x = p * 2^n,
 * with L2E = 0x1.715476p+0 (1/ln 2), LN2_HI = 0x1.63p-1 (355/512),
 * LN2_LO = -0x1.bd0106p-13 (ln 2 - 355/512), C3..C7 = 1/3!..1/7! rounded to
 * single precision (0x1.555556p-3, 0x1.555556p-5, 0x1.111112p-7,
 * 0x1.6c16c2p-10, 0x1.a01a02p-13); within 0.7 ulp of e^x.
 */
Q8_API int q8_swiglu_quantize(const float *gate_up, int64_t M, int64_t F, void *out_blocks,
                              unsigned flags, void *stream);

/*
 * q8_repack_weights -- move row-contiguous Q8_0 weight blocks into the packed
 * layout the GEMV streams.  A one-time step (Ember repacks each layer's projection
 * weights once at load time into 16-row tiles; Ferro keeps its device weights
 * in a coalesced block-major, row-minor layout, item 1).
 *
 *   src_blocks [N][K/32] blocks (34 bytes each), 2-byte aligned.
 *   dst        q8_packed_bytes(N, K) bytes, 16-byte aligned; must not
 *              overlap src.
 *
 * Packed layout (same bytes, new order).  Rows are grouped in tiles of R
 * rows, R = q8_packed_tile_rows(N): the smallest of 16, 32, 64 for which the
 * tile count ceil(N/R) is at most 152 (about one tile per SM of a GB300),
 * else 128.  The last tile holds r = N - R*t rows.  Blocks are grouped in
 * chunks of 8 (the last chunk holds kb = K/32 - 8*c blocks).  Tile t starts
 * at byte R*t*(K/32)*34; inside it chunk c starts at byte r*8*c*34 and holds,
 * for j < kb, h < 2, i < r, the 16 quants q[R*t+i][8c+j][16h..16h+15] at byte
 * ((2j+h)*r+i)*16, followed by the kb*r scales, scale (j, i) at byte
 * kb*r*32 + (j*r+i)*2.  Every chunk starts on a 16-byte boundary of dst, and
 * the chunks of a tile are contiguous, so a kernel streams each chunk with
 * one bulk copy.
 */
Q8_API int q8_repack_weights(const void *src_blocks, int64_t N, int64_t K, void *dst,
                      void *stream);

/*
 * q8_gemm -- y = W (Q8_0, packed) times the quantized activations.
 * (Ferro item 1; Ferro README, "Using LFM2.5 language models": decode batches
 * of one to four tokens run a GEMV split along K; the exactness contract
 * above.)
 *
 *   W         packed weights from q8_repack_weights, 16-byte aligned.
 *   N         output rows, 1 <= N <= 2^31-1.
 *   K         positive multiple of 32.
 *   A_blocks  [M][K/32] activation blocks (q8_quantize_act), 2-byte aligned.
 *   M         activation rows, 1 <= M <= Q8_MAX_M.  Decode batches (up to
 *             32 rows) run in one launch; more rows run as launches of 32
 *             rows, each streaming W again, with the same per-row
 *             arithmetic, so a prefill row is bitwise the row decoded alone
 *             (Ferro README, "Exactness contract": a row's result does not
 *             depend on the other rows of the launch).  For many rows,
 *             q8_gemm_prefill reuses each weight tile across 128 rows (its
 *             own per-row order, not bitwise the decoded row).
 *   y         [M][N] fp32 output, row-major, 4-byte aligned; overwritten.
 *   workspace q8_workspace_bytes(N, K, M) bytes (may be NULL when that is 0),
 *             16-byte aligned.  Its first 16384 bytes hold per-tile tickets
 *             and must be zero before the first call that uses it; every
 *             call leaves them zero when it completes, and the rest of the
 *             workspace is scratch.  One workspace (sized for the largest
 *             shape) can therefore serve any sequence of calls on one stream;
 *             calls that may run at the same time must not share one.  After
 *             q8_device_error reports a failure, zero it again.
 *   flags     0 or Q8_FLAG_PDL.  With Q8_FLAG_PDL the kernel is launched as a
 *             programmatic dependent of the previous work on `stream` and
 *             starts streaming W before that work has finished; it waits for
 *             it before reading A_blocks or writing y/workspace.  The caller
 *             promises that no unfinished earlier work on the stream writes W.
 *             Q8_FLAG_TCGEN05 (alone or with Q8_FLAG_PDL): on matrices packed
 *             in 128-row tiles, passes of 9-16 activation rows compute their
 *             block dots with tcgen05 MMAs (int8 converted exactly to fp16,
 *             fp32 accumulators in tensor memory, one per block) instead of
 *             the default mma.sync tensor path; other shapes ignore it.  The
 *             result is bitwise the same.  It is measured slower on GB300
 *             (each round converts the weights to fp16 in shared memory and
 *             reads every block's accumulator back from tensor memory, one
 *             step after the other) and kept for comparison.
 */
Q8_API int q8_gemm(const void *W, int64_t N, int64_t K, const void *A_blocks, int M,
            float *y, void *workspace, size_t workspace_bytes, unsigned flags,
            void *stream);

/*
 * q8_fused_quant_gemm -- quantize fp32 activations inside the GEMV, then the
 * product (Ferro item 3: the producing kernels emit the next GEMM's int8 input; the
 * README also measures GEMVs with the quantization fused into their
 * prologue).  Every CTA quantizes the activation blocks it
 * needs with the same rule as q8_quantize_act, bit for bit, so
 * y equals q8_gemm(W, q8_quantize_act(x)) bitwise.
 *
 *   x            [M][K] fp32, row-major, 16-byte aligned.
 *   A_blocks_out optional (may be NULL): receives q8_quantize_act(x), for
 *                reuse by a later GEMV that reads the same input; 2-byte
 *                aligned, q8_blocks_bytes(M, K) bytes.
 *   Other arguments as q8_gemm.
 */
Q8_API int q8_fused_quant_gemm(const void *W, int64_t N, int64_t K, const float *x,
                        int M, float *y, void *A_blocks_out, void *workspace,
                        size_t workspace_bytes, unsigned flags, void *stream);

/*
 * q8_gemm_swiglu / q8_fused_quant_gemm_swiglu -- the gate/up GEMV with SwiGLU
 * in its epilogue: it writes the quantized input of the down projection,
 * q8_quantize_act(silu(gate) * up), instead of y (Ferro README, "How the iGPU
 * path is fast", item 3: SwiGLU emits the next GEMM's int8 input directly).
 * One launch replaces the GEMV and q8_swiglu_quantize.  silu and the
 * rounding are those of q8_swiglu_quantize, applied to the outputs this GEMV
 * computes (bitwise those of q8_gemm / q8_fused_quant_gemm on the same W).
 *
 *   W          packed (q8_repack_weights) N = 2F rows of K, 16-byte aligned,
 *              whose rows are gate and up interleaved in groups of G =
 *              q8_packed_tile_rows(2F) / 2 rows: for every g, rows
 *              [2gG, 2gG + G) are gate rows [gG, gG + G) and rows
 *              [2gG + G, 2gG + 2G) are up rows [gG, gG + G).
 *   F          outputs per row of h; q8_packed_tile_rows(2F) must be 64 or
 *              128 and F a multiple of G, else Q8_ESHAPE.
 *   K, M       as q8_gemm; the product must not need a split along K for
 *              this M (true for F >= 2432 with 64-row tiles, F >= 4864
 *              with 128-row tiles, and K <= 8192), else Q8_ESHAPE.
 *   A_blocks / x  the activations, as q8_gemm / q8_fused_quant_gemm.
 *   out_blocks [M][F/32] blocks of h (2-byte aligned).
 *   flags      0 or Q8_FLAG_PDL.  No workspace is needed.
 */
Q8_API int q8_gemm_swiglu(const void *W, int64_t F, int64_t K, const void *A_blocks, int M,
                          void *out_blocks, unsigned flags, void *stream);
Q8_API int q8_fused_quant_gemm_swiglu(const void *W, int64_t F, int64_t K, const float *x, int M,
                                      void *out_blocks, unsigned flags, void *stream);

/*
 * q8_gemm_noalloc -- q8_gemm without a workspace argument, for callers that
 * cannot allocate device memory (for example a plugin inside an application
 * whose own allocator owns the device, or a latency-critical loop that must
 * not pay cudaMalloc's latency and implicit synchronization).  The pages have
 * no counterpart; it is a packaging variant of q8_gemm and computes the same
 * bits.
 *
 * What q8_gemm keeps in its workspace (partial sums of a split along K, the
 * activations staged once per call) goes to a scratch array of
 * Q8_NOALLOC_SCRATCH_BYTES compiled into the library: it occupies that much
 * memory on every GPU that loads the library, until the process exits.
 * Neither this call nor the library allocates anything.  When the staged
 * activations would not fit, the call stages them in every CTA instead (the
 * same bits); shapes whose split alone needs more scratch return
 * Q8_ESCRATCH before anything is enqueued (q8_workspace_bytes(N, K, M) is an
 * upper bound of the size; 0 means no scratch is used and any size works).
 *
 * Every call shares the one array and it keeps the last call's contents:
 * calls that may run at the same time on the GPU (other streams, other host
 * threads) race on it and must be serialized by the caller.  Each split call
 * first clears the array's ticket area with an asynchronous memset on
 * `stream`; on those shapes Q8_FLAG_PDL therefore overlaps the kernel with
 * the memset, not with the caller's previous kernel.  The first call on a
 * device looks up the array's device address (cudaGetSymbolAddress, with
 * that device current) and keeps it; make that first call before any stream
 * capture, and do not use the library across a cudaDeviceReset of that
 * device (the address belongs to the context that looked it up).
 *
 * flags is 0 or Q8_FLAG_PDL (the tcgen05 option is not offered here).
 * Arguments, alignment and errors otherwise as q8_gemm.
 */
#define Q8_NOALLOC_SCRATCH_BYTES (4u << 20)
Q8_API int q8_gemm_noalloc(const void *W, int64_t N, int64_t K, const void *A_blocks,
                           int M, float *y, unsigned flags, void *stream);

/*
 * q8_gemm_prefill / q8_fused_quant_gemm_prefill -- the prefill tile GEMM:
 * y = W (Q8_0, packed) times M activation rows (the tokens of a prompt),
 * each 128-row weight tile reused across 128 activation rows.  (Ferro
 * README, "Exactness contract": prefill rows always take the tile GEMM, so
 * a row's arithmetic does not depend on how many rows share the launch, and
 * a prompt filled in slices equals the prompt filled at once; "How the iGPU
 * path is fast", item 1: int8 block dots of Q8_0 weights and activations
 * quantized per 32-block.)
 *
 * Every output is the same function of its two rows, whatever M is and
 * wherever the row sits: with isum_b the exact int32 dot of block b,
 * s_b = fp32(d_w[n][b] * d_a[m][b]) (both binary16 scales widened to fp32),
 *   sigma = +0; sigma = fma(isum_b, s_b, sigma) for the blocks b of one
 *           segment of Q8_PREFILL_SEGMENT consecutive blocks, in order;
 *   of the nseg segments the first ceil(nseg/2) form the low half, the
 *   rest the high half:
 *   Y_lo = +0; Y_lo = Y_lo + sigma for the low half's segments, in order;
 *   Y_hi = +0; Y_hi = Y_hi + sigma for the high half's segments, in order;
 *   y[m][n] = Y_lo + Y_hi.
 * (IEEE single precision, round to nearest even, fma rounded once.)  The
 * two halves let a launch with few output tiles (at most half as many as
 * the GPU has SMs) split every tile along K over two CTAs without changing
 * any bit; the low half's CTA then waits, bounded, for the high half's, so
 * if other work keeps the launch's CTAs from all being resident at once the
 * call reports a timeout through q8_device_error instead of hanging.  This
 * is not the decode order of q8_gemm, so a prefill row is not bitwise the
 * decoded row; both are within the library's tolerance of the exact sum:
 * here |y - exact| <= (17 + ceil(K/512)) * 2^-24 * S with S the sum of the
 * block terms' magnitudes, below 1e-5 * S for K <= Q8_MAX_PREFILL_K.
 *
 *   W          packed weights from q8_repack_weights, 16-byte aligned.
 *   N          output rows, 1 <= N <= 2^31-1.
 *   K          positive multiple of 32, at most Q8_MAX_PREFILL_K.
 *   A_blocks   [M][K/32] activation blocks (q8_quantize_act), 2-byte aligned
 *              (q8_gemm_prefill).
 *   x          [M][K] fp32 activations, 4-byte aligned, quantized first
 *              exactly as q8_quantize_act does (q8_fused_quant_gemm_prefill).
 *   M          activation rows, >= 1; ceil(N/128) * ceil(M/128) output
 *              tiles at most 2^31 - 1 (else Q8_ESHAPE).
 *   y          [M][N] fp32 output, row-major, 4-byte aligned; overwritten.
 *   A_blocks_out  (fused call only, may be NULL) receives the [M][K/32]
 *              blocks of x, 2-byte aligned.
 *   workspace  16-byte aligned, at least q8_prefill_workspace_bytes(K, M)
 *              bytes, not overlapping the other buffers: it receives 4096
 *              bytes of flags for tiles split along K (cleared by the call
 *              itself), the activation blocks packed in 128-row tiles and,
 *              in the fused call without A_blocks_out, the blocks of x.
 *              Scratch only; calls that may run at the same time must not
 *              share one.
 *   flags      0 or Q8_FLAG_PDL (the first launch is a programmatic
 *              dependent of the previous work on the stream; the call waits
 *              for that work before it reads anything).
 * A call is two launches (three when fused): pack (quantize), GEMM.
 */
Q8_API size_t q8_prefill_workspace_bytes(int64_t K, int M);
Q8_API int q8_gemm_prefill(const void *W, int64_t N, int64_t K, const void *A_blocks, int M,
                           float *y, void *workspace, size_t workspace_bytes, unsigned flags,
                           void *stream);
Q8_API int q8_fused_quant_gemm_prefill(const void *W, int64_t N, int64_t K, const float *x, int M,
                                       float *y, void *A_blocks_out, void *workspace,
                                       size_t workspace_bytes, unsigned flags, void *stream);

/*
 * q8_kv_quantize / q8_kv_dequantize -- the int8 KV cache codec ("Ferro"
 * README, "Exactness, scheduling and operations (LM serving)", item "KV
 * cache": K/V rows stored as int8 with one fp32 scale per 32 values, the
 * q8_0 scheme of llama.cpp applied to the cache; written by the cache-write
 * step, dequantized where attention reads the cache).
 *
 * Codebook: for each 32-value block, d = amax / 127 in fp32 and q_i =
 * roundf(x_i * (1/d)) with 1/d from the fp32 d -- the quants are exactly
 * those q8_quantize_act gives the same block -- but the scale is kept as the
 * fp32 d itself (not rounded to binary16).  Dequantization: x'_i = q_i * d,
 * one single-precision multiply (round to nearest even).
 *
 * Cache layout (caller-owned device memory, q8_kv_cache_bytes(capacity, D)
 * bytes in two planes): quants int8 [capacity][D], row s of slot s; scales
 * fp32 [capacity][D/32], scale b of slot s covers quants 32b..32b+31 of
 * that slot.  36 bytes per 32 values.
 *
 *   x          [rows][D] fp32 K or V rows (e.g. one token's row of all KV
 *              heads of a layer), 16-byte aligned.
 *   rows       1 <= rows <= 2^31 - 1.
 *   D          positive multiple of 32, at most Q8_MAX_KV_D.
 *   slots      device int32 [rows], 4-byte aligned: the cache slot of each
 *              row (a paged cache's slot map), or NULL for slot = row.  A slot
 *              outside [0, capacity) is skipped: nothing is written for that
 *              row (q8_kv_dequantize writes zeros for it), and
 *              q8_device_error then reports (-Q8_ESHAPE) << 8 | 8.
 *   capacity   slots in the cache, 1 <= capacity <= 2^31 - 1.
 *   cache_q, cache_d  the planes, 4-byte aligned.  Rows given the same slot
 *              in one call race (any one of them may win, block by block).
 *   out        [rows][D] fp32 (q8_kv_dequantize), 16-byte aligned: row r is
 *              the dequantized slot slots[r].
 *   flags      0 or Q8_FLAG_PDL.
 * The written quants and scales, and the dequantized values, are bit-exact
 * with the rule above for finite inputs.
 */
#define Q8_MAX_KV_D (1 << 24)
Q8_API size_t q8_kv_cache_bytes(int64_t capacity, int64_t D);
Q8_API int q8_kv_quantize(const float *x, int64_t rows, int64_t D, const int32_t *slots,
                          int64_t capacity, int8_t *cache_q, float *cache_d, unsigned flags,
                          void *stream);
Q8_API int q8_kv_dequantize(const int8_t *cache_q, const float *cache_d, int64_t capacity,
                            int64_t D, const int32_t *slots, int64_t rows, float *out,
                            unsigned flags, void *stream);

/* ---- test hooks (not on the hot path) ----------------------------------- */

/* Inverse of q8_repack_weights: packed (16-byte aligned) -> [N][K/32] blocks
 * (2-byte aligned). */
Q8_API int q8_unpack_weights(const void *packed, int64_t N, int64_t K,
                      void *dst_blocks, void *stream);

/* Exact per-block int32 dots from packed W and activation blocks:
 * isum[m][n][b] (int32, [M][N][K/32], 4-byte aligned), 1 <= M <= Q8_MAX_DOTS_M. */
Q8_API int q8_block_dots(const void *W, int64_t N, int64_t K, const void *A_blocks,
                  int M, int32_t *isum, void *stream);

/* Read and clear the device-side error word of the current device (waits for
 * the device).  *code = 0 when no kernel reported a failure; otherwise a
 * status byte shifted left by 8 ORed with what happened where: 1 a GEMV's
 * copy stream, 2 a GEMV's consumers, 4 a GEMV's drain of copies in flight;
 * 16 the prefill GEMM's worker warps, 32 its drain, 64 its MMA issuer, 128
 * its copy issuer -- each a bounded device wait (2 s) that gave up, status
 * -Q8_ETIMEOUT; 8 a KV codec row whose slot lay outside the cache (that row
 * skipped), status -Q8_ESHAPE when it is the only bit.  A kernel whose wait
 * gave up stops its work and returns; its outputs are undefined.  Returns a
 * status. */
Q8_API int q8_device_error(unsigned *code);

/* Test hook: the time limit, in ns, of the decode GEMV kernels' waits on
 * their copy ring (the weight stream and, with 9 or more rows, the
 * activation staging), for every launch enqueued after this call; 0
 * restores the default of 2 s.  A kernel whose wait gives up reports it in
 * q8_device_error, stops, lets the copies it issued land (with the full 2 s
 * bound, whatever the limit), and returns; its outputs are undefined.  Lets
 * a test make the failure path run without any fault.  Process-wide; not
 * for use while other threads launch GEMVs.  Returns Q8_OK. */
Q8_API int q8_set_wait_limit_ns(uint64_t ns);

/* Properties the library uses: SM count and compute capability of the
 * current device. */
Q8_API int q8_device_info(int *sm_count, int *cc_major, int *cc_minor);

#ifdef __cplusplus
}
#endif

#endif /* Q8_H */
