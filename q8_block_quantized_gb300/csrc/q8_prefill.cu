// q8_prefill.cu -- the prefill tile GEMM: M activation rows (the tokens of a
// prompt) against packed Q8_0 weights, each 128-row weight tile reused
// across 128 activation rows (Ferro README, "Exactness contract": prefill
// rows always take the tile GEMM; "How the iGPU path is fast", item 1: int8
// block dots, activations quantized per 32-block).
//
// One CTA computes one 128 (weight rows) x 128 (activation rows) output
// tile at a time, persistent over the tiles.  Per 32-block b:
//   - the worker warps convert the block's int8 quants of both operands to
//     fp16 (exact) in the no-swizzle K-major layout of the tensor cores;
//   - one thread issues two tcgen05.mma (K = 16 each) into a 128 x 128 fp32
//     accumulator in tensor memory: every entry is the exact integer block
//     dot isum_b (|isum| <= 516128 < 2^24);
//   - the worker warps read the accumulator back (tcgen05.ld) and fold it
//     into their rows' sums in the fixed order below, on the CUDA cores.
// The MMA of block b runs while the workers convert block b + 1's operands
// and fold block b - 1 (two accumulators, two operand buffers; a fold two
// blocks behind with three of each measured slower).
//
// Fixed order of one output y[m][n] (the same whatever M is and wherever
// row m sits in the launch, so a prompt filled in slices equals the prompt
// filled at once):
//   s_b   = fp32(d_w[n][b] * d_a[m][b])
//   sigma = fma(isum_b, s_b, sigma) over the blocks of a segment of 16
//           (in order, from +0)
//   Y     = Y + sigma over the segments (in order, from +0)
// This is not the decode GEMV's tree; both are within the tolerance of the
// exact sum, the prefill order within (17 + ceil(NB/16)) u S for u = 2^-24.
#include <cuda_runtime.h>

#include <mutex>

#include "q8_device.cuh"
#include "q8_internal.h"

namespace q8 {
namespace {

constexpr int PF_TN = Q8_PREFILL_TILE_ROWS;  // weight rows per tile: MMA M, tensor-memory lanes
constexpr int PF_TM = Q8_PREFILL_TILE_ROWS;  // activation rows per tile: MMA N
constexpr int PF_SEG = Q8_PREFILL_SEGMENT;   // blocks per segment of the summation order
constexpr int PF_NW = 8;                     // worker warps
constexpr int PF_WT = PF_NW * 32;            // worker threads
constexpr int PF_THREADS = PF_WT + 32;       // + one producer warp
constexpr int PF_STAGES = 2;
constexpr int PF_CHUNK = MAX_TILE_ROWS * CHUNK_BLOCKS * BLOCK_BYTES;  // 34816: one chunk of 128 rows
constexpr int PF_STAGE = 2 * PF_CHUNK;                                // weights, then activations
constexpr int PF_SLICE = 128 * 16 * 2;  // fp16 operand of one MMA: 128 rows x 16 k
constexpr int PF_OPS = 4 * PF_SLICE;    // one block: weight halves 0, 1; activation halves 0, 1
constexpr int PF_NBUF = 2;              // accumulators and operand buffers in flight
constexpr int PF_DA_BUFS = PF_NBUF + 1; // activation scales: written at conversion, read a block later
constexpr uint32_t PF_TMEM_COLS = 512;  // accumulators of two blocks (128 columns each), then the sums Y
constexpr uint32_t PF_Y_COL = PF_NBUF * PF_TM;
constexpr size_t PF_OFF_OPS = (size_t)PF_STAGES * PF_STAGE;
constexpr size_t PF_OFF_DA = PF_OFF_OPS + (size_t)PF_NBUF * PF_OPS;
constexpr size_t PF_OFF_BAR = PF_OFF_DA + (size_t)PF_DA_BUFS * PF_TM * sizeof(float);
constexpr size_t PF_SMEM = PF_OFF_BAR + (2 * PF_STAGES + PF_NBUF + 1) * sizeof(uint64_t) + 4 * sizeof(int);
static_assert(PF_Y_COL + PF_TM <= PF_TMEM_COLS, "tensor-memory columns");
static_assert(PF_OFF_OPS % 1024 == 0, "operand buffers aligned");
static_assert(PF_SMEM <= 232448, "shared memory per CTA");
static_assert(PF_TN == 128 && PF_TM == 128, "one MMA shape: M = N = 128");

enum : unsigned { ERR_PF_PRODUCER = 8u, ERR_PF_WORKER = 16u, ERR_PF_DRAIN = 32u };

struct PrefillArgs {
  const uint8_t* W;  // packed weights, tiles of RW rows
  const uint8_t* A;  // packed activations, tiles of 128 rows
  float* y;          // [M][N]
  int64_t N, M, NB, nch;
  int64_t tn, tm, tiles;  // output tiles along N, along M, in all
  int RW;
  unsigned* err;
};

// The 16 fp16 values of quants q (one row, 16 consecutive k) at dst and
// dst + 128: two core matrices along K of the no-swizzle K-major layout
// (row r of an operand at (r / 8) * 256 + (r % 8) * 16).
__device__ __forceinline__ void put_f16_row(uint8_t* dst, uint4 q) {
  uint32_t o[8];
  i8x4_to_h2x2(q.x, o[0], o[1]);
  i8x4_to_h2x2(q.y, o[2], o[3]);
  i8x4_to_h2x2(q.z, o[4], o[5]);
  i8x4_to_h2x2(q.w, o[6], o[7]);
  *reinterpret_cast<uint4*>(dst) = make_uint4(o[0], o[1], o[2], o[3]);
  *reinterpret_cast<uint4*>(dst + 128) = make_uint4(o[4], o[5], o[6], o[7]);
}

__device__ __forceinline__ float half_at(const uint8_t* p) {
  return __half2float(*reinterpret_cast<const __half*>(p));
}

// Producer (one thread): per tile and chunk, the chunk of the 128/RW weight
// tiles and of the activation tile, each one bulk copy (a ragged tail of
// under 16 bytes by hand), completing on full[stage].
__device__ __forceinline__ void pf_produce(const PrefillArgs& a, uint8_t* smem, uint64_t* full,
                                           uint64_t* empty, volatile int* misc) {
  const uint64_t pol_w = l2_policy_evict_normal();  // other CTAs read the same weight tile
  const uint64_t pol_a = l2_policy_evict_last();    // every weight tile's CTA reads it
  const int G = PF_TN / a.RW;
  int stage = 0;
  uint32_t phase = 0;
  int issued = 0;
  for (int64_t T = blockIdx.x; T < a.tiles; T += gridDim.x) {
    const int64_t nt = T / a.tm, mt = T - (T / a.tm) * a.tm;
    const int ra = tile_rows(mt, a.M, PF_TM);
    for (int64_t c = 0; c < a.nch; ++c) {
      if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, WAIT_LIMIT_NS)) {
        atomicOr(a.err, ERR_PF_PRODUCER);
        misc[3] = 1;
        return;
      }
      const int kb = chunk_blocks(c, a.NB);
      uint8_t* dst = smem + (size_t)stage * PF_STAGE;
      for (int g = 0; g <= G; ++g) {  // g < G: weight tiles; g == G: the activation tile
        const uint8_t* src;
        uint8_t* d;
        uint32_t bytes;
        uint64_t pol;
        if (g < G) {
          const int64_t tw = nt * G + g;
          if (tw * a.RW >= a.N) continue;
          const int rw = tile_rows(tw, a.N, a.RW);
          src = a.W + chunk_offset(tw, c, rw, a.RW, a.NB);
          d = dst + (size_t)g * a.RW * CHUNK_BLOCKS * BLOCK_BYTES;
          bytes = (uint32_t)(kb * rw * BLOCK_BYTES);
          pol = pol_w;
        } else {
          src = a.A + chunk_offset(mt, c, ra, PF_TM, a.NB);
          d = dst + PF_CHUNK;
          bytes = (uint32_t)(kb * ra * BLOCK_BYTES);
          pol = pol_a;
        }
        const uint32_t bulk = bytes & ~15u;
        for (uint32_t k = bulk; k < bytes; ++k) d[k] = src[k];
        if (bulk) {
          mbar_expect_tx(&full[stage], bulk);
          bulk_g2s(d, src, bulk, &full[stage], pol);
        }
      }
      mbar_arrive(&full[stage]);
      misc[1] = ++issued;
      if (++stage == PF_STAGES) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
}

__global__ void __launch_bounds__(PF_THREADS, 1) prefill_kernel(const PrefillArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + PF_OFF_BAR);
  uint64_t* empty = full + PF_STAGES;
  uint64_t* mma_bar = empty + PF_STAGES;
  // misc[0]: the workers' abort flag (written and read only by workers);
  // misc[1]: chunks issued; misc[2]: tensor-memory base; misc[3]: producer stopped
  volatile int* misc = reinterpret_cast<volatile int*>(mma_bar + PF_NBUF + 1);
  float* da_s = reinterpret_cast<float*>(smem + PF_OFF_DA);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < PF_STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], PF_NW);
    }
    for (int p = 0; p < PF_NBUF; ++p) mbar_init(&mma_bar[p], 1);
    misc[0] = 0;
    misc[1] = 0;
    misc[3] = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(reinterpret_cast<uint32_t*>(const_cast<int*>(misc + 2)), PF_TMEM_COLS);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = static_cast<uint32_t>(misc[2]);
  pdl_launch_dependents();
  pdl_wait();  // activations and y belong to the previous work on the stream

  // worker state that the drain at the end needs (thread 0's copy)
  int consumed = 0;
  uint32_t pending = 0u;  // bit p: an MMA into accumulator p not yet waited for
  uint32_t mph = 0u;      // bit p: parity of accumulator p's next MMA completion

  if (warp == PF_NW) {
    if (lane == 0) pf_produce(a, smem, full, empty, misc);
    __syncwarp();
  } else {
    // thread (warp w, lane l): weight row `row` of the tile = tensor-memory
    // lane 32 (w % 4) + l, which it also converts; columns [64 hf, 64 hf + 64)
    // of the accumulators; half hf of each block's 32 quants when converting
    const int row = tid & (PF_TN - 1);
    const int hf = tid >> 7;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int G = PF_TN / a.RW;
    const int g = row / a.RW, ii = row - g * a.RW;
    const uint32_t IDESC = umma_idesc_f16(PF_TN, PF_TM);
    int stage = 0;
    uint32_t sphase = 0;
    int64_t bc = 0;  // blocks this CTA has issued, over all its tiles
    bool dead = false;

    for (int64_t T = blockIdx.x; T < a.tiles && !dead; T += gridDim.x) {
      const int64_t nt = T / a.tm, mt = T - (T / a.tm) * a.tm;
      const int ra = tile_rows(mt, a.M, PF_TM);
      const int64_t tw = nt * G + g;
      const int rw = tw * a.RW < a.N ? tile_rows(tw, a.N, a.RW) : 0;
      const bool wv = ii < rw;  // this row exists (n < N)
      uint64_t sig[32];         // sigma of columns 64 hf + 2e, + 2e + 1
#pragma unroll
      for (int e = 0; e < 32; ++e) sig[e] = 0ull;
      bool first_seg = true;
      // the block whose accumulator is still to be read
      int64_t q1_blk = -1;
      int q1_pb = 0, q1_d = 0;
      float q1_dw = 0.0f;

      // Fold the accumulator of block b (buffer pb, activation scales d3,
      // weight scale dw) into sigma; at a segment's end into Y; at the
      // tile's end store Y.  Warp-uniform control flow throughout.
      auto fold = [&](int64_t b, int pb, int d3, float dw) {
        bool ok = mbar_wait_bounded(&mma_bar[pb], (mph >> pb) & 1u, WAIT_LIMIT_NS);
        if (!ok) {
          atomicOr(a.err, ERR_PF_WORKER);
          misc[0] = 1;
        }
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {
          mph ^= 1u << pb;
          pending &= ~(1u << pb);
        }
        tc_fence_after_sync();
        if (!ok) return;
        const float* dap = da_s + d3 * PF_TM + hf * 64;
        const uint64_t dw2 = f2_pack(dw, dw);
        const uint32_t acc = tmem + lane_base + (uint32_t)(pb * PF_TM + hf * 64);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          uint32_t u0[16], u1[16];
          tmem_ld16(acc + q * 32, u0);
          tmem_ld16(acc + q * 32 + 16, u1);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float4 d4 = *reinterpret_cast<const float4*>(dap + q * 32 + 4 * e);
            const uint32_t* u = e < 4 ? u0 : u1;
            const int k = (e & 3) * 4;
            const uint64_t s01 = f2_mul(dw2, f2_pack(d4.x, d4.y));
            const uint64_t s23 = f2_mul(dw2, f2_pack(d4.z, d4.w));
            sig[q * 16 + 2 * e] = f2_fma(f2_pack(__uint_as_float(u[k]), __uint_as_float(u[k + 1])), s01,
                                         sig[q * 16 + 2 * e]);
            sig[q * 16 + 2 * e + 1] = f2_fma(f2_pack(__uint_as_float(u[k + 2]), __uint_as_float(u[k + 3])), s23,
                                             sig[q * 16 + 2 * e + 1]);
          }
        }
        const bool last = b == a.NB - 1;
        if (!last && (b + 1) % PF_SEG != 0) return;
        // end of a segment: Y = Y + sigma (Y = +0 + sigma for the first)
        const uint32_t ycol = tmem + lane_base + PF_Y_COL + (uint32_t)(hf * 64);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t yv[16];
          if (first_seg) {
#pragma unroll
            for (int k = 0; k < 16; ++k) yv[k] = 0u;
          } else {
            tmem_ld16(ycol + q * 16, yv);
            tmem_ld_wait();
          }
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const uint64_t y2 = f2_add(f2_pack(__uint_as_float(yv[2 * e]), __uint_as_float(yv[2 * e + 1])),
                                       sig[q * 8 + e]);
            float lo, hi;
            f2_unpack(y2, lo, hi);
            yv[2 * e] = __float_as_uint(lo);
            yv[2 * e + 1] = __float_as_uint(hi);
            sig[q * 8 + e] = 0ull;
          }
          if (last) {
            const int64_t n = nt * PF_TN + row;
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              const int m = hf * 64 + q * 16 + k;
              if (wv && m < ra) a.y[(mt * PF_TM + m) * a.N + n] = __uint_as_float(yv[k]);
            }
          } else {
            tmem_st16(ycol + q * 16, yv);
          }
        }
        if (!last) tmem_st_wait();
        first_seg = false;
      };

      for (int64_t c = 0; c < a.nch && !dead; ++c) {
        const bool got = mbar_wait_bounded(&full[stage], sphase, WAIT_LIMIT_NS);
        if (got) {
          ++consumed;  // chunks whose copies have landed
        } else {
          atomicOr(a.err, ERR_PF_WORKER);
          misc[0] = 1;
        }
        const int kb = chunk_blocks(c, a.NB);
        const uint8_t* cw = smem + (size_t)stage * PF_STAGE + (size_t)g * a.RW * CHUNK_BLOCKS * BLOCK_BYTES;
        const uint8_t* ca = smem + (size_t)stage * PF_STAGE + PF_CHUNK;
        for (int j = 0; j < kb; ++j) {
          const int pb = (int)(bc % PF_NBUF), d3 = (int)(bc % PF_DA_BUFS);
          uint8_t* ops = smem + PF_OFF_OPS + (size_t)pb * PF_OPS;
          float dw = 0.0f;
          if (got) {
            const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
            const uint4 qw = wv ? lds128(cw + chunk_quant_off(j, hf, ii, rw)) : zero;
            put_f16_row(ops + hf * PF_SLICE + (row >> 3) * 256 + (row & 7) * 16, qw);
            const uint4 qa = row < ra ? lds128(ca + chunk_quant_off(j, hf, row, ra)) : zero;
            put_f16_row(ops + (2 + hf) * PF_SLICE + (row >> 3) * 256 + (row & 7) * 16, qa);
            if (hf == 0) da_s[d3 * PF_TM + row] = row < ra ? half_at(ca + chunk_scale_off(j, row, ra, kb)) : 0.0f;
            dw = wv ? half_at(cw + chunk_scale_off(j, ii, rw, kb)) : 0.0f;
          }
          if (j == kb - 1) {  // this warp has read all it needs of the stage
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stage]);
          }
          fence_proxy_async_smem();
          tc_fence_before_sync();
          named_bar_sync(1, PF_WT);
          if (misc[0] != 0) {  // read after the barrier: the same in every worker
            dead = true;
            break;
          }
          if (tid == 0) {
            tc_fence_after_sync();
#pragma unroll
            for (int h = 0; h < 2; ++h)
              umma_f16(tmem + (uint32_t)(pb * PF_TM),
                       umma_smem_desc(smem_u32(ops + h * PF_SLICE), 128, 256),
                       umma_smem_desc(smem_u32(ops + (2 + h) * PF_SLICE), 128, 256), IDESC, h == 1);
            umma_commit(&mma_bar[pb]);
          }
          pending |= 1u << pb;
          if (q1_blk >= 0) fold(q1_blk, q1_pb, q1_d, q1_dw);
          q1_blk = c * CHUNK_BLOCKS + j;
          q1_pb = pb;
          q1_d = d3;
          q1_dw = dw;
          ++bc;
        }
        if (dead) break;
        if (++stage == PF_STAGES) {
          stage = 0;
          sphase ^= 1u;
        }
      }
      if (!dead && q1_blk >= 0) fold(q1_blk, q1_pb, q1_d, q1_dw);
    }
  }

  __syncthreads();
  if (tid == 0 && (misc[0] != 0 || misc[3] != 0)) {
    // stopped early: let the MMAs and copies in flight land before the
    // tensor memory and the CTA's shared memory are given back
    for (int p = 0; p < PF_NBUF; ++p)
      if (((pending >> p) & 1u) && !mbar_wait_bounded(&mma_bar[p], (mph >> p) & 1u, WAIT_LIMIT_NS))
        atomicOr(a.err, ERR_PF_DRAIN);
    const int issued = misc[1];
    for (int k = consumed; k < issued; ++k)
      if (!mbar_wait_bounded(&full[k % PF_STAGES], (uint32_t)((k / PF_STAGES) & 1), WAIT_LIMIT_NS))
        atomicOr(a.err, ERR_PF_DRAIN);
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, PF_TMEM_COLS);
  }
}

std::mutex g_pf_mu;
bool g_pf_attr[64] = {};

}  // namespace

cudaError_t launch_prefill(const DeviceInfo& dev, const uint8_t* W, int64_t N, int64_t K, const uint8_t* A_packed,
                           int64_t M, float* y, bool pdl, cudaStream_t s) {
  cudaError_t e;
  {
    std::lock_guard<std::mutex> lk(g_pf_mu);
    if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
    if (!g_pf_attr[dev.device]) {
      e = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)PF_SMEM);
      if (e != cudaSuccess) return e;
      g_pf_attr[dev.device] = true;
    }
  }
  unsigned* err = nullptr;
  if ((e = device_error_word(dev.device, &err)) != cudaSuccess) return e;
  PrefillArgs a;
  a.W = W;
  a.A = A_packed;
  a.y = y;
  a.N = N;
  a.M = M;
  a.NB = K / QK;
  a.nch = (a.NB + CHUNK_BLOCKS - 1) / CHUNK_BLOCKS;
  a.RW = layout_tile_rows(N);
  a.tn = (N + PF_TN - 1) / PF_TN;
  a.tm = (M + PF_TM - 1) / PF_TM;
  a.tiles = a.tn * a.tm;
  a.err = err;
  const int64_t grid = a.tiles < dev.sm_count ? a.tiles : dev.sm_count;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(PF_THREADS);
  cfg.dynamicSmemBytes = PF_SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, prefill_kernel, a);
}

}  // namespace q8
