// q8_prefill.cu -- the prefill tile GEMM: M activation rows (the tokens of a
// prompt) against packed Q8_0 weights, each 128-row weight tile reused
// across 128 activation rows (Ferro README, "Exactness contract": prefill
// rows always take the tile GEMM; "How the iGPU path is fast", item 1: int8
// block dots, activations quantized per 32-block).
//
// One CTA computes one 128 (weight rows) x 128 (activation rows) output
// tile at a time, persistent over the tiles.  Per 32-block b:
//   - the worker warps convert the block's int8 quants of both operands to
//     fp16 (exact) in the no-swizzle K-major layout of the tensor cores, and
//     the activation scales d_a to fp32 in shared memory;
//   - one thread issues two tcgen05.mma (K = 16 each) into a 128 x 128 fp32
//     accumulator in tensor memory: every entry is the exact integer block
//     dot isum_b (|isum| <= 516128 < 2^24);
//   - the worker warps read the accumulator back (tcgen05.ld) and fold it
//     into their rows' sums in the fixed order below: per output and block
//     one multiply (d_w d_a, exact) and one fma, two outputs per f32x2 op.
// The MMA of block b runs while the workers convert block b + 1 and fold
// block b - 1 (two accumulators, two operand buffers).  Tensor memory: the
// two accumulators and the segment sums Y (384 of 512 columns).  Warp
// roles: 8 worker warps (two warpgroups, 216 registers each after
// setmaxnreg) convert and fold; in a third warpgroup (72 registers) one
// thread issues a block's MMAs once all 8 workers have converted it, and
// another issues the bulk copies of a chunk into a stage once all 8 have
// converted the last block of the chunk it held.  Only mbarriers connect
// them; a CTA-wide barrier per block and a single thread issuing both MMAs
// and copies measured 1.6x slower, as did the scale products by a rank-1
// MMA (its accumulator fits only once, which chained each block's MMA
// latency behind the previous block's fold).
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
#include "q8_f32x2.cuh"
#include "q8_internal.h"

namespace q8 {
namespace {

// ---- helpers only this kernel uses (PTX wrappers) ----------------------------
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// A warp reads 16 consecutive 32-bit tensor-memory columns of its 32 lanes
// (tcgen05.ld; taddr: first lane in bits 31..16, column below), or stores
// them (tcgen05.st).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u32(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

constexpr int PF_TN = Q8_PREFILL_TILE_ROWS;  // weight rows per tile: MMA M, tensor-memory lanes
constexpr int PF_TM = Q8_PREFILL_TILE_ROWS;  // activation rows per tile: MMA N
constexpr int PF_SEG = Q8_PREFILL_SEGMENT;   // blocks per segment of the summation order
constexpr int PF_NW = 8;                     // worker warps (warpgroups 0 and 1)
constexpr int PF_WT = PF_NW * 32;
constexpr int PF_THREADS = PF_WT + 128;      // + warpgroup 2: MMA issuer, copy issuer, two idle warps
// Registers: launched at 65536 / 384 = 168 per thread; warpgroup 2 gives
// back down to 72, the workers take 216: per SM sub-partition
// 2 x 32 x 216 + 32 x 72 = 16128 <= 16384, in all
// 256 x 216 + 128 x 72 = 64512 = 384 x 168.
constexpr int PF_REG_LAUNCH = 168, PF_REG_WORKER = 216, PF_REG_ISSUER = 72;
static_assert(PF_WT * PF_REG_WORKER + 128 * PF_REG_ISSUER <= PF_THREADS * PF_REG_LAUNCH, "register split");
constexpr int PF_STAGES = 2;
constexpr int PF_CHUNK = MAX_TILE_ROWS * CHUNK_BLOCKS * BLOCK_BYTES;  // 34816: one chunk of 128 rows
constexpr int PF_STAGE = 2 * PF_CHUNK;                                // weights, then activations
constexpr int PF_SLICE = 128 * 16 * 2;  // fp16 operand of one MMA: 128 rows x 16 k
constexpr int PF_OPS = 4 * PF_SLICE;    // one block: weight halves 0, 1; activation halves 0, 1
constexpr int PF_NBUF = 2;              // accumulators and operand buffers in flight
// fp32 activation scales of a block: written at its conversion, read at its
// fold a block later; a warp can be at most three blocks ahead of another
constexpr int PF_DA_BUFS = 4;
constexpr uint32_t PF_Y_COL = PF_NBUF * PF_TM;  // the running sum Y of the current half
constexpr uint32_t PF_YLO_COL = PF_Y_COL + PF_TM;  // the low half's sum, kept for the end
constexpr uint32_t PF_TMEM_COLS = 512;
constexpr size_t PF_OFF_OPS = (size_t)PF_STAGES * PF_STAGE;
constexpr size_t PF_OFF_DA = PF_OFF_OPS + (size_t)PF_NBUF * PF_OPS;
constexpr size_t PF_OFF_BAR = PF_OFF_DA + (size_t)PF_DA_BUFS * PF_TM * sizeof(float);
constexpr size_t PF_SMEM = PF_OFF_BAR + (2 * PF_STAGES + 2 * PF_NBUF) * sizeof(uint64_t) + 4 * sizeof(int);
static_assert(PF_OFF_OPS % 1024 == 0, "operand buffers aligned");
static_assert(PF_SMEM <= 232448, "shared memory per CTA");
static_assert(PF_TN == 128 && PF_TM == 128, "one MMA shape: M = N = 128");
static_assert(PF_YLO_COL + PF_TM <= PF_TMEM_COLS, "tensor-memory columns");
// A launch with few output tiles splits each along K into its low and high
// half (two CTAs): the high half's CTA stores its sums into y and raises one
// flag per worker warp; the low half's CTA adds them to its own.  The flags
// (PF_FLAG_BYTES at the start of the workspace) are cleared by the pack
// kernel that precedes every GEMM launch.
constexpr int PF_FLAG_TILES = 128;  // split tiles at most (8 flags of 4 bytes each)
static_assert(PF_FLAG_TILES * 8 * 4 <= PREFILL_FLAG_BYTES, "split flags fit the workspace's flag area");

enum : unsigned { ERR_PF_WORKER = 16u, ERR_PF_DRAIN = 32u, ERR_PF_ISSUER = 64u, ERR_PF_PRODUCER = 128u };

struct PrefillArgs {
  const uint8_t* W;  // packed weights, tiles of RW rows
  const uint8_t* A;  // packed activations, tiles of 128 rows
  float* y;          // [M][N]
  unsigned* flags;   // split: [tile][8 worker warps], zero at the start
  int64_t N;
  int M, NB, nch;
  int tm, tiles;     // output tiles along M, in all (< 2^31, checked on the host)
  int RW;
  int split;         // 1, or 2: item = (tile, half), one item per CTA
  int h;             // segments of the low half: ceil(nseg / 2)
  unsigned* err;
};

// The chunks of item T (tile T / split, half T % split): all of K, or the
// low half's segments (2 chunks each) or the rest.
__device__ __forceinline__ void pf_item(const PrefillArgs& a, int T, int& tile, int& part, int& c0, int& c1) {
  tile = T / a.split;
  part = T - tile * a.split;
  const int cm = a.h * (Q8_PREFILL_SEGMENT / CHUNK_BLOCKS);
  c0 = (a.split == 2 && part == 1) ? cm : 0;
  c1 = (a.split == 2 && part == 0) ? cm : a.nch;
}

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

// Chunk c of tile (nt, mt) into stage `stage`: the chunk of each of the
// 128/RW weight tiles and of the activation tile, one bulk copy each (a
// ragged tail under 16 bytes by hand), completing on full[stage].
__device__ __noinline__ void pf_issue(const PrefillArgs& a, uint8_t* smem, uint64_t* full, int nt, int mt, int c,
                                      int stage) {
  const int ra = tile_rows(mt, a.M, PF_TM);
  const int kb = chunk_blocks(c, a.NB);
  const int G = PF_TN / a.RW;
  uint8_t* dst = smem + (size_t)stage * PF_STAGE;
  const uint64_t pol_w = l2_policy_evict_normal();  // the other m-tiles' CTAs read the same weights
  const uint64_t pol_a = l2_policy_evict_last();    // every weight tile's CTA reads the activations
  for (int g = 0; g <= G; ++g) {  // g < G: weight tiles; g == G: the activation tile
    const uint8_t* src;
    uint8_t* d;
    uint32_t bytes;
    uint64_t pol;
    if (g < G) {
      const int64_t tw = (int64_t)nt * G + g;
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
    for (uint32_t i = bulk; i < bytes; ++i) d[i] = src[i];
    if (bulk) {
      mbar_expect_tx(&full[stage], bulk);
      bulk_g2s(d, src, bulk, &full[stage], pol);
    }
  }
  mbar_arrive(&full[stage]);
}

// The copy issuer: this CTA's chunks in order, chunk k into stage k % 2
// once the 8 workers have released the stage (chunk k - 2 converted).
__device__ __forceinline__ void pf_producer(const PrefillArgs& a, uint8_t* smem, uint64_t* full, uint64_t* empty,
                                            volatile int* misc) {
  uint32_t k = 0;
  for (int T = blockIdx.x; T < a.tiles * a.split; T += gridDim.x) {
    int tile, part, c0, c1;
    pf_item(a, T, tile, part, c0, c1);
    const int nt = tile / a.tm, mt = tile - nt * a.tm;
    for (int c = c0; c < c1; ++c, ++k) {
      const int stage = (int)(k & 1u);
      if (misc[0] != 0 || !mbar_wait_bounded(&empty[stage], ((k >> 1) & 1u) ^ 1u, WAIT_LIMIT_NS)) {
        if (misc[0] == 0) atomicOr(a.err, ERR_PF_PRODUCER);
        misc[0] = 1;
        misc[1] = (int)k;  // copies issued
        return;
      }
      pf_issue(a, smem, full, nt, mt, c, stage);
    }
  }
  misc[1] = (int)k;
}

// The MMA issuer: per block, once the 8 workers have arrived on opready
// (operands converted, and their fold of the block two back, which used the
// same accumulator, done), the block's two MMAs and their commit.
__device__ __forceinline__ void pf_issuer(const PrefillArgs& a, uint8_t* smem, uint64_t* opready, uint64_t* mma_bar,
                                          volatile int* misc, uint32_t tmem) {
  const uint32_t IDESC = umma_idesc_f16(PF_TN, PF_TM);
  uint32_t b = 0;           // blocks issued (only its low bits are used)
  uint32_t mma_issued = 0;  // bit p: parity of accumulator p's MMAs so far; bit 2 + p: any
  bool stop = false;
  for (int T = blockIdx.x; T < a.tiles * a.split && !stop; T += gridDim.x) {
    int tile, part, c0, c1;
    pf_item(a, T, tile, part, c0, c1);
    for (int c = c0; c < c1 && !stop; ++c) {
      const int kb = chunk_blocks(c, a.NB);
      for (int j = 0; j < kb; ++j, ++b) {
        const int pb = (int)(b & 1u);
        if (misc[0] != 0 || !mbar_wait_bounded(&opready[pb], (b >> 1) & 1u, WAIT_LIMIT_NS)) {
          if (misc[0] == 0) atomicOr(a.err, ERR_PF_ISSUER);
          misc[0] = 1;
          stop = true;
          break;
        }
        tc_fence_after_sync();
        uint8_t* ops = smem + PF_OFF_OPS + (size_t)pb * PF_OPS;
#pragma unroll
        for (int h = 0; h < 2; ++h)
          umma_f16(tmem + (uint32_t)(pb * PF_TM), umma_smem_desc(smem_u32(ops + h * PF_SLICE), 128, 256),
                   umma_smem_desc(smem_u32(ops + (2 + h) * PF_SLICE), 128, 256), IDESC, h == 1);
        umma_commit(&mma_bar[pb]);
        mma_issued = (mma_issued ^ (1u << pb)) | (4u << pb);
      }
    }
  }
  if (misc[0] != 0) {
    // stopped early: let the MMAs in flight land before the tensor memory
    // is given back (the last MMA on accumulator p completes the phase of
    // parity bit p ^ 1)
    for (int p = 0; p < PF_NBUF; ++p)
      if (((mma_issued >> (2 + p)) & 1u) &&
          !mbar_wait_bounded(&mma_bar[p], ((mma_issued >> p) & 1u) ^ 1u, WAIT_LIMIT_NS))
        atomicOr(a.err, ERR_PF_DRAIN);
  }
}

// The outputs of one closing half (one warp; its thread holds weight row n
// and 64 consecutive activation rows of the tile: yp = &y[m0][n], stepped by
// N; mleft of them exist).  v = this half's sums (tensor memory at yc):
//   add_lo:  y = Y_lo (tensor memory at yl) + v;
//   combine: y = v + the other CTA's high-half sums, read from y once its
//            warp's flag is up (false if it does not come);
//   publish: y = v, then the flag;  otherwise y = v.
__device__ __noinline__ bool pf_outputs(uint32_t yc, uint32_t yl, float* yp, int64_t N, int mleft, bool add_lo,
                                        bool combine, bool publish, unsigned* flag) {
  const int lane = threadIdx.x & 31;
  if (combine) {
    bool ready = true;
    if (lane == 0) {
      const uint64_t t0 = globaltimer_ns();
      while (ld_acquire_u32(flag) == 0u) {
        if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
          ready = false;
          break;
        }
      }
    }
    if (__shfl_sync(0xffffffffu, ready ? 1 : 0, 0) == 0) return false;
  }
#pragma unroll 1
  for (int q = 0; q < 8; ++q) {
    uint32_t v[8], lv[8];
    tmem_ld8(yc + q * 8, v);
    if (add_lo) tmem_ld8(yl + q * 8, lv);
    tmem_ld_wait();
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      float o = __uint_as_float(v[k]);
      if (add_lo) o = __fadd_rn(__uint_as_float(lv[k]), o);  // Y_lo + Y_hi
      const bool in = q * 8 + k < mleft;
      if (combine && in) o = __fadd_rn(o, __ldcg(yp));  // Y_lo + Y_hi, Y_hi from the other CTA
      if (in) *yp = o;
      yp += N;
    }
  }
  if (publish) {
    __syncwarp();
    if (lane == 0) {
      __threadfence();
      st_release_u32(flag, 1u);
    }
  }
  return true;
}

__global__ void __launch_bounds__(PF_THREADS, 1) prefill_kernel(const PrefillArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + PF_OFF_BAR);
  uint64_t* empty = full + PF_STAGES;
  uint64_t* opready = empty + PF_STAGES;
  uint64_t* mma_bar = opready + PF_NBUF;
  // misc[0]: abort flag; misc[1]: chunks the producer issued; misc[2]: tensor-memory base
  volatile int* misc = reinterpret_cast<volatile int*>(mma_bar + PF_NBUF);
  float* da_s = reinterpret_cast<float*>(smem + PF_OFF_DA);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < PF_STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], PF_NW);
    }
    for (int p = 0; p < PF_NBUF; ++p) {
      mbar_init(&opready[p], PF_NW);
      mbar_init(&mma_bar[p], 1);
    }
    misc[0] = 0;
    misc[1] = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(reinterpret_cast<uint32_t*>(const_cast<int*>(misc + 2)), PF_TMEM_COLS);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = static_cast<uint32_t>(misc[2]);
  pdl_launch_dependents();
  pdl_wait();  // activations and y belong to the previous work on the stream

  uint32_t consumed = 0;  // chunks whose copies the workers saw land (warp 0's count)
  if (warp >= PF_NW) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(PF_REG_ISSUER));
    if (warp == PF_NW && lane == 0) pf_issuer(a, smem, opready, mma_bar, misc, tmem);
    if (warp == PF_NW + 1 && lane == 0) pf_producer(a, smem, full, empty, misc);
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(PF_REG_WORKER));
    // thread (warp w, lane l): weight row `row` of the tile = tensor-memory
    // lane 32 (w % 4) + l, which it also converts; columns [64 hf, 64 hf + 64)
    // of the accumulators; half hf of each block's 32 quants when converting
    const int row = tid & (PF_TN - 1);
    const int hf = tid >> 7;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int G = PF_TN / a.RW;
    const int g = row / a.RW, ii = row - g * a.RW;
    uint32_t bc = 0;    // blocks converted, over all this CTA's tiles (low bits used)
    uint32_t kseq = 0;  // chunks
    bool dead = false;

    for (int T = blockIdx.x; T < a.tiles * a.split && !dead; T += gridDim.x) {
      int tile, part, c0, c1;
      pf_item(a, T, tile, part, c0, c1);
      const int nt = tile / a.tm, mt = tile - (tile / a.tm) * a.tm;
      const int ra = tile_rows(mt, a.M, PF_TM);
      const int64_t tw = (int64_t)nt * G + g;
      const int rw = tw * a.RW < a.N ? tile_rows(tw, a.N, a.RW) : 0;
      const bool wv = ii < rw;  // this row exists (n < N)
      uint64_t sig[32];         // sigma of columns 64 hf + 2e, + 2e + 1
#pragma unroll
      for (int e = 0; e < 32; ++e) sig[e] = 0ull;
      bool first_seg = true;
      int q1_blk = -1;  // the block whose accumulator is still to be read
      uint32_t q1_bc = 0;
      float q1_dw = 0.0f;

      // Fold block b (the CTA's block number bcn: accumulator bcn % 2,
      // activation scales bcn % 4, weight scale dw) into sigma; at a
      // segment's end into Y; at the tile's end store Y.  Warp-uniform.
      auto fold = [&](int b, uint32_t bcn, float dw) -> bool {
        const int pb = (int)(bcn & 1u);
        bool ok = mbar_wait_bounded(&mma_bar[pb], (bcn >> 1) & 1u, WAIT_LIMIT_NS);
        ok = __all_sync(0xffffffffu, ok);
        tc_fence_after_sync();
        if (!ok) return false;
        const uint32_t acc = tmem + lane_base + (uint32_t)(pb * PF_TM + hf * 64);
        const float* dap = da_s + (bcn % PF_DA_BUFS) * PF_TM + hf * 64;
        const uint64_t dw2 = f2_pack(dw, dw);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t u[16];
          tmem_ld16(acc + q * 16, u);  // isum
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float4 d4 = *reinterpret_cast<const float4*>(dap + q * 16 + 4 * e);
            const uint64_t s01 = f2_mul(dw2, f2_pack(d4.x, d4.y));  // d_w * d_a, exact
            const uint64_t s23 = f2_mul(dw2, f2_pack(d4.z, d4.w));
            sig[q * 8 + 2 * e] = f2_fma(f2_pack(__uint_as_float(u[4 * e]), __uint_as_float(u[4 * e + 1])), s01,
                                        sig[q * 8 + 2 * e]);
            sig[q * 8 + 2 * e + 1] = f2_fma(f2_pack(__uint_as_float(u[4 * e + 2]), __uint_as_float(u[4 * e + 3])),
                                            s23, sig[q * 8 + 2 * e + 1]);
          }
        }
        const bool last = b == a.NB - 1;
        if (!last && (b + 1) % PF_SEG != 0) return true;
        const int segi = b / PF_SEG;
        const bool lo_end = !last && segi == a.h - 1;  // the low half closes; the high half follows
        // A half closes with v = Y + sigma:
        //   whole K here, low half: v is kept in tensor memory (Y_lo), the high half starts from +0;
        //   whole K here, last block: y = Y_lo + v (y = v when K has one segment);
        //   split tile, low half: y = v + the high half's sums, once that half's warp published them;
        //   split tile, high half: y = v, then this warp's flag.
        const bool keep_lo = a.split == 1 && lo_end;
        const bool add_lo = a.split == 1 && last && segi >= a.h;
        const bool combine = a.split == 2 && part == 0;
        const bool publish = a.split == 2 && part == 1;
        const bool fin = (lo_end || last) && !keep_lo;  // y is written below
        const uint32_t yc = tmem + lane_base + PF_Y_COL + (uint32_t)(hf * 64);
        const uint32_t yl = tmem + lane_base + PF_YLO_COL + (uint32_t)(hf * 64);
        // pass 1: Y = Y + sigma (from +0 at a half's first segment) into tensor
        // memory -- the running sum, or the low half's sum (Y_lo)
        const uint32_t dst = keep_lo ? yl : yc;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t yv[16];
          if (first_seg) {
#pragma unroll
            for (int k = 0; k < 16; ++k) yv[k] = 0u;
          } else {
            tmem_ld16(yc + q * 16, yv);
            tmem_ld_wait();
          }
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            float lo, hi;
            f2_unpack(f2_add(f2_pack(__uint_as_float(yv[2 * e]), __uint_as_float(yv[2 * e + 1])), sig[q * 8 + e]),
                      lo, hi);
            sig[q * 8 + e] = 0ull;
            yv[2 * e] = __float_as_uint(lo);
            yv[2 * e + 1] = __float_as_uint(hi);
          }
          tmem_st16(dst + q * 16, yv);
        }
        tmem_st_wait();
        first_seg = keep_lo;  // the high half starts from +0
        if (!fin) return true;
        // pass 2: the outputs (out of line: once per tile and half)
        return pf_outputs(yc, yl, a.y + ((int64_t)mt * PF_TM + hf * 64) * a.N + (int64_t)nt * PF_TN + row, a.N,
                          wv ? ra - hf * 64 : 0, add_lo, combine, publish, a.flags + (size_t)tile * PF_NW + warp);
      };

      for (int c = c0; c < c1 && !dead; ++c, ++kseq) {
        const int stage = (int)(kseq & 1u);
        const bool got =
            __all_sync(0xffffffffu, misc[0] == 0 && mbar_wait_bounded(&full[stage], (kseq >> 1) & 1u, WAIT_LIMIT_NS));
        if (!got) {
          dead = true;
          break;
        }
        if (warp == 0) ++consumed;
        const int kb = chunk_blocks(c, a.NB);
        const uint8_t* cw = smem + (size_t)stage * PF_STAGE + (size_t)g * a.RW * CHUNK_BLOCKS * BLOCK_BYTES;
        const uint8_t* ca = smem + (size_t)stage * PF_STAGE + PF_CHUNK;
        for (int j = 0; j < kb; ++j) {
          const int pb = (int)(bc & 1u);
          uint8_t* ops = smem + PF_OFF_OPS + (size_t)pb * PF_OPS;
          const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
          const int rofs = (row >> 3) * 256 + (row & 7) * 16;
          const uint4 qw = wv ? lds128(cw + chunk_quant_off(j, hf, ii, rw)) : zero;
          put_f16_row(ops + hf * PF_SLICE + rofs, qw);
          const uint4 qa = row < ra ? lds128(ca + chunk_quant_off(j, hf, row, ra)) : zero;
          put_f16_row(ops + (2 + hf) * PF_SLICE + rofs, qa);
          if (hf == 1) da_s[(bc % PF_DA_BUFS) * PF_TM + row] = row < ra ? half_at(ca + chunk_scale_off(j, row, ra, kb)) : 0.0f;
          const float dw = wv ? half_at(cw + chunk_scale_off(j, ii, rw, kb)) : 0.0f;
          fence_proxy_async_smem();
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&opready[pb]);
            if (j == kb - 1) mbar_arrive(&empty[stage]);  // this warp is done with the stage
          }
          if (q1_blk >= 0 && !fold(q1_blk, q1_bc, q1_dw)) {
            dead = true;
            break;
          }
          q1_blk = c * CHUNK_BLOCKS + j;
          q1_bc = bc;
          q1_dw = dw;
          ++bc;
        }
      }
      if (!dead && q1_blk >= 0 && !fold(q1_blk, q1_bc, q1_dw)) dead = true;
    }
    if (dead) {
      if (lane == 0) atomicOr(a.err, ERR_PF_WORKER);
      misc[0] = 1;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (tid == 0 && misc[0] != 0) {
    // stopped early: let the copies in flight land before the shared
    // memory is given back
    const uint32_t issued = (uint32_t)misc[1];
    for (uint32_t k = consumed; k < issued; ++k)
      if (!mbar_wait_bounded(&full[k & 1u], (k >> 1) & 1u, WAIT_LIMIT_NS)) atomicOr(a.err, ERR_PF_DRAIN);
  }
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, PF_TMEM_COLS);
  }
}

std::mutex g_pf_mu;
bool g_pf_attr[64] = {};

}  // namespace

// Split along K when the output tiles fill at most half of the SMs and K has
// at least two segments: every tile becomes two CTAs (all resident at once,
// one CTA per SM), each with half of the segments.
bool prefill_splits(const DeviceInfo& dev, int64_t N, int64_t K, int64_t M) {
  const int64_t tiles = ((N + PF_TN - 1) / PF_TN) * ((M + PF_TM - 1) / PF_TM);
  const int64_t nseg = (K / QK + PF_SEG - 1) / PF_SEG;
  return nseg >= 2 && tiles <= PF_FLAG_TILES && 2 * tiles <= dev.sm_count;
}

cudaError_t launch_prefill(const DeviceInfo& dev, const uint8_t* W, int64_t N, int64_t K, const uint8_t* A_packed,
                           int64_t M, float* y, unsigned* flags, bool pdl, cudaStream_t s) {
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
  a.M = (int)M;
  a.NB = (int)(K / QK);
  a.nch = (a.NB + CHUNK_BLOCKS - 1) / CHUNK_BLOCKS;
  a.RW = layout_tile_rows(N);
  const int64_t tn = (N + PF_TN - 1) / PF_TN, tm = (M + PF_TM - 1) / PF_TM;
  if (tn * tm > INT32_MAX) return cudaErrorInvalidValue;
  a.tm = (int)tm;
  a.tiles = (int)(tn * tm);
  a.err = err;
  a.flags = flags;
  const int nseg = (a.NB + PF_SEG - 1) / PF_SEG;
  a.h = (nseg + 1) / 2;
  a.split = prefill_splits(dev, N, K, M) ? 2 : 1;
  const int64_t items = (int64_t)a.tiles * a.split;
  const int64_t grid = items < dev.sm_count ? items : dev.sm_count;
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
