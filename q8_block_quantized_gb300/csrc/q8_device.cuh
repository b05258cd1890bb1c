// q8_device.cuh -- device-side building blocks shared by the libq8 kernels:
// the packed layout arithmetic, the quantization rule, the int8 block dot,
// the canonical block-term rounding and the fixed reduction tree, plus thin
// wrappers for mbarrier, bulk copy and programmatic-dependent-launch PTX.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

#include "q8.h"

namespace q8 {

constexpr int QK = Q8_QK;
constexpr int BLOCK_BYTES = Q8_BLOCK_BYTES;
constexpr int MAX_TILE_ROWS = 128;
constexpr int CHUNK_BLOCKS = Q8_CHUNK_BLOCKS;
// Tile count the packed layout aims at: about one tile per SM of a GB300.
constexpr int LAYOUT_TARGET_TILES = 152;

// ---------------------------------------------------------------------------
// Packed layout (described in q8.h, q8_repack_weights).  Rows are grouped in
// tiles of R rows (R depends only on N), blocks in chunks of 8.
// ---------------------------------------------------------------------------
__host__ __device__ __forceinline__ int layout_tile_rows(int64_t N) {
  for (int R = 16; R < MAX_TILE_ROWS; R *= 2)
    if ((N + R - 1) / R <= LAYOUT_TARGET_TILES) return R;
  return MAX_TILE_ROWS;
}
__host__ __device__ __forceinline__ int tile_rows(int64_t t, int64_t N, int R) {
  int64_t r = N - t * R;
  return (int)(r < R ? r : R);
}
__host__ __device__ __forceinline__ int64_t tile_offset(int64_t t, int R, int64_t nb) {
  return t * R * nb * BLOCK_BYTES;
}
__host__ __device__ __forceinline__ int64_t chunk_offset(int64_t t, int64_t c, int r, int R, int64_t nb) {
  return tile_offset(t, R, nb) + (int64_t)r * (c * CHUNK_BLOCKS) * BLOCK_BYTES;
}
__host__ __device__ __forceinline__ int chunk_blocks(int64_t c, int64_t nb) {
  const int64_t k = nb - c * CHUNK_BLOCKS;
  return (int)(k < CHUNK_BLOCKS ? k : CHUNK_BLOCKS);
}
// byte offset, inside a chunk of kb blocks x r rows, of the 16 quants
// (block j, half h, row i) and of the scale (block j, row i)
__host__ __device__ __forceinline__ int chunk_quant_off(int j, int h, int i, int r) {
  return ((2 * j + h) * r + i) * 16;
}
__host__ __device__ __forceinline__ int chunk_scale_off(int j, int i, int r, int kb) {
  return kb * r * 32 + (j * r + i) * 2;
}

// ---------------------------------------------------------------------------
// Correctly rounded amax / 127 and 1 / d without the division routines.  The
// quantization rule needs both exactly (their bits decide the quants); the
// IEEE division and reciprocal routines carry data-dependent slow paths
// whose branches keep the compiler from overlapping the blocks of a batch.
// Both functions below use only IEEE multiplies and fmas, so their results
// do not depend on the machine; each was checked against IEEE division on
// the host (every non-negative finite float for the quotient; every
// subnormal and every significand at the boundary and typical exponents for
// the reciprocal, whose steps are exponent-independent in between).
// ---------------------------------------------------------------------------

// a / 127 for a >= 0: Markstein's correction of the estimate q0 = a * RN(1/127)
// with the exact fma remainder a - 127 q0 (P. Markstein, "Computation of
// elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 34(1), 1990).  inf and NaN pass through (a / 127 = a for them).
__device__ __forceinline__ float div127_rn(float a) {
  const float r = 0x1.020408p-7f;  // RN(1/127)
  const float q0 = __fmul_rn(a, r);
  const float rem = __fmaf_rn(-q0, 127.0f, a);
  const float q1 = __fmaf_rn(rem, r, q0);
  return (a <= 3.40282347e38f) ? q1 : a;
}

// 1 / d for a normal d with a normal reciprocal (d <= 2^126): a first
// estimate from the bit pattern (exponent negated, significand mirrored;
// relative error at most 1/8), then Newton-Raphson steps y += y (1 - d y)
// with fma, each squaring the relative error.  After four steps the result
// is the correctly rounded reciprocal except when the significand of d is all
// ones: 1/d then lies just above a rounding tie that the last step resolves
// downwards, so the answer is one ulp up (the known exception of the fma
// correction step in Markstein's theorem).
__device__ __forceinline__ float rcp_rn_normal(float d) {
  float y = __uint_as_float(0x7EF00000u - __float_as_uint(d));
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float e = __fmaf_rn(-d, y, 1.0f);
    y = __fmaf_rn(y, e, y);
  }
  return ((__float_as_uint(d) & 0x7FFFFFu) == 0x7FFFFFu) ? __uint_as_float(__float_as_uint(y) + 1u) : y;
}

// The reciprocal the quantization rule takes, for d = amax/127 (0 <= d <=
// 2^121, or inf/NaN): 0 for d = 0 and for d = inf; a subnormal d is scaled by
// 2^24 first and the result scaled back (exact, or the correctly rounded
// overflow to inf).
__device__ __forceinline__ float rcp_rn(float d) {
  const bool sub = d < 0x1p-126f;
  const float ds = sub ? __fmul_rn(d, 0x1p24f) : d;
  const float ys = rcp_rn_normal(ds);
  const float y = sub ? __fmul_rn(ys, 0x1p24f) : ys;
  return (d == 0.0f || d > 3.40282347e38f) ? 0.0f : y;
}

// ---------------------------------------------------------------------------
// Quantization of one 32-value block, one value per lane of a full warp.
// d = amax / 127 (fp32, correctly rounded), id = 1/d (correctly rounded; 0
// when d == 0), q = roundf(x * id) (ties away from zero), scale stored as
// binary16 (RNE).  Every operation is an explicitly rounded single-precision
// intrinsic, so the result does not depend on compiler flags.
// ---------------------------------------------------------------------------
struct LaneQuant {
  int q;            // this lane's quant, in [-127, 127]
  uint16_t d16;     // the block's binary16 scale bits (same on every lane)
  float d_stored;   // float value of d16 (what the products use)
};

__device__ __forceinline__ LaneQuant quantize_lane(float x) {
  float amax = fabsf(x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float d = div127_rn(amax);
  const float id = rcp_rn(d);
  // the conversion (cvt.rzi, saturating) takes +-inf (1/d = inf, d below
  // 2^-128) to the int range and NaN (0 * inf) to 0; the clamp then gives
  // [-127, 127]
  LaneQuant out;
  out.q = min(max(__float2int_rz(roundf(__fmul_rn(x, id))), -127), 127);
  const __half h = __float2half_rn(d);
  out.d16 = __half_as_ushort(h);
  out.d_stored = __half2float(h);
  return out;
}

// The same rule with the block's 32 values spread over fewer lanes gives the
// same single-precision results, so the bits match quantize_lane's:
//  - amax: max is exact and order-free, so any tree of maxima will do;
//  - d and 1/d come from the same correctly rounded functions;
//  - the clamp: |x * (1/d)| <= 127 * (1 + 2^-22) < 127.5 whenever 1/d is
//    finite, so roundf lands in [-127, 127]; with 1/d = inf (d below
//    2^-128) the products are +-inf, which the conversion (cvt.rzi,
//    saturating) takes to the int range and the lower bound to -127 (the
//    pack saturates the upper side), or NaN for x = 0, which it takes to 0.
__device__ __forceinline__ int q8_of(float v) { return max(__float2int_rz(roundf(v)), -127); }

// packed[k] holds quants 4k..4k+3, low byte first.
// cvt.pack.sat.s8.s32.b32 d, x, y, z puts y in byte 0, x in byte 1 and the
// low 16 bits of z in bytes 2-3; so (a, b, c, d) land in bytes 0..3.
__device__ __forceinline__ uint32_t pack4_s8(int a, int b, int c, int d) {
  uint32_t hi, r;
  asm("cvt.pack.sat.s8.s32.b32 %0, %1, %2, 0;" : "=r"(hi) : "r"(d), "r"(c));
  asm("cvt.pack.sat.s8.s32.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(b), "r"(a), "r"(hi));
  return r;
}

// The same rule for B blocks at once, each spread over 8 consecutive lanes
// of a warp: lane s of a group (s = lane % 8) holds values 4s..4s+3 of its
// block in v[q] and gets back their 4 quants packed (low byte first) in
// w[q]; every lane of the group gets the stored scale in d[q].  Each
// shuffle level is taken for all B blocks together so their dependency
// chains overlap.  All 32 lanes of the warp must call it (full-mask
// shuffles; a lane with nothing to quantize passes zeros).  With
// STORED16 = false, d[q] is the fp32 scale amax / 127 itself (the int8 KV
// cache keeps it unrounded); the quants are the same either way.
template <int B, bool STORED16 = true>
__device__ __forceinline__ void quantize_group8(const float4 (&v)[B], uint32_t (&w)[B], float (&d)[B]) {
  float am[B];
#pragma unroll
  for (int q = 0; q < B; ++q)
    am[q] = fmaxf(fmaxf(fabsf(v[q].x), fabsf(v[q].y)), fmaxf(fabsf(v[q].z), fabsf(v[q].w)));
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) {
    float t[B];
#pragma unroll
    for (int q = 0; q < B; ++q) t[q] = __shfl_xor_sync(0xffffffffu, am[q], o);
#pragma unroll
    for (int q = 0; q < B; ++q) am[q] = fmaxf(am[q], t[q]);
  }
#pragma unroll
  for (int q = 0; q < B; ++q) {
    const float dq = div127_rn(am[q]);
    const float id = rcp_rn(dq);
    d[q] = STORED16 ? __half2float(__float2half_rn(dq)) : dq;
    w[q] = pack4_s8(q8_of(__fmul_rn(v[q].x, id)), q8_of(__fmul_rn(v[q].y, id)),
                    q8_of(__fmul_rn(v[q].z, id)), q8_of(__fmul_rn(v[q].w, id)));
  }
}

// ---------------------------------------------------------------------------
// Fused producers' arithmetic, shared by their kernels and the GEMV's SwiGLU
// epilogue.
// ---------------------------------------------------------------------------
// The 8 lanes of a group store one block: lane s the quants of values
// 4s..4s+3 (bytes 2+4s..5+4s, 2-byte aligned), lane 0 also the scale.
__device__ __forceinline__ void store_block_lane(uint8_t* ob, int sub, uint32_t w, float d) {
  uint16_t* o16 = reinterpret_cast<uint16_t*>(ob);
  o16[1 + 2 * sub] = (uint16_t)(w & 0xffffu);
  o16[2 + 2 * sub] = (uint16_t)(w >> 16);
  if (sub == 0) o16[0] = __half_as_ushort(__float2half_rn(d));  // d is a binary16 value: exact
}

// e^x by a fixed single-precision procedure: Cody and Waite's reduction
// x = n ln2 + r, ln2 split into 355/512 (9 significant bits: n * 355/512 is
// exact for |n| <= 128) and the rest of ln2 rounded to single precision, one
// fused multiply-add per step; the Taylor polynomial of degree 7 of e^r in
// Horner form, one fused multiply-add per step (|r| <= 0.35); scaling by 2^n
// (exact).  Outside [-87, 88] the result is 0 or +infinity.
constexpr float EXP_LOG2E = 0x1.715476p+0f;    // 1/ln 2, rounded
constexpr float EXP_LN2_HI = 0x1.63p-1f;       // 355/512
constexpr float EXP_LN2_LO = -0x1.bd0106p-13f; // ln 2 - 355/512, rounded
constexpr float EXP_C3 = 0x1.555556p-3f;       // 1/3!
constexpr float EXP_C4 = 0x1.555556p-5f;       // 1/4!
constexpr float EXP_C5 = 0x1.111112p-7f;       // 1/5!
constexpr float EXP_C6 = 0x1.6c16c2p-10f;      // 1/6!
constexpr float EXP_C7 = 0x1.a01a02p-13f;      // 1/7!

__device__ __forceinline__ float exp_cw(float x) {
  if (x > 88.0f) return __int_as_float(0x7f800000);
  if (x < -87.0f) return 0.0f;
  const float n = rintf(__fmul_rn(x, EXP_LOG2E));
  const float r = __fmaf_rn(-n, EXP_LN2_LO, __fmaf_rn(-n, EXP_LN2_HI, x));
  float p = EXP_C7;
  p = __fmaf_rn(p, r, EXP_C6);
  p = __fmaf_rn(p, r, EXP_C5);
  p = __fmaf_rn(p, r, EXP_C4);
  p = __fmaf_rn(p, r, EXP_C3);
  p = __fmaf_rn(p, r, 0.5f);
  p = __fmaf_rn(p, r, 1.0f);
  p = __fmaf_rn(p, r, 1.0f);
  return __fmul_rn(p, __int_as_float(((int)n + 127) << 23));  // 2^n, -126 <= n <= 127
}

__device__ __forceinline__ float swiglu_one(float g, float u) {
  return __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, exp_cw(-g))), u);
}

// ---------------------------------------------------------------------------
// int8 block dot (exact int32) and the canonical block term.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int dot_block(const uint4& w0, const uint4& w1, const uint4& a0,
                                         const uint4& a1) {
  int s = 0;
  s = __dp4a((int)w0.x, (int)a0.x, s);
  s = __dp4a((int)w0.y, (int)a0.y, s);
  s = __dp4a((int)w0.z, (int)a0.z, s);
  s = __dp4a((int)w0.w, (int)a0.w, s);
  s = __dp4a((int)w1.x, (int)a1.x, s);
  s = __dp4a((int)w1.y, (int)a1.y, s);
  s = __dp4a((int)w1.z, (int)a1.z, s);
  s = __dp4a((int)w1.w, (int)a1.w, s);
  return s;
}

// t_b = float(isum) * (d_w * d_a): the scale product of two binary16 values is
// exact in fp32, float(isum) is exact (|isum| <= 516128 < 2^24), so the term
// is rounded exactly once.
__device__ __forceinline__ float block_term(int isum, float dw, float da) {
  return __fmul_rn(__int2float_rn(isum), __fmul_rn(dw, da));
}

__device__ __forceinline__ float tadd(float a, float b) { return __fadd_rn(a, b); }

// ---------------------------------------------------------------------------
// int8 -> fp16 for the tensor-core path.  For a byte x in [-128, 127],
// (x + 128) written into the low byte of the binary16 pattern 0x6400
// (= 1024, exponent 25, ulp 1) encodes 1024 + x + 128 exactly; subtracting
// 1152 (0x6480) leaves x, exactly.  Four int8 -> two half2:
//   lo = {x0, x1}, hi = {x2, x3} (low half first).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void i8x4_to_h2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t f = w ^ 0x80808080u;
  const uint32_t l = __byte_perm(f, 0x64646464u, 0x5140);
  const uint32_t h = __byte_perm(f, 0x64646464u, 0x5342);
  const __half2 bias = __halves2half2(__ushort_as_half((unsigned short)0x6480),
                                      __ushort_as_half((unsigned short)0x6480));
  const __half2 rl = __hsub2(*reinterpret_cast<const __half2*>(&l), bias);
  const __half2 rh = __hsub2(*reinterpret_cast<const __half2*>(&h), bias);
  lo = *reinterpret_cast<const uint32_t*>(&rl);
  hi = *reinterpret_cast<const uint32_t*>(&rh);
}

// D = A * B + C, m16n8k16, fp16 inputs, fp32 accumulate (warp-wide).
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// The same with C = 0 (D = A * B), and both forms without `volatile`: pure
// register arithmetic the compiler may schedule freely.
__device__ __forceinline__ void mma_16816_c0(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  const float z = 0.0f;
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(z));
}
__device__ __forceinline__ void mma_16816_acc(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------------------
// Small PTX wrappers.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
// Adds `bytes` to the transaction count of the current phase (no arrival).
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Non-blocking test of an mbarrier phase.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// The same two waits acquiring at cluster scope: for phases completed by
// arrivals of other CTAs of the cluster (mbar_arrive_remote).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_test_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait on an mbarrier phase: false after `limit_ns` without progress.
// A try_wait may suspend the thread for a time the hardware chooses, so a
// limit below a millisecond (only set by tests) polls with test_wait instead
// and is then honoured to the clock's resolution.  CLUSTER: acquire at
// cluster scope, always polling (phases completed by other CTAs' arrivals
// are waited for without suspending the thread).
constexpr uint64_t SHORT_WAIT_NS = 1000000ull;
template <bool CLUSTER>
__device__ __forceinline__ bool mbar_probe(uint64_t* bar, uint32_t parity, bool poll) {
  if constexpr (CLUSTER) {
    return poll ? mbar_test_wait_cluster(bar, parity) : mbar_try_wait_cluster(bar, parity);
  } else {
    return poll ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity);
  }
}
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const bool poll = CLUSTER || limit_ns < SHORT_WAIT_NS;
  if (mbar_probe<CLUSTER>(bar, parity, poll)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_probe<CLUSTER>(bar, parity, poll)) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}
// One contiguous global -> shared bulk copy, completing on `bar` (tx bytes).
// dst and src 16-byte aligned, bytes a positive multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
// The same without an L2 cache hint (data that many CTAs read).
__device__ __forceinline__ void bulk_g2s_nohint(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// ---------------------------------------------------------------------------
// 5th-generation tensor cores (tcgen05): tensor memory, MMA, read-back.
// ---------------------------------------------------------------------------
// Shared-memory matrix descriptor, no swizzle: start address, leading byte
// offset (between core matrices along K), stride byte offset (between core
// matrices along M/N), descriptor version 1 at bit 46.  A core matrix is 8
// rows of 16 contiguous bytes.
__device__ __forceinline__ uint64_t umma_smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo & 0x3FFFFu) >> 4) << 16) |
         ((uint64_t)((sbo & 0x3FFFFu) >> 4) << 32) | ((uint64_t)1 << 46);
}
// Instruction descriptor of kind::f16: fp32 accumulator, fp16 A and B, both
// K-major, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t umma_idesc_f16(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// Warp-wide: allocate `ncols` tensor-memory columns (a power of two >= 32);
// the base address is written to shared memory at `slot`.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t base, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(ncols) : "memory");
}
// D[tmem] (+)= A . B^T, one thread issues; accumulate = false starts D at 0.
__device__ __forceinline__ void umma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}
// The mbarrier receives one arrival when every MMA issued so far by this
// thread has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}
// A warp reads 8 consecutive 32-bit columns of its 32 lanes (lane = row):
// taddr holds the warp's first lane in bits 31..16 and the column below.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&v)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
               : "r"(taddr)
               : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Generic-proxy shared-memory writes become visible to the async proxy
// (operands written by threads, read by tcgen05.mma).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Thread-block clusters: rank, size, barrier, distributed shared memory.
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
// all threads of every warp that calls these must call them together
__device__ __forceinline__ void cluster_arrive_aligned() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_aligned() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// arrival of a single thread (no wait)
__device__ __forceinline__ void cluster_arrive_one() {
  asm volatile("barrier.cluster.arrive.release;" ::: "memory");
}
// address of the same shared-memory location in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_cluster_u16(uint32_t addr, unsigned short v) {
  asm volatile("st.shared::cluster.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}
__device__ __forceinline__ float4 ld_cluster_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
// Arrival on the mbarrier at `remote` (a shared::cluster address, e.g. from
// mapa_shared), releasing at cluster scope what happened before it.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t remote) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote) : "memory");
}


// Programmatic dependent launch: no-ops when the grid was launched normally.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
__device__ __forceinline__ uint4 lds128(const void* p) {
  return *reinterpret_cast<const uint4*>(p);
}
__device__ __forceinline__ uint32_t lds32(const void* p) {
  return *reinterpret_cast<const uint32_t*>(p);
}

// 32 quants of an unaligned 34-byte block (2-byte aligned) as two uint4.
// Loads bypass L1 (ld.global.cg): the block may have been written by the
// kernel this one depends on.
__device__ __forceinline__ void load_block_quants_u16(const uint8_t* blk, uint4& a0, uint4& a1) {
  const unsigned short* p = reinterpret_cast<const unsigned short*>(blk + 2);
  uint32_t w[8];
#pragma unroll
  for (int k = 0; k < 8; ++k)
    w[k] = (uint32_t)__ldcg(p + 2 * k) | ((uint32_t)__ldcg(p + 2 * k + 1) << 16);
  a0 = make_uint4(w[0], w[1], w[2], w[3]);
  a1 = make_uint4(w[4], w[5], w[6], w[7]);
}

// Device time limit for every spin on an mbarrier (2 s).
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;

}  // namespace q8
