// q8_gemv_impl.cuh -- the Q8_0 decode GEMV kernel, templated on the packed
// tile height R, the activation rows per pass MT and whether the activation
// is quantized in the kernel (FUSED).
//
// Work decomposition.  The packed layout groups rows in tiles of R rows
// (R in {16, 32, 64, 128}, chosen from N so a matrix has about one tile per
// SM) and blocks in chunks of 8; the chunks of a tile are contiguous.  A
// pipeline round is P = 128/R consecutive chunks of one tile (one contiguous
// bulk copy of up to 34,816 bytes).  A work unit is one tile times RU
// consecutive rounds; usually a unit covers all of K and a tile is one unit.
// A CTA is 8 consumer warps and one producer warp, one CTA per SM.
//
// DP4A path (MT <= 4).  Consumer thread t owns row i = t % R, part p =
// (t / R) % P (chunk p of each round) and half t / 128 of that chunk (4
// blocks), which halves a round's latency.  For each block it computes the
// exact int32 dot of its row with every activation row (__dp4a), the
// canonical term t_b = float(isum) * (d_w * d_a), and the pairwise tree of
// its blocks.  Within a quarter warp the 8 lanes read 8 consecutive rows of
// one chunk (distinct banks) and the same activation block (a broadcast).
// Tensor path (MT >= 8).  A warp computes 16-row slices of a chunk with
// mma.sync on int8 values converted exactly to fp16 (8 slices per round,
// one per warp); the block terms and trees are the same as on the DP4A path.
// Either way the values of a round meet in shared memory, and each row is
// then merged by CG = min(256 / R, MT) threads that own MT / CG output
// columns each.
//
// Pipeline.  One lane of the producer warp issues one cp.async.bulk copy per
// round into a ring of shared-memory stages, completing on mbarriers; every
// wait is bounded and a failed wait sets the device error word and aborts.
//
// Reduction order.  The sum over blocks b is the pairwise tree over b,
// padded with zeros to a power of two.  A chunk (8 aligned blocks) is a
// subtree; a round (P aligned chunks) is a subtree, formed by the part-0
// thread of each row from the P chunk values (exchanged through shared
// memory) in pairwise order; rounds are merged with a binary counter (merge
// with the left sibling while the index bit is 1; what is left at the end
// merges from the lowest level up, which is what zero padding gives), so a
// unit is a subtree too, and when a tile is split along K into S > 1 units,
// the unit values are merged the same way.  The result for an output depends
// only on its row of W, its row of activations and K.
//
// Split along K (S > 1: large K with many activation rows, or few tiles).
// Each unit writes its row values to the workspace and takes a ticket on the
// tile's counter; the CTA holding the last ticket merges the S values in
// index order, writes y and resets the counter.  No CTA waits for another.
//
// Programmatic dependent launch.  The producer starts streaming W at once
// (W is immutable); the consumers execute griddepcontrol.wait before reading
// activations or writing anything.
#pragma once

#include <cuda_runtime.h>

#include <atomic>

#include "q8_device.cuh"
#include "q8_internal.h"

namespace q8 {

constexpr int MAX_SPLITS = 128;
constexpr int SPLIT_LEVELS = 8;  // binary counter levels for S <= 128
// Workspace layout: a fixed prefix of tile tickets, then the partials.  The
// prefix has the same size for every call, so partials written by one call
// never land on the tickets of another call that shares the workspace.
constexpr int MAX_SPLIT_TILES = 4096;
constexpr size_t TICKET_BYTES = (size_t)MAX_SPLIT_TILES * 4;
constexpr int MAX_ROUNDS_PER_UNIT = 64;


enum : unsigned { ERR_PRODUCER_WAIT = 1u, ERR_CONSUMER_WAIT = 2u, ERR_DRAIN_WAIT = 4u };

template <int R>
struct RCfg {
  static constexpr int P = 128 / R;                                  // parts (chunks per round)
  static constexpr int STAGE_BYTES = P * R * CHUNK_BLOCKS * BLOCK_BYTES;  // 34816
};

template <int MT>
struct MCfg {
  // consumer warps: 8 (on the DP4A path each thread takes half a chunk, 4
  // blocks, which halves the latency of a round; on the tensor path each
  // warp takes one 16-row slice of a round; the 288-thread CTA also keeps
  // one CTA per SM)
  static constexpr int NCW = 8;
  // threads per (row, chunk) on the DP4A path; the tensor path computes a
  // round as 8 slices of 16 rows, 8 / NCW per warp
  static constexpr int HALVES = MT >= 8 ? 1 : NCW * 32 / 128;
  static constexpr int THREADS = (NCW + 1) * 32;      // + the producer warp
  static constexpr int STAGES = MT <= 2 ? 3 : 2;
  // CTAs per SM the kernel is compiled for: one.  Registers are not capped
  // for a second CTA: a co-resident CTA of the next kernel (started early by
  // PDL) prefetches while the current kernel, which is on the critical path,
  // still streams and computes, and measured slower (the 288-thread kernel
  // at 96 registers and two CTAs per SM: 0.373 ms per M = 1 step; uncapped,
  // one CTA per SM: 0.326 ms)
  static constexpr int MIN_CTAS = 1;
  // activation staging: passes of NCW*4 = 32 blocks (8 lanes per block),
  // STAGE_BATCH passes with their loads in flight together (K = 2048 in one
  // batch; larger batches measured slower for every row count)
  static constexpr int STAGE_BATCH = 2;
  // blocks one CTA stages by itself (one batch: passes of NCW*4 blocks)
  // before the planner shares the staging among the CTAs of a cluster
  static constexpr int STAGE_TARGET = NCW * 4 * STAGE_BATCH;
  // bytes of staged activations: 256 blocks of MT rows (padded rows on the
  // tensor path, binary16 scales), so K = 8192 fits one unit and needs no
  // split along K (a split restages the activations for every unit)
  static constexpr int ACT_BUDGET = MT == 1 ? 8704 : MT == 2 ? 17408 : MT == 4 ? 34816
                                  : MT * (256 * 32 + 16) + MT * 256 * 2;
};

// Activation rows at or above this use the tensor-core path.
constexpr int TC_MIN_MT = 8;

// Kernel variants (template parameter V): the default, the tcgen05 block
// dots (VAR_TCGEN05) and the SwiGLU epilogue (VAR_SWIGLU).
constexpr int VAR_DEFAULT = 0, VAR_TCGEN05 = 1, VAR_SWIGLU = 2;

// 5th-generation tensor-core path (tcgen05), selected per call: tiles
// of 128 rows (one chunk per round) with 16 activation rows.  Each round the consumer warps convert
// the chunk's int8 weights and the round's activation blocks exactly to fp16
// in the MMA's canonical layout (no swizzle, K-major: core matrices of 8 rows
// x 16 bytes, 128 bytes apart along k, 256 bytes apart along rows), one
// thread issues two 128 x 16 x 16 MMAs per block into tensor memory (a fresh
// fp32 accumulator per block: every partial sum is an integer below 2^24, so
// it holds the exact block dot), and the consumers read the block dots back
// for the canonical terms and trees.
template <int R, int MT, int V>
struct UCfg {
  static constexpr bool ON = V == VAR_TCGEN05 && R == 128 && MT == 16;
  static constexpr int SLICE_A = 128 * 16 * 2;  // one 16-wide k slice of the 128 weight rows, fp16
  static constexpr int SLICE_B = MT * 16 * 2;   // the same slice of the activation rows
  static constexpr int A_BYTES = ON ? 2 * CHUNK_BLOCKS * SLICE_A : 0;
  static constexpr int B_BYTES = ON ? 2 * CHUNK_BLOCKS * SLICE_B : 0;
  static constexpr int TMEM_COLS = CHUNK_BLOCKS * MT;  // block j's dots in columns [MT j, MT j + MT)
  // flags, then (tcgen05) the MMA mbarrier and the TMEM base, then the two
  // consumer abort flags
  static constexpr int CAB = ON ? 8 : 4;
  static constexpr int MISC_INTS = CAB + 2;
};
// dynamic shared memory a CTA may use on sm_103 (227 KB)
constexpr int SMEM_LIMIT = 232448;

// activation bytes of one unit (RU rounds of P chunks) in shared memory,
// laid out for MT rows: quants [MT][blocks][32] (on the tensor path with 16
// bytes of padding per row, so its loads of 8 rows hit distinct banks), then
// scales [MT][blocks]
__host__ __device__ constexpr int act_row_bytes(int MT, int UB) {
  return UB * 32 + (MT >= TC_MIN_MT ? 16 : 0);
}
__host__ __device__ constexpr int act_bytes(int MT, int P, int RU) {
  return MT * act_row_bytes(MT, P * RU * CHUNK_BLOCKS) + MT * P * RU * CHUNK_BLOCKS * 2;
}

// bytes of staged activations a unit may use: MCfg's budget, or on the
// tcgen05 path what the stages and the fp16 operands leave of SMEM_LIMIT
template <int R, int MT, int V>
__host__ __device__ constexpr int act_budget() {
  return UCfg<R, MT, V>::ON
             ? (SMEM_LIMIT - MCfg<MT>::STAGES * RCfg<R>::STAGE_BYTES - UCfg<R, MT, V>::A_BYTES -
                UCfg<R, MT, V>::B_BYTES - 2 * MCfg<MT>::STAGES * 8 - UCfg<R, MT, V>::MISC_INTS * 4) / 16 * 16
             : MCfg<MT>::ACT_BUDGET;
}

template <int R, int MT, int V>
__host__ __device__ constexpr int ru_max() {
  int c = MAX_ROUNDS_PER_UNIT;
  while (c > 1 && act_bytes(MT, RCfg<R>::P, c) > act_budget<R, MT, V>()) c >>= 1;
  return c;
}
__host__ __device__ constexpr int log2_floor(int v) { return v <= 1 ? 0 : 1 + log2_floor(v >> 1); }

// row stride (floats) of the exchange buffer: odd on the tensor path, where
// a thread's MT values would otherwise share banks with its neighbours'
template <int MT>
constexpr int red_stride() {
  return MT >= TC_MIN_MT ? MT + 1 : MT;
}

// per-round exchange of chunk values between the parts of a row (and, on
// the tensor path, from the MMA fragment layout to one thread per row):
// [2 buffers][P parts][R rows][red_stride]
template <int R, int MT, int V>
constexpr int red_bytes() {
  return !UCfg<R, MT, V>::ON && (RCfg<R>::P > 1 || MT >= TC_MIN_MT || MCfg<MT>::HALVES > 1)
             ? 2 * MCfg<MT>::HALVES * 128 * red_stride<MT>() * 4
             : 0;
}

template <int R, int MT, int V>
constexpr size_t gemv_smem_bytes(int act = act_budget<R, MT, V>()) {
  return (size_t)MCfg<MT>::STAGES * RCfg<R>::STAGE_BYTES + UCfg<R, MT, V>::A_BYTES + UCfg<R, MT, V>::B_BYTES + act +
         red_bytes<R, MT, V>() + 2 * MCfg<MT>::STAGES * sizeof(uint64_t) + UCfg<R, MT, V>::MISC_INTS * sizeof(int);
}

struct GemvArgs {
  const uint8_t* W;
  const uint8_t* A;      // activation blocks [M][NB] (unfused)
  const float* x;        // fp32 activations [M][K] (fused)
  uint8_t* A_out;        // fused: optional activation blocks out
  float* y;              // [M][N]
  uint8_t* h_blocks;     // SwiGLU epilogue: blocks of silu(gate) * up [M][N/64], or null (y written)
  float* ws_part;        // [S][M][N] partials (S > 1)
  unsigned* ws_cnt;      // [T] tickets (S > 1)
  unsigned* err;         // device error word
  uint64_t wait_ns;      // limit of the ring's producer and consumer waits (WAIT_LIMIT_NS unless a test shortens it)
  int64_t N;
  int NB, nch, T, M, RU, S, units;
  int act_smem;          // bytes of the activation staging area of this launch (<= ACT_BUDGET, 16 | x)
};

// ---- producer: one lane streams the rounds of every unit of this CTA ----
// In a cluster (CL > 1) the producer lane takes part in the two cluster
// barrier phases (see the kernel): it arrives for phase 1 before streaming,
// issues the first STAGES rounds (which never wait), then waits for phase 1
// and arrives for phase 2, so the start of streaming does not wait for the
// rest of the cluster.
template <int R, int STAGES>
__device__ __forceinline__ void produce(const GemvArgs& a, uint8_t* stage_buf, uint64_t* full,
                                        uint64_t* empty, volatile int* misc, uint32_t CL) {
  constexpr int P = RCfg<R>::P;
  const uint64_t pol = l2_policy_evict_first();
  int stage = 0;
  uint32_t phase = 0;
  int issued = 0;
  bool cluster_done = (CL == 1);
  bool stop = false;
  for (int u = blockIdx.x; u < a.units && !stop; u += gridDim.x) {
    const int t = u / a.S, s = u - (u / a.S) * a.S;
    const int r = tile_rows(t, a.N, R);
    const int c0 = s * a.RU * P;
    const int nrounds = min(a.RU, (a.nch - c0 + P - 1) / P);
    for (int rho = 0; rho < nrounds; ++rho) {
      if (!cluster_done && issued == STAGES) {
        asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
        cluster_arrive_one();
        cluster_done = true;
      }
      if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, a.wait_ns)) {
        atomicOr(a.err, ERR_PRODUCER_WAIT);
        misc[0] = 1;
        stop = true;
        break;
      }
      if (misc[0]) {
        stop = true;
        break;
      }
      // the round's chunks are contiguous: one copy (ragged tail by hand)
      const int cb = c0 + rho * P;
      const int ce = min(cb + P, a.nch);
      const uint8_t* src = a.W + chunk_offset(t, cb, r, R, a.NB);
      const uint32_t bytes = (uint32_t)(((int64_t)min(ce * CHUNK_BLOCKS, a.NB) - (int64_t)cb * CHUNK_BLOCKS) *
                                        r * BLOCK_BYTES);
      const uint32_t bulk = bytes & ~15u;
      uint8_t* dst = stage_buf + (size_t)stage * RCfg<R>::STAGE_BYTES;
      for (uint32_t k = bulk; k < bytes; ++k) dst[k] = src[k];  // < 16 bytes
      mbar_arrive_expect_tx(&full[stage], bulk);
      bulk_g2s(dst, src, bulk, &full[stage], pol);
      misc[2] = ++issued;
      if (++stage == STAGES) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
  if (!cluster_done) {
    asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
    cluster_arrive_one();
  }
}

// Staged activation blocks of a unit, in block order: quants of row m,
// block blk at q + m*mq + blk*32 (mq = act_row_bytes), its binary16 scale at
// d[m*UB + blk], UB = blocks per unit.
struct ActLayout {
  uint8_t* q;
  __half* d;
  int UB, mq;
};

__device__ __forceinline__ ActLayout act_layout(uint8_t* base, int MT, int UB) {
  ActLayout L;
  L.UB = UB;
  L.mq = act_row_bytes(MT, UB);
  L.q = base;
  L.d = reinterpret_cast<__half*>(base + (size_t)MT * L.mq);
  return L;
}

// Stage the activation blocks [b0, b0 + nblk) of rows < M.  Eight
// consecutive lanes take one block: lane s = threadIdx.x % 8 loads (and, on
// the fused path, quantizes with its 7 neighbours) values 4s..4s+3 and stores
// their 4 quants; lane 0 of the group stores the scale.  The blocks of all
// rows form one sequence (row-major); with a cluster of CL CTAs that all need
// the same blocks, CTA c takes every CL-th of them (c, c+CL, ...) and writes
// each into the staging area of every CTA of the cluster (distributed shared
// memory); the caller then waits on the cluster barrier.  A pass covers 16
// blocks; BATCH passes have their loads in flight together.
template <bool CLUSTER>
__device__ __forceinline__ void put_word(const ActLayout& L, int m, int blk, int sub, uint32_t w,
                                         __half d, uint32_t CL) {
  uint32_t* dst = reinterpret_cast<uint32_t*>(L.q + m * L.mq + blk * 32) + sub;
  __half* dd = L.d + m * L.UB + blk;
  if constexpr (!CLUSTER) {
    *dst = w;
    if (sub == 0) *dd = d;
  } else {
    const uint32_t q0 = smem_u32(dst), d0 = smem_u32(dd);
    for (uint32_t c = 0; c < CL; ++c) {
      st_cluster_u32(mapa_shared(q0, c), w);
      if (sub == 0) st_cluster_u16(mapa_shared(d0, c), __half_as_ushort(d));
    }
  }
}

template <bool FUSED, bool CLUSTER, int NT, int BATCH>
__device__ __forceinline__ void stage_activations(const GemvArgs& a, const ActLayout& L, int b0,
                                                  int nblk, uint32_t rank, uint32_t CL) {
  constexpr int BPP = NT / 8;  // blocks per pass
  const int64_t K = (int64_t)a.NB * QK;
  const int total = a.M * nblk;
  const int mine = (total - (int)rank + (int)CL - 1) / (int)CL;  // blocks rank, rank+CL, ...
  const int sub = threadIdx.x & 7, slot = threadIdx.x >> 3;
  const int step = BPP * (int)CL;  // sequence distance between passes
  // trip counts are uniform across the CTA: the shuffles inside see full warps
  for (int base = 0; base < mine; base += BPP * BATCH) {
    // row and block of this thread's first block of the batch (one division
    // per batch), then stepped forward pass by pass
    int k = (base + slot) * (int)CL + (int)rank, m = 0;
    if (a.M > 1) {
      m = k / nblk;
      k -= m * nblk;
    }
    int mm[BATCH], kk[BATCH];
    bool on[BATCH];
#pragma unroll
    for (int q = 0; q < BATCH; ++q) {
      on[q] = base + q * BPP + slot < mine;
      mm[q] = m;
      kk[q] = k;
      k += step;
      while (k >= nblk && m < a.M) {  // once per step when nblk >= step
        k -= nblk;
        ++m;
      }
    }
    if constexpr (FUSED) {
      float4 v[BATCH];
#pragma unroll
      for (int q = 0; q < BATCH; ++q)
        v[q] = on[q] ? __ldcg(reinterpret_cast<const float4*>(a.x + (int64_t)mm[q] * K +
                                                               (int64_t)(b0 + kk[q]) * QK) +
                              sub)
                     : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      uint32_t w[BATCH];
      float d[BATCH];
      quantize_group8<BATCH>(v, w, d);
#pragma unroll
      for (int q = 0; q < BATCH; ++q)
        if (on[q]) put_word<CLUSTER>(L, mm[q], kk[q], sub, w[q], __float2half_rn(d[q]), CL);  // exact
    } else {
      // a block is 34 bytes (2-byte aligned): the scale, then 32 quants
      uint32_t w[BATCH];
      unsigned short dbits[BATCH];
#pragma unroll
      for (int q = 0; q < BATCH; ++q) {
        w[q] = 0u;
        dbits[q] = 0;
        if (on[q]) {
          const unsigned short* blk = reinterpret_cast<const unsigned short*>(
              a.A + ((int64_t)mm[q] * a.NB + b0 + kk[q]) * BLOCK_BYTES);
          w[q] = (uint32_t)__ldcg(blk + 1 + 2 * sub) | ((uint32_t)__ldcg(blk + 2 + 2 * sub) << 16);
          if (sub == 0) dbits[q] = __ldcg(blk);
        }
      }
#pragma unroll
      for (int q = 0; q < BATCH; ++q)
        if (on[q]) put_word<CLUSTER>(L, mm[q], kk[q], sub, w[q], __ushort_as_half(dbits[q]), CL);
    }
  }
}

// Fused path: the CTAs that own row tile 0 publish the quantized activations
// of their K range (every K range is covered once by tile 0).
template <int NT>
__device__ __forceinline__ void write_act_blocks(const GemvArgs& a, const ActLayout& L, int b0,
                                                 int nblk) {
  const int total = a.M * nblk;
  for (int idx = threadIdx.x; idx < total; idx += NT) {
    const int m = idx / nblk, blk = idx - m * nblk;
    uint8_t* ob = a.A_out + ((int64_t)m * a.NB + b0 + blk) * BLOCK_BYTES;
    const uint16_t d16 = __half_as_ushort(L.d[m * L.UB + blk]);
    const uint8_t* q = L.q + m * L.mq + blk * 32;
    unsigned short* o16 = reinterpret_cast<unsigned short*>(ob);
    o16[0] = d16;
#pragma unroll
    for (int k = 0; k < 16; ++k) o16[1 + k] = (unsigned short)(q[2 * k] | (q[2 * k + 1] << 8));
  }
}

// Block term of row i for block j of the chunk against every activation row.
// Two independent dp4a chains per block keep the dependent latency short.
template <int MT>
__device__ __forceinline__ void block_terms(const uint8_t* cq, const uint8_t* sc, int r, int i,
                                            int j, const uint8_t* aq, const __half* ad, int mq,
                                            int md, float (&out)[MT]) {
  const uint4 w0 = lds128(cq + ((2 * j) * r + i) * 16);
  const uint4 w1 = lds128(cq + ((2 * j + 1) * r + i) * 16);
  const float dw =
      __half2float(__ushort_as_half(*reinterpret_cast<const unsigned short*>(sc + (j * r + i) * 2)));
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    const uint8_t* am = aq + m * mq + j * 32;
    const uint4 a0 = lds128(am), a1 = lds128(am + 16);
    int s0 = __dp4a((int)w0.x, (int)a0.x, 0);
    int s1 = __dp4a((int)w1.x, (int)a1.x, 0);
    s0 = __dp4a((int)w0.y, (int)a0.y, s0);
    s1 = __dp4a((int)w1.y, (int)a1.y, s1);
    s0 = __dp4a((int)w0.z, (int)a0.z, s0);
    s1 = __dp4a((int)w1.z, (int)a1.z, s1);
    s0 = __dp4a((int)w0.w, (int)a0.w, s0);
    s1 = __dp4a((int)w1.w, (int)a1.w, s1);
    out[m] = block_term(s0 + s1, dw, __half2float(ad[m * md + j]));  // integer sum: exact
  }
}

// One chunk (kb <= 8 blocks; blocks at or past kb count as zero) of row i:
// the pairwise tree of its blocks, per activation row.  aq/ad point at the
// chunk's first activation block; mq/md are the strides between activation
// rows.  All 8 blocks are computed in straight-line code and the terms of
// blocks past kb are replaced by zero (their reads stay inside the stage and
// staging buffers, whatever they hold), so partial chunks need no second copy
// of the code.  Rows m >= M are computed on whatever the staging area holds
// and never stored.
template <int MT>
__device__ __forceinline__ void chunk_value(const uint8_t* cq, int r, int kb, int i,
                                            const uint8_t* aq, const __half* ad, int mq, int md,
                                            float (&v)[MT]) {
  const uint8_t* sc = cq + kb * r * 32;
  float q[2][MT];
#pragma unroll
  for (int h4 = 0; h4 < 2; ++h4) {
    float p0[MT], p1[MT];
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      float ta[MT], tb[MT];
      const int j = 4 * h4 + 2 * h2;
      block_terms<MT>(cq, sc, r, i, j, aq, ad, mq, md, ta);
      block_terms<MT>(cq, sc, r, i, j + 1, aq, ad, mq, md, tb);
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        ta[m] = (j < kb) ? ta[m] : 0.0f;
        tb[m] = (j + 1 < kb) ? tb[m] : 0.0f;
        (h2 ? p1 : p0)[m] = tadd(ta[m], tb[m]);
      }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) q[h4][m] = tadd(p0[m], p1[m]);
  }
#pragma unroll
  for (int m = 0; m < MT; ++m) v[m] = tadd(q[0][m], q[1][m]);
}

// Half a chunk: the 4-block subtree of blocks j0..j0+3 (j0 = 0 or 4), the
// same straight-line code and masking as chunk_value; the two halves' values
// merge into the chunk value (the top node of the 8-block tree).
template <int MT>
__device__ __forceinline__ void chunk_value_half(const uint8_t* cq, int r, int kb, int i, int j0,
                                                 const uint8_t* aq, const __half* ad, int mq, int md,
                                                 float (&v)[MT]) {
  const uint8_t* sc = cq + kb * r * 32;
  float pp[2][MT];
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
    float ta[MT], tb[MT];
    const int j = j0 + 2 * h2;
    block_terms<MT>(cq, sc, r, i, j, aq, ad, mq, md, ta);
    block_terms<MT>(cq, sc, r, i, j + 1, aq, ad, mq, md, tb);
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      ta[m] = (j < kb) ? ta[m] : 0.0f;
      tb[m] = (j + 1 < kb) ? tb[m] : 0.0f;
      pp[h2][m] = tadd(ta[m], tb[m]);
    }
  }
#pragma unroll
  for (int m = 0; m < MT; ++m) v[m] = tadd(pp[0][m], pp[1][m]);
}

// Tensor-core path: one warp computes a 16-row slice of one chunk against
// MT activation rows.  Per block and 16-wide half of it, the int8 weights
// and activations are converted exactly to fp16 and multiplied with
// mma.sync m16n8k16 (fp32 accumulate; every partial sum is an integer below
// 2^24, so the accumulator holds the exact int32 block dot).  Inside each
// half the 16 k positions are permuted identically for A and B (thread tig
// takes bytes 4tig..4tig+3 for its k pairs 2tig, 2tig+1 and 2tig+8,
// 2tig+9), which leaves the dot unchanged and makes every fragment one
// 32-bit shared-memory load.  Each block term is then rounded exactly as on
// the DP4A path and the 8 terms are summed in the same pairwise tree.
// out[nt][e]: rows row0 + g (e = 0, 1) and row0 + g + 8 (e = 2, 3), activation
// rows 8nt + 2tig + (e & 1); g = lane / 4, tig = lane % 4.
template <int MT>
__device__ __forceinline__ void block_terms_mma(const uint8_t* cq, const uint8_t* sc, int r, int row0,
                                                int j, const uint8_t* aq, const __half* ad, int mq,
                                                int md, float (&t)[MT / 8][4]) {
  constexpr int NTL = MT / 8;
  const int lane = threadIdx.x & 31, g = lane >> 2, tig = lane & 3;
  float acc[NTL][4];
#pragma unroll
  for (int nt = 0; nt < NTL; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[nt][e] = 0.0f;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t a[4];
    i8x4_to_h2x2(lds32(cq + ((2 * j + h) * r + row0 + g) * 16 + 4 * tig), a[0], a[2]);
    i8x4_to_h2x2(lds32(cq + ((2 * j + h) * r + row0 + g + 8) * 16 + 4 * tig), a[1], a[3]);
#pragma unroll
    for (int nt = 0; nt < NTL; ++nt) {
      uint32_t b0, b1;
      i8x4_to_h2x2(lds32(aq + (8 * nt + g) * mq + j * 32 + 16 * h + 4 * tig), b0, b1);
      mma_16816(acc[nt], a, b0, b1);
    }
  }
  const float dw0 =
      __half2float(__ushort_as_half(*reinterpret_cast<const unsigned short*>(sc + (j * r + row0 + g) * 2)));
  const float dw1 = __half2float(
      __ushort_as_half(*reinterpret_cast<const unsigned short*>(sc + (j * r + row0 + g + 8) * 2)));
#pragma unroll
  for (int nt = 0; nt < NTL; ++nt) {
    const float da0 = __half2float(ad[(8 * nt + 2 * tig) * md + j]);
    const float da1 = __half2float(ad[(8 * nt + 2 * tig + 1) * md + j]);
    t[nt][0] = __fmul_rn(acc[nt][0], __fmul_rn(dw0, da0));
    t[nt][1] = __fmul_rn(acc[nt][1], __fmul_rn(dw0, da1));
    t[nt][2] = __fmul_rn(acc[nt][2], __fmul_rn(dw1, da0));
    t[nt][3] = __fmul_rn(acc[nt][3], __fmul_rn(dw1, da1));
  }
}

template <int MT>
__device__ __forceinline__ void chunk_value_mma(const uint8_t* cq, int r, int kb, int row0,
                                                const uint8_t* aq, const __half* ad, int mq, int md,
                                                float (&v)[MT / 8][4]) {
  constexpr int NTL = MT / 8;
  const uint8_t* sc = cq + kb * r * 32;
  float q[2][NTL][4];
#pragma unroll
  for (int h4 = 0; h4 < 2; ++h4) {
    float p2[2][NTL][4];
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      float ta[NTL][4], tb[NTL][4];
      const int j = 4 * h4 + 2 * h2;
      // straight-line over all 8 blocks; blocks past kb count as zero
      block_terms_mma<MT>(cq, sc, r, row0, j, aq, ad, mq, md, ta);
      block_terms_mma<MT>(cq, sc, r, row0, j + 1, aq, ad, mq, md, tb);
#pragma unroll
      for (int nt = 0; nt < NTL; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          ta[nt][e] = (j < kb) ? ta[nt][e] : 0.0f;
          tb[nt][e] = (j + 1 < kb) ? tb[nt][e] : 0.0f;
          p2[h2][nt][e] = tadd(ta[nt][e], tb[nt][e]);
        }
    }
#pragma unroll
    for (int nt = 0; nt < NTL; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) q[h4][nt][e] = tadd(p2[0][nt][e], p2[1][nt][e]);
  }
#pragma unroll
  for (int nt = 0; nt < NTL; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) v[nt][e] = tadd(q[0][nt][e], q[1][nt][e]);
}

// tcgen05 path: 16 int8 values (one row's half block) to 16 fp16, written as
// the two core-matrix rows of a canonical K-major slice (k 0..7 at dst, k
// 8..15 at dst + 128).  The weights and the activations go through the same
// conversion, so their k order is permuted identically and every dot is
// unchanged.
__device__ __forceinline__ void store_f16_slice(uint8_t* dst, uint4 q) {
  uint32_t o[8];
  i8x4_to_h2x2(q.x, o[0], o[1]);
  i8x4_to_h2x2(q.y, o[2], o[3]);
  i8x4_to_h2x2(q.z, o[4], o[5]);
  i8x4_to_h2x2(q.w, o[6], o[7]);
  *reinterpret_cast<uint4*>(dst) = make_uint4(o[0], o[1], o[2], o[3]);
  *reinterpret_cast<uint4*>(dst + 128) = make_uint4(o[4], o[5], o[6], o[7]);
}

// pairwise tree of the P chunk values of a round (P a power of two); with
// H = 2 halves per chunk, a chunk's value is first the sum of its halves'
// (stored hstride apart)
template <int P, int H>
__device__ __forceinline__ float tree_of(const float* w, int stride, int hstride) {
  if constexpr (P == 1) {
    return H == 2 ? tadd(w[0], w[hstride]) : w[0];
  } else {
    return tadd(tree_of<P / 2, H>(w, stride, hstride),
                tree_of<P / 2, H>(w + (P / 2) * stride, stride, hstride));
  }
}

// SwiGLU epilogue of one tile: ysm holds the tile's outputs [R][MT] (the
// first R/2 rows gate rows j, the last R/2 the up rows of the same j); 8
// lanes per 32 consecutive j form h = silu(gate) * up and quantize it into
// block t * R/64 + jb of each activation row (only in the VAR_SWIGLU
// kernels, so the other kernels' registers are untouched).
template <int R, int MT, int NT>
__device__ __forceinline__ void swiglu_epilogue(const float* ysm, uint8_t* h_blocks, int64_t N, int M, int t,
                                             bool ok) {
  constexpr int JB = R / 64;  // output blocks per tile and row
  const int sub = threadIdx.x & 7, grp = threadIdx.x >> 3;
  for (int t0 = 0; t0 < MT * JB; t0 += NT / 8) {  // the same trip count in every thread
    const int task = t0 + grp;
    const int m = task / JB, jb = task - (task / JB) * JB;
    const bool on = ok && task < MT * JB && m < M;
    float hv[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if (on) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int jj = jb * 32 + 4 * sub + e;
        hv[e] = swiglu_one(ysm[jj * MT + m], ysm[(R / 2 + jj) * MT + m]);
      }
    }
    float4 v[1] = {make_float4(hv[0], hv[1], hv[2], hv[3])};
    uint32_t w[1];
    float d[1];
    quantize_group8<1>(v, w, d);
    if (on) store_block_lane(h_blocks + ((int64_t)m * (N / 64) + (int64_t)t * JB + jb) * BLOCK_BYTES, sub, w[0], d[0]);
  }
}

template <int R, int MT, bool FUSED, int V>
__global__ void __launch_bounds__(MCfg<MT>::THREADS, MCfg<MT>::MIN_CTAS) gemv_kernel(const GemvArgs a) {
  constexpr int P = RCfg<R>::P;
  constexpr int NCW = MCfg<MT>::NCW;
  constexpr int NT = NCW * 32;  // consumer threads
  constexpr int STAGES = MCfg<MT>::STAGES;
  constexpr int LV = log2_floor(ru_max<R, MT, V>()) + 1;
  constexpr bool TC = MT >= TC_MIN_MT;  // tensor-core path
  constexpr int HALVES = MCfg<MT>::HALVES;
  constexpr bool EXCHANGE = (P > 1) || TC || (HALVES > 1);
  // the abort decision is taken after the per-round exchange barrier
  static_assert(EXCHANGE || UCfg<R, MT, V>::ON, "every instantiation meets at a barrier each round");
  constexpr int RS = red_stride<MT>();
  constexpr int BAR_CONSUMERS = 1;  // named barrier of the consumer warps
  constexpr bool UM = UCfg<R, MT, V>::ON;  // tcgen05 path
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* stage_buf = smem;
  uint8_t* umA = smem + (size_t)STAGES * RCfg<R>::STAGE_BYTES;  // fp16 operands (tcgen05 path)
  uint8_t* umB = umA + UCfg<R, MT, V>::A_BYTES;
  uint8_t* act_base = umB + UCfg<R, MT, V>::B_BYTES;
  // the activation area is sized per launch (the unit's blocks), the rest follows it
  float* red = reinterpret_cast<float*>(act_base + a.act_smem);  // [2][HALVES][P][R][RS]
  uint64_t* full = reinterpret_cast<uint64_t*>(act_base + a.act_smem + red_bytes<R, MT, V>());
  uint64_t* empty = full + STAGES;
  volatile int* misc = reinterpret_cast<volatile int*>(empty + STAGES);
  // misc[0]: abort flag (set by the producer or a consumer; stops the
  // producer, starts the drain), misc[1]: "this CTA combines the tile",
  // misc[2]: rounds issued; tcgen05 path: misc[4..5] the MMA mbarrier, misc[6]
  // the tensor-memory base; misc[CAB], misc[CAB + 1]: the consumers' abort
  // flags, by parity of the round barriers.  A consumer whose wait gave up
  // sets the flag of the next round barrier before arriving there, and every
  // consumer reads that flag after passing it: between two barriers no one
  // writes the flag the others are reading, so all consumers leave at the same
  // barrier (misc[0], which the producer may set at any moment, is never read
  // for that decision).
  volatile int* cab = misc + UCfg<R, MT, V>::CAB;
  int bc = 0;  // round barriers passed (the same in every consumer)
  uint64_t* mma_bar = reinterpret_cast<uint64_t*>(const_cast<int*>(misc) + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(const_cast<int*>(misc) + 6);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NCW);
    }
    misc[0] = 0;
    misc[1] = 0;
    misc[2] = 0;
    cab[0] = 0;
    cab[1] = 0;
    if constexpr (UM) mbar_init(mma_bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_dependents();
  // A cluster (launched only when every unit covers all of K, so every CTA
  // stages the same blocks) stages its activations cooperatively.  Barrier
  // phase 1: every CTA of the cluster is running before any writes into
  // another's shared memory.  Phase 2: all staged blocks have landed.
  const uint32_t CL = cluster_nctarank();
  const uint32_t crank = cluster_ctarank();
  if (warp == NCW) {
    if (CL > 1) {
      // phase 1 for the producer warp: lane 0 arrives now and waits inside
      // produce(); lanes 1-31 arrive, wait and exit (exited threads do not
      // take part in phase 2)
      __syncwarp();
      cluster_arrive_aligned();
      if (lane != 0) {
        asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
        return;
      }
    }
    if (lane == 0) produce<R, STAGES>(a, stage_buf, full, empty, misc, CL);
    return;
  }
  if (CL > 1) {  // phase 1: every CTA of the cluster is running
    cluster_arrive_aligned();
    cluster_wait_aligned();
  }
  uint32_t tmem = 0;     // tensor memory of the block dots (tcgen05 path)
  uint32_t mphase = 0;   // parity of the MMA mbarrier's next completion
  if constexpr (UM) {
    if (warp == 0) tmem_alloc(tmem_slot, UCfg<R, MT, V>::TMEM_COLS);
    tc_fence_before_sync();
    named_bar_sync(BAR_CONSUMERS, NT);
    tc_fence_after_sync();
    tmem = *tmem_slot;
  }

  const int i = threadIdx.x % R;        // row inside the tile
  const int p = (threadIdx.x / R) % P;  // part: chunk p of each round
  const int hb = threadIdx.x / 128;     // half of the chunk (blocks 4hb..) when HALVES == 2
  // After each round's exchange, row i is merged by CG threads (t % R = i),
  // each owning MC of the MT output columns: the merge work and the binary
  // counter's registers are shared out.
  constexpr int CG = EXCHANGE ? (NT / R < MT ? NT / R : MT) : 1;
  constexpr int MC = MT / CG;
  const int mcg = threadIdx.x / R;
  const bool merger = mcg < CG;  // merges, counts and stores columns [mcg*MC, +MC) of row i
  const int UB = a.RU * P * CHUNK_BLOCKS;  // activation blocks per unit
  // laid out for MT rows (the planner sized the unit for MT), so rows
  // M <= m < MT read inside the staging area
  const ActLayout L = act_layout(act_base, MT, UB);
  int stage = 0;
  uint32_t phase = 0;
  int consumed = 0;
  bool ok = true;
  bool waited = false;
  int staged_s = -1;

  for (int u = blockIdx.x; u < a.units; u += gridDim.x) {
    const int t = u / a.S, s = u - (u / a.S) * a.S;
    const int r = tile_rows(t, a.N, R);
    const int c0 = s * a.RU * P;
    const int nrounds = min(a.RU, (a.nch - c0 + P - 1) / P);
    const int b0 = c0 * CHUNK_BLOCKS;
    const int nblk = min(UB, a.NB - b0);
    const int64_t n = (int64_t)t * R + i;

    if (!waited) {
      pdl_wait();
      waited = true;
    }
    if (s != staged_s) {  // units with the same K range reuse the staged blocks
      if (CL > 1) {        // once per CTA: the planner clusters only when S == 1
        stage_activations<FUSED, true, NT, MCfg<MT>::STAGE_BATCH>(a, L, b0, nblk, crank, CL);
        __syncwarp();
        cluster_arrive_aligned();
        cluster_wait_aligned();
      } else {
        named_bar_sync(BAR_CONSUMERS, NT);
        stage_activations<FUSED, false, NT, MCfg<MT>::STAGE_BATCH>(a, L, b0, nblk, 0u, 1u);
        named_bar_sync(BAR_CONSUMERS, NT);
      }
      staged_s = s;
    }
    if constexpr (FUSED) {
      if (a.A_out != nullptr && t == 0) write_act_blocks<NT>(a, L, b0, nblk);
    }

    float slot[MC][LV];
#pragma unroll
    for (int c = 0; c < MC; ++c)
#pragma unroll
      for (int l = 0; l < LV; ++l) slot[c][l] = 0.0f;

    for (int rho = 0; rho < nrounds; ++rho) {
      // the abort decision must be the same for every consumer (they meet
      // at the exchange barrier below), so it is read after that barrier
      const bool got = mbar_wait_bounded(&full[stage], phase, a.wait_ns);
      if (!got) {
        atomicOr(a.err, ERR_CONSUMER_WAIT);
        misc[0] = 1;
        cab[bc & 1] = 1;  // read by every consumer after the next round barrier
      }
      float mv[MC];  // this thread's merged columns of the round
      if constexpr (UM) {
        // the round is one chunk of the tile (P == 1); rows past r are zero,
        // blocks past kb are not multiplied and count as zero
        const int c = c0 + rho;
        const int kb = chunk_blocks(c, a.NB);
        const uint8_t* cq = stage_buf + (size_t)stage * RCfg<R>::STAGE_BYTES;
        if (got) {
#pragma unroll 1
          for (int task = threadIdx.x; task < kb * 2 * 128; task += NT) {
            const int row = task & 127, jh = task >> 7;  // jh = 2 * block + half
            const uint4 q = row < r ? lds128(cq + chunk_quant_off(jh >> 1, jh & 1, row, r)) : make_uint4(0u, 0u, 0u, 0u);
            store_f16_slice(umA + jh * UCfg<R, MT, V>::SLICE_A + (row >> 3) * 256 + (row & 7) * 16, q);
          }
#pragma unroll 1
          for (int task = threadIdx.x; task < kb * 2 * MT; task += NT) {
            const int m = task % MT, jh = task / MT;
            const uint4 q = lds128(L.q + m * L.mq + (rho * CHUNK_BLOCKS + (jh >> 1)) * 32 + (jh & 1) * 16);
            store_f16_slice(umB + jh * UCfg<R, MT, V>::SLICE_B + (m >> 3) * 256 + (m & 7) * 16, q);
          }
        }
        fence_proxy_async_smem();
        named_bar_sync(BAR_CONSUMERS, NT);
        const bool go = cab[bc & 1] == 0;  // the same in every consumer
        ++bc;
        if (go && threadIdx.x == 0) {
          tc_fence_after_sync();
          constexpr uint32_t IDESC = umma_idesc_f16(128, MT);
          for (int jh = 0; jh < 2 * kb; ++jh)
            umma_f16(tmem + (uint32_t)(MT * (jh >> 1)),
                     umma_smem_desc(smem_u32(umA + jh * UCfg<R, MT, V>::SLICE_A), 128, 256),
                     umma_smem_desc(smem_u32(umB + jh * UCfg<R, MT, V>::SLICE_B), 128, 256), IDESC, (jh & 1) != 0);
          umma_commit(mma_bar);
        }
        bool done = false;
        if (go) {
          done = mbar_wait_bounded(mma_bar, mphase, WAIT_LIMIT_NS);
          if (!done) {
            atomicOr(a.err, ERR_CONSUMER_WAIT);
            misc[0] = 1;
            cab[bc & 1] = 1;
          }
          done = __all_sync(0xffffffffu, done);  // tcgen05.ld is warp-collective
          if (done) mphase ^= 1u;
          tc_fence_after_sync();
        }
        // thread (row i, column group mcg) reads its row's dots of tokens
        // [MC mcg, MC mcg + MC): warp w reaches lanes 32 (w % 4) .. + 31.  The
        // two 4-block halves of the chunk are read and summed one after the
        // other (fewer live registers); the tree is that of the other paths.
        float half_sum[2][MC];
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t u[4][MC];
          if (done) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
              if (4 * hf + j < kb)
                tmem_ld8(tmem + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)(MT * (4 * hf + j) + MC * mcg), u[j]);
            tmem_ld_wait();
          }
          float dw[4];
#pragma unroll
          for (int j = 0; j < 4; ++j)
            dw[j] = (4 * hf + j < kb && i < r)
                        ? __half2float(*reinterpret_cast<const __half*>(cq + chunk_scale_off(4 * hf + j, i, r, kb)))
                        : 0.0f;
#pragma unroll
          for (int cc = 0; cc < MC; ++cc) {
            const __half* da = L.d + (mcg * MC + cc) * UB + rho * CHUNK_BLOCKS + 4 * hf;
            float t[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
              t[j] = (done && 4 * hf + j < kb)
                         ? __fmul_rn(__uint_as_float(u[j][cc]), __fmul_rn(dw[j], __half2float(da[j])))
                         : 0.0f;
            half_sum[hf][cc] = tadd(tadd(t[0], t[1]), tadd(t[2], t[3]));
          }
        }
#pragma unroll
        for (int cc = 0; cc < MC; ++cc) mv[cc] = tadd(half_sum[0][cc], half_sum[1][cc]);
        // a stage is released (and counted) only when its round was received:
        // after a failed wait no stage with a copy in flight is reused, and
        // the drain below waits for each of them
        __syncwarp();
        if (got) {
          if (lane == 0) mbar_arrive(&empty[stage]);
          ++consumed;
        }
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
        tc_fence_before_sync();
        named_bar_sync(BAR_CONSUMERS, NT);  // operands and tensor memory free for the next round
        const bool ab = cab[bc & 1] != 0;
        ++bc;
        if (!go || ab) {
          ok = false;
          break;
        }
      } else {
        float v[MT];
  #pragma unroll
        for (int m = 0; m < MT; ++m) v[m] = 0.0f;
        const int xpar = consumed & 1;
        float* rb = red + (size_t)xpar * HALVES * P * R * RS;  // [HALVES][P][R][RS]
        if constexpr (TC) {
          // 8 slices (16 rows x one chunk) per round, 8/NCW per warp (a loop, not
          // unrolled: one copy of the slice code keeps the instruction cache warm)
          const int g = lane >> 2, tig = lane & 3;
  #pragma unroll 1
          for (int k = 0; k < 8 / NCW; ++k) {
            const int sl = warp + k * NCW;
            const int ps = sl / (R / 16), row0 = (sl % (R / 16)) * 16;
            const int c = c0 + rho * P + ps;
            float cv[MT / 8][4];
  #pragma unroll
            for (int nt = 0; nt < MT / 8; ++nt)
  #pragma unroll
              for (int e = 0; e < 4; ++e) cv[nt][e] = 0.0f;
            if (got && c < a.nch) {
              const int blk = (rho * P + ps) * CHUNK_BLOCKS;
              const uint8_t* cq = stage_buf + (size_t)stage * RCfg<R>::STAGE_BYTES + ps * (r * CHUNK_BLOCKS * BLOCK_BYTES);
              chunk_value_mma<MT>(cq, r, chunk_blocks(c, a.NB), row0, L.q + blk * 32, L.d + blk, L.mq, UB, cv);
            }
  #pragma unroll
            for (int nt = 0; nt < MT / 8; ++nt)
  #pragma unroll
              for (int e = 0; e < 4; ++e)
                rb[(ps * R + row0 + g + (e >> 1) * 8) * RS + 8 * nt + 2 * tig + (e & 1)] = cv[nt][e];
          }
        } else {
          const int c = c0 + rho * P + p;
          if (got && c < a.nch) {
            const int blk = (rho * P + p) * CHUNK_BLOCKS;  // first block of the chunk in the unit
            const uint8_t* cq = stage_buf + (size_t)stage * RCfg<R>::STAGE_BYTES + p * (r * CHUNK_BLOCKS * BLOCK_BYTES);
            if constexpr (HALVES == 1)
              chunk_value<MT>(cq, r, chunk_blocks(c, a.NB), i, L.q + blk * 32, L.d + blk, L.mq, UB, v);
            else
              chunk_value_half<MT>(cq, r, chunk_blocks(c, a.NB), i, 4 * hb, L.q + blk * 32, L.d + blk, L.mq,
                                   UB, v);
          }
          if constexpr (EXCHANGE) {
  #pragma unroll
            for (int m = 0; m < MT; ++m) rb[((hb * P + p) * R + i) * RS + m] = v[m];
          }
        }
        // a stage is released (and counted) only when its round was received
        __syncwarp();
        if (got) {
          if (lane == 0) mbar_arrive(&empty[stage]);
          ++consumed;
        }
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
        if constexpr (EXCHANGE) {
          // the P chunk values of row i meet in shared memory; the buffer
          // written in round k was last read in round k-2, before the barrier
          // of round k-1 that every writer has passed
          named_bar_sync(BAR_CONSUMERS, NT);
          const bool ab = cab[bc & 1] != 0;
          ++bc;
          if (ab) {
            ok = false;
            break;
          }
          if (!merger) continue;
  #pragma unroll
          for (int c = 0; c < MC; ++c) mv[c] = tree_of<P, HALVES>(rb + i * RS + mcg * MC + c, R * RS, P * R * RS);
        } else {
          if (!got) {  // (unreachable: every instantiation exchanges, see the static_assert)
            ok = false;
            break;
          }
  #pragma unroll
          for (int c = 0; c < MC; ++c) mv[c] = v[c];  // CG == 1: the thread's own row
        }
      }
      // binary counter over the round subtrees (merging threads)
      bool placed = false;
#pragma unroll
      for (int l = 0; l < LV; ++l) {
        if (!placed) {
          if ((rho >> l) & 1) {
#pragma unroll
            for (int c = 0; c < MC; ++c) mv[c] = tadd(slot[c][l], mv[c]);
          } else {
#pragma unroll
            for (int c = 0; c < MC; ++c) slot[c][l] = mv[c];
            placed = true;
          }
        }
      }
    }

    // what is left merges from the lowest level up (= zero padding)
    float pv[MC];
    bool have = false;
#pragma unroll
    for (int c = 0; c < MC; ++c) pv[c] = 0.0f;
#pragma unroll
    for (int l = 0; l < LV; ++l) {
      if ((nrounds >> l) & 1) {
#pragma unroll
        for (int c = 0; c < MC; ++c) pv[c] = have ? tadd(slot[c][l], pv[c]) : slot[c][l];
        have = true;
      }
    }

    if (a.S == 1) {
      if constexpr (V != VAR_SWIGLU) {
        if (ok && merger && i < r) {
#pragma unroll
          for (int c = 0; c < MC; ++c) {
            const int m = mcg * MC + c;
            if (m < a.M) a.y[(int64_t)m * a.N + n] = pv[c];
          }
        }
      } else {
        // SwiGLU epilogue: the outputs meet in the exchange buffer ([R][MT],
        // after every thread is past the last round's exchange), then
        // swiglu_epilogue forms and quantizes h.
        float* ysm = red;
        named_bar_sync(BAR_CONSUMERS, NT);
        if (merger) {
#pragma unroll
          for (int c = 0; c < MC; ++c) ysm[i * MT + mcg * MC + c] = pv[c];
        }
        named_bar_sync(BAR_CONSUMERS, NT);
        swiglu_epilogue<R, MT, NT>(ysm, a.h_blocks, a.N, a.M, t, ok);
        named_bar_sync(BAR_CONSUMERS, NT);  // the exchange buffer is free for the next unit
      }
      continue;
    }

    // split along K: publish the unit value, take a ticket, last one combines
    if (ok && merger && i < r) {
#pragma unroll
      for (int c = 0; c < MC; ++c) {
        const int m = mcg * MC + c;
        if (m < a.M) a.ws_part[((int64_t)s * a.M + m) * a.N + n] = pv[c];
      }
    }
    __threadfence();
    named_bar_sync(BAR_CONSUMERS, NT);
    if (threadIdx.x == 0) {
      const bool any_abort = misc[0] != 0;
      const unsigned prev = any_abort ? 0u : atomicAdd(&a.ws_cnt[t], 1u);
      misc[1] = (!any_abort && prev == (unsigned)(a.S - 1)) ? 1 : 0;
    }
    named_bar_sync(BAR_CONSUMERS, NT);
    if (misc[1]) {
      __threadfence();
      if (i < r) {
        for (int m = p + hb * P; m < a.M; m += P * (NT / 128)) {  // every thread of the row takes some m
          float sl[SPLIT_LEVELS];
#pragma unroll
          for (int l = 0; l < SPLIT_LEVELS; ++l) sl[l] = 0.0f;
          const float* part = a.ws_part + (int64_t)m * a.N + n;
          const int64_t sstride = (int64_t)a.M * a.N;
          for (int s0 = 0; s0 < a.S; s0 += 16) {
            float pv16[16];
#pragma unroll
            for (int k = 0; k < 16; ++k)  // 16 independent loads in flight
              pv16[k] = (s0 + k < a.S) ? __ldcg(part + (int64_t)(s0 + k) * sstride) : 0.0f;
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              const int ss = s0 + k;
              if (ss < a.S) {
                float v = pv16[k];
                bool placed = false;
#pragma unroll
                for (int l = 0; l < SPLIT_LEVELS; ++l) {
                  if (!placed) {
                    if ((ss >> l) & 1) {
                      v = tadd(sl[l], v);
                    } else {
                      sl[l] = v;
                      placed = true;
                    }
                  }
                }
              }
            }
          }
          float out = 0.0f;
          bool h = false;
#pragma unroll
          for (int l = 0; l < SPLIT_LEVELS; ++l) {
            if ((a.S >> l) & 1) {
              out = h ? tadd(sl[l], out) : sl[l];
              h = true;
            }
          }
          a.y[(int64_t)m * a.N + n] = out;
        }
      }
      if (threadIdx.x == 0) a.ws_cnt[t] = 0u;
    }
  }

  // After a failed wait: let rounds that were issued but not received by
  // warp 0 land before the CTA's shared memory goes away.  Those stages were
  // never released, so each has at most one copy in flight; the drain keeps
  // the full bound whatever limit the ring's waits had.
  if (threadIdx.x == 0 && misc[0]) {
    for (int k = consumed; k < misc[2]; ++k) {
      if (!mbar_wait_bounded(&full[k % STAGES], (uint32_t)((k / STAGES) & 1), WAIT_LIMIT_NS)) {
        atomicOr(a.err, ERR_DRAIN_WAIT);
        break;
      }
    }
  }
  if constexpr (UM) {
    // the warp that allocated the tensor memory frees it once every consumer
    // is done with it; after an abort an MMA may still be in flight, which
    // lands first (bounded)
    tc_fence_before_sync();
    named_bar_sync(BAR_CONSUMERS, NT);
    if (warp == 0) {
      if (lane == 0 && misc[0]) (void)mbar_wait_bounded(mma_bar, mphase, WAIT_LIMIT_NS);
      __syncwarp();
      tmem_dealloc(tmem, UCfg<R, MT, V>::TMEM_COLS);
    }
  }
}

// Every libq8 kernel asks for the largest shared-memory carveout (the same
// for all, so an SM switching between kernels needs no reconfiguration).
// The attributes are set once per instantiation and device (a bit per
// device, set after success), not on every launch.
constexpr int ATTR_MAX_DEVICES = 64;
template <int R, int MT, bool FUSED, int V>
cudaError_t set_attributes() {
  static std::atomic<uint64_t> done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev >= 0 && dev < ATTR_MAX_DEVICES) ? (uint64_t)1 << dev : 0;
  if (bit != 0 && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(gemv_kernel<R, MT, FUSED, V>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)gemv_smem_bytes<R, MT, V>());
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(gemv_kernel<R, MT, FUSED, V>, cudaFuncAttributePreferredSharedMemoryCarveout,
                           (int)cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_release);
  return e;
}

template <int R, int MT, bool FUSED, int V>
cudaError_t launch_gemv_t(const GemvArgs& args, int grid, int cluster, bool pdl, cudaStream_t s) {
  cudaError_t e = set_attributes<R, MT, FUSED, V>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(MCfg<MT>::THREADS);
  cfg.dynamicSmemBytes = gemv_smem_bytes<R, MT, V>(args.act_smem);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (cluster > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = cluster;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, gemv_kernel<R, MT, FUSED, V>, args);
}

// CTAs of this instantiation that fit on an SM, queried once per device.
template <int R, int MT, bool FUSED, int V>
int occupancy_t() {
  static std::atomic<int> cached[ATTR_MAX_DEVICES];  // 0: not queried yet (static storage: zero)
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= ATTR_MAX_DEVICES) return 0;
  const int c = cached[dev].load(std::memory_order_acquire);
  if (c != 0) return c > 0 ? c : 0;
  if (set_attributes<R, MT, FUSED, V>() != cudaSuccess) return 0;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, gemv_kernel<R, MT, FUSED, V>, MCfg<MT>::THREADS,
                                                    gemv_smem_bytes<R, MT, V>()) != cudaSuccess)
    return 0;
  cached[dev].store(occ > 0 ? occ : -1, std::memory_order_release);
  return occ;
}

// Whether clusters of `cluster` CTAs of this kernel can be resident at all.
template <int R, int MT, bool FUSED, int V>
bool cluster_fits_t(int cluster) {
  if (set_attributes<R, MT, FUSED, V>() != cudaSuccess) return false;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster);
  cfg.blockDim = dim3(MCfg<MT>::THREADS);
  cfg.dynamicSmemBytes = gemv_smem_bytes<R, MT, V>();
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, gemv_kernel<R, MT, FUSED, V>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return n > 0;
}

// The variants a tile height and row count instantiate: the default always,
// tcgen05 for 128-row tiles with 16 rows, the SwiGLU epilogue for 64- and
// 128-row tiles; another request falls back to the default.
template <int R, int MT, bool FUSED>
cudaError_t launch_gemv_v(const GemvArgs& args, int var, int grid, int cluster, bool pdl, cudaStream_t s) {
  if constexpr (R == 128 && MT == 16) {
    if (var == VAR_TCGEN05) return launch_gemv_t<R, MT, FUSED, VAR_TCGEN05>(args, grid, cluster, pdl, s);
  }
  if constexpr (R >= 64) {
    if (var == VAR_SWIGLU) return launch_gemv_t<R, MT, FUSED, VAR_SWIGLU>(args, grid, cluster, pdl, s);
  }
  return launch_gemv_t<R, MT, FUSED, VAR_DEFAULT>(args, grid, cluster, pdl, s);
}
template <int R, int MT, bool FUSED>
int occupancy_v(int var) {
  if constexpr (R == 128 && MT == 16) {
    if (var == VAR_TCGEN05) return occupancy_t<R, MT, FUSED, VAR_TCGEN05>();
  }
  return occupancy_t<R, MT, FUSED, VAR_DEFAULT>();  // the SwiGLU variant has the default's resources
}
template <int R, int MT, bool FUSED>
bool cluster_fits_v(int var, int c) {
  if constexpr (R == 128 && MT == 16) {
    if (var == VAR_TCGEN05) return cluster_fits_t<R, MT, FUSED, VAR_TCGEN05>(c);
  }
  return cluster_fits_t<R, MT, FUSED, VAR_DEFAULT>(c);
}

// Per-R translation units instantiate these for every MT and FUSED.
template <int R>
cudaError_t launch_gemv_r(const GemvArgs& args, int MT, bool fused, int var, int grid, int cluster, bool pdl,
                         cudaStream_t s);
template <int R>
int occupancy_r(int MT, bool fused, int var);
template <int R>
bool cluster_fits_r(int MT, bool fused, int var, int cluster);

#define Q8_INSTANTIATE_R(R)                                                                          \
  template <>                                                                                        \
  cudaError_t launch_gemv_r<R>(const GemvArgs& args, int MT, bool fused, int var, int grid,          \
                               int cluster, bool pdl, cudaStream_t s) {                              \
    switch (MT) {                                                                                    \
      case 1: return fused ? launch_gemv_v<R, 1, true>(args, var, grid, cluster, pdl, s)             \
                           : launch_gemv_v<R, 1, false>(args, var, grid, cluster, pdl, s);           \
      case 2: return fused ? launch_gemv_v<R, 2, true>(args, var, grid, cluster, pdl, s)             \
                           : launch_gemv_v<R, 2, false>(args, var, grid, cluster, pdl, s);           \
      case 4: return fused ? launch_gemv_v<R, 4, true>(args, var, grid, cluster, pdl, s)             \
                           : launch_gemv_v<R, 4, false>(args, var, grid, cluster, pdl, s);           \
      case 8: return fused ? launch_gemv_v<R, 8, true>(args, var, grid, cluster, pdl, s)             \
                           : launch_gemv_v<R, 8, false>(args, var, grid, cluster, pdl, s);           \
      default: return fused ? launch_gemv_v<R, 16, true>(args, var, grid, cluster, pdl, s)           \
                            : launch_gemv_v<R, 16, false>(args, var, grid, cluster, pdl, s);         \
    }                                                                                                \
  }                                                                                                  \
  template <>                                                                                        \
  int occupancy_r<R>(int MT, bool fused, int var) {                                                  \
    switch (MT) {                                                                                    \
      case 1: return fused ? occupancy_v<R, 1, true>(var) : occupancy_v<R, 1, false>(var);           \
      case 2: return fused ? occupancy_v<R, 2, true>(var) : occupancy_v<R, 2, false>(var);           \
      case 4: return fused ? occupancy_v<R, 4, true>(var) : occupancy_v<R, 4, false>(var);           \
      case 8: return fused ? occupancy_v<R, 8, true>(var) : occupancy_v<R, 8, false>(var);           \
      default: return fused ? occupancy_v<R, 16, true>(var) : occupancy_v<R, 16, false>(var);        \
    }                                                                                                \
  }                                                                                                  \
  template <>                                                                                        \
  bool cluster_fits_r<R>(int MT, bool fused, int var, int c) {                                       \
    switch (MT) {                                                                                    \
      case 1: return fused ? cluster_fits_v<R, 1, true>(var, c) : cluster_fits_v<R, 1, false>(var, c); \
      case 2: return fused ? cluster_fits_v<R, 2, true>(var, c) : cluster_fits_v<R, 2, false>(var, c); \
      case 4: return fused ? cluster_fits_v<R, 4, true>(var, c) : cluster_fits_v<R, 4, false>(var, c); \
      case 8: return fused ? cluster_fits_v<R, 8, true>(var, c) : cluster_fits_v<R, 8, false>(var, c); \
      default: return fused ? cluster_fits_v<R, 16, true>(var, c) : cluster_fits_v<R, 16, false>(var, c); \
    }                                                                                                \
  }

}  // namespace q8
