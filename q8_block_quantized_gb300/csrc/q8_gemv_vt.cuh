// q8_gemv_vt.cuh -- the decode GEMV for 4 to 32 activation rows per launch.
//
// Work decomposition.  A virtual tile is 128 consecutive output rows: G =
// 128 / R tiles of the packed layout (R = 16, 32, 64 or 128 rows, fixed by
// N).  A work unit is one virtual tile times RU consecutive chunks of 8
// blocks along K; a tile is split along K into S units when that is needed
// to fill the SMs or to fit the unit's activations in shared memory (the
// split units' values are merged by the CTA that finishes last).  A round is
// one chunk of every tile of the virtual tile: G bulk copies into one stage
// of a ring (one 128-row chunk, 34,816 bytes).  Compared with one tile of R
// rows per CTA over all of K, a CTA stages the activations of a K range S
// times shorter, which is what the cost of a unit grows with once several
// activation rows share the launch.
//
// Block dots.  Consumer warp w owns rows 16w..16w+15 of the virtual tile.
// Per block and 16-wide half it converts its int8 weight fragments exactly
// to fp16 (byte permute against 0x64, then a subtraction: exact for
// [-128, 127]) and multiplies them with mma.sync m16n8k16 (fp32 accumulate;
// every partial sum is an integer below 2^24, so the accumulator holds the
// exact int32 block dot) by the activation fragments, which were converted
// to fp16 once when the unit's activations were staged.  Inside each half,
// thread tig takes the k values 4tig..4tig+3 for its k pairs (2tig, 2tig+1)
// and (2tig+8, 2tig+9) in both operands: the dot is unchanged and each
// fragment is one shared-memory load.  (On GB300 fp16 mma.sync runs 4x the
// operations per second of int8 mma.sync or dp4a.)
//
// Reduction order.  The terms t_b = float(isum) * (d_w * d_a) are summed
// in the canonical order of the library: the pairwise tree over the block
// index, padded with zeros to a power of two.  A chunk is an aligned
// 8-block subtree (computed in registers), rounds merge with a binary
// counter per warp (merge with the left sibling while the round index bit
// is 1; leftovers merge from the lowest level up = zero padding), and split
// units merge the same way in split order.  So an output's bits depend only
// on its row of W, its row of activations and K: they equal those of the
// one- and two-row kernel and do not depend on M, the batch position, the
// split or the tile height.
//
// Pipeline.  One lane of the producer warp streams every unit's rounds into
// the ring (bounded mbarrier waits; a failed wait sets the device error
// word and aborts the CTA).  The consumers execute griddepcontrol.wait
// before reading activations or writing anything, so with programmatic
// dependent launch the weights stream while the previous kernel finishes.
#pragma once

#include <cuda_runtime.h>

#include "q8_device.cuh"
#include "q8_f32x2.cuh"
#include "q8_internal.h"

namespace q8 {
namespace vt {

constexpr int VR = 128;                                       // rows of a virtual tile
constexpr int NCW = 8;                                        // consumer warps, one 16-row slice each
constexpr int NT = NCW * 32;                                  // consumer threads
constexpr int THREADS = NT + 32;                              // + the producer warp
constexpr int STAGES = 3;
constexpr int STAGE_BYTES = VR * CHUNK_BLOCKS * BLOCK_BYTES;  // 34,816
constexpr int SLOT_UNIT = CHUNK_BLOCKS * BLOCK_BYTES;         // 272 bytes per row of a chunk
constexpr int SMEM_LIMIT = 232448;                            // dynamic shared memory of one CTA
constexpr int MISC_BYTES = (2 * STAGES + 3) * 8 + 24;         // mbarriers + flags
constexpr int ACT_BUDGET = SMEM_LIMIT - STAGES * STAGE_BYTES - MISC_BYTES;
constexpr int MAX_SPLITS = 64;
constexpr int MAX_CLUSTER = 8;                                 // portable cluster size
constexpr int SPLIT_LV = 7;                                   // counter levels for S <= 127
constexpr int MAX_TILES_SPLIT = 4096;                         // tickets in the workspace prefix
constexpr size_t TICKET_BYTES = (size_t)MAX_TILES_SPLIT * 4;

enum : unsigned { ERR_PRODUCER_WAIT = 1u, ERR_CONSUMER_WAIT = 2u, ERR_DRAIN_WAIT = 4u };

__host__ __device__ constexpr int ilog2(int v) { return v <= 1 ? 0 : 1 + ilog2(v >> 1); }

// Shared memory for the raw activation copies of the staging: at least
// RAW_MIN bytes (one 32-row piece of 8 fp32 blocks), otherwise what the ring
// and the staged activations leave.
constexpr int RAW_MIN = 32 * 8 * 128;

template <int MT>
struct Cfg {
  static constexpr int NTL = MT < 8 ? 1 : MT / 8;  // n-tiles of 8 activation rows
  static constexpr int MP = NTL * 8;               // staged activation rows (padded to the n-tiles)
  // staged bytes per block of a unit: MP rows of 32 fp16 quants + MP fp32 scales
  static constexpr int PER_BLOCK = MP * 64 + MP * 4;
  // blocks of a unit's K range (a multiple of 8)
  // (RAW_MIN bytes stay free for the raw copies the staging works from)
  static constexpr int UB_MAX = (ACT_BUDGET - RAW_MIN - MP * 32) / PER_BLOCK / CHUNK_BLOCKS * CHUNK_BLOCKS;
  static constexpr int RU_MAX = UB_MAX / CHUNK_BLOCKS;
  static constexpr int LV = ilog2(RU_MAX) + 1;     // round counter levels
  // staging passes (32 blocks each) with their loads in flight together
  static constexpr int BATCH = MT >= 8 ? 8 : 4;
};

// Staged activations of a unit (UB blocks): fp16 quants of row m, block b at
// q + m * rsb + b * 64 (rsb = UB * 64 + 32: rows 32 bytes apart modulo 128,
// so the 8 rows of a fragment load hit distinct banks), fp32 scales
// block-major at d[b * MP + m] (a thread's two columns are one 8-byte load).
__host__ __device__ constexpr int act_rsb(int UB) { return UB * 64 + 32; }
template <int MT>
__host__ __device__ constexpr int act_bytes(int UB) {
  return Cfg<MT>::MP * act_rsb(UB) + UB * Cfg<MT>::MP * 4;
}
// Every launch takes the whole SMEM_LIMIT: ring, staged activations, then
// the raw area (the rest), then the mbarriers and flags.
template <int MT>
__host__ __device__ constexpr int raw_bytes(int UB) {
  return (SMEM_LIMIT - STAGES * STAGE_BYTES - act_bytes<MT>(UB) - MISC_BYTES) / 16 * 16;
}
constexpr size_t smem_bytes() { return (size_t)SMEM_LIMIT; }

struct Args {
  const uint8_t* W;
  const uint8_t* A;      // activation blocks [M][NB] (unfused)
  const float* x;        // fp32 activations [M][K] (fused)
  uint8_t* A_out;        // fused: optional activation blocks out
  float* y;              // [M][N]
  float* ws_part;        // [S][M][Np] partials (S > 1)
  unsigned* ws_cnt;      // [TV] tickets (S > 1)
  unsigned* err;         // device error word
  uint64_t wait_ns;      // limit of the ring's and the staging's waits (WAIT_LIMIT_NS unless a test shortens it)
  int64_t N;
  int NB, nch, T, R, G, TV, M, RU, S, units, UB, Np;
  int raw_bytes;         // shared memory for the staging's raw copies (raw_bytes<MT>(UB))
  // optional: the staged activations of every K range, prepared by the image
  // kernel ([S] images of act_bytes<MT>(UB) bytes, 16-byte aligned); the
  // staging is then one bulk copy per unit
  const uint8_t* img;
  // CTAs of a cluster (1: none).  With cl = S > 1 each cluster owns whole
  // virtual tiles, its CTA of rank s the K split s, and the splits combine
  // through distributed shared memory instead of the workspace.
  int cl;
};

// Units of this CTA: first, first + step, ... below end.  Plain launches
// take units blockIdx.x, blockIdx.x + gridDim.x, ...; in a cluster the CTA
// of rank s takes split s of virtual tiles cid, cid + ncl, ... (cid: its
// cluster, ncl: the clusters of the grid; clusters are consecutive CTAs).
struct UnitRange {
  int first, step, end;
};
__device__ __forceinline__ UnitRange unit_range(const Args& a) {
  if (a.cl > 1) {
    const int rank = (int)blockIdx.x % a.cl, cid = (int)blockIdx.x / a.cl;
    return {rank * a.TV + cid, (int)gridDim.x / a.cl, (rank + 1) * a.TV};
  }
  return {(int)blockIdx.x, (int)gridDim.x, a.units};
}

__device__ __forceinline__ uint2 lds64(const void* p) { return *reinterpret_cast<const uint2*>(p); }

// ---- producer: one lane streams the rounds of every unit of this CTA -------
// In a cluster the producer lane also completes the cluster barrier that
// the kernel opens (mbarriers initialised everywhere): it waits once its
// first STAGES rounds are issued, so streaming does not wait for the cluster.
__device__ __forceinline__ void produce(const Args& a, uint8_t* stage_buf, uint64_t* full, uint64_t* empty,
                                        volatile int* misc) {
  const uint64_t pol = l2_policy_evict_first();
  int stage = 0;
  uint32_t phase = 0;
  int issued = 0;
  bool stop = false;
  bool cluster_done = a.cl == 1;
  const int slot = a.R * SLOT_UNIT;
  const UnitRange ur = unit_range(a);
  for (int u = ur.first; u < ur.end && !stop; u += ur.step) {
    const int s = u / a.TV, tv = u - s * a.TV;
    const int c0 = s * a.RU;
    const int nr = min(a.RU, a.nch - c0);
    for (int rho = 0; rho < nr; ++rho) {
      if (!cluster_done && issued == STAGES) {
        asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
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
      const int c = c0 + rho;
      const int kb = chunk_blocks(c, a.NB);
      uint8_t* dst0 = stage_buf + (size_t)stage * STAGE_BYTES;
      uint32_t total = 0;
      for (int g = 0; g < a.G; ++g) {  // ragged tails (< 16 bytes each) by hand, before the arrival
        const int t = tv * a.G + g;
        if (t >= a.T) break;
        const int r = tile_rows(t, a.N, a.R);
        const uint8_t* src = a.W + chunk_offset(t, c, r, a.R, a.NB);
        const uint32_t bytes = (uint32_t)(kb * r * BLOCK_BYTES);
        const uint32_t bulk = bytes & ~15u;
        uint8_t* dst = dst0 + (size_t)g * slot;
        for (uint32_t k = bulk; k < bytes; ++k) dst[k] = src[k];
        total += bulk;
      }
      mbar_arrive_expect_tx(&full[stage], total);
      for (int g = 0; g < a.G; ++g) {
        const int t = tv * a.G + g;
        if (t >= a.T) break;
        const int r = tile_rows(t, a.N, a.R);
        const uint32_t bulk = (uint32_t)(kb * r * BLOCK_BYTES) & ~15u;
        if (bulk > 0)
          bulk_g2s(dst0 + (size_t)g * slot, a.W + chunk_offset(t, c, r, a.R, a.NB), bulk, &full[stage], pol);
      }
      misc[2] = ++issued;
      if (++stage == STAGES) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
  if (!cluster_done) asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}

// ---- activation staging ------------------------------------------------------
// The unit's activation blocks [b0, b0 + nblk) of rows < M, converted into
// the staged layout: fp16 quants (exact) and fp32 scales (the binary16
// value, exact).  The raw data comes into shared memory by bulk copies in
// pieces of PB blocks of every row (one thread issues one copy per row, so a
// piece costs one round trip to L2), then eight consecutive lanes take one
// block: lane s holds values 4s..4s+3 (fused: quantized in the warp exactly
// as q8_quantize_act does; unfused: the block's quants), lane 0 the scale.
//   fused:   raw row m holds x[m][32 (b0 + p0) ...] as fp32, 128 bytes a block;
//   unfused: raw row m holds the bytes of the 34-byte blocks at the same
//            offset modulo 16 as in global memory: the 16-byte-aligned body
//            by a bulk copy, the unaligned head and tail (< 16 bytes each)
//            by plain loads, so nothing outside the blocks is read.
template <int MT>
__device__ __forceinline__ void put_block(uint8_t* aq, float* ad, int rsb, int m, int blk, int sub, uint32_t w,
                                          float d) {
  uint32_t lo, hi;
  i8x4_to_h2x2(w, lo, hi);
  *reinterpret_cast<uint2*>(aq + (size_t)m * rsb + blk * 64 + sub * 8) = make_uint2(lo, hi);
  if (sub == 0) ad[blk * Cfg<MT>::MP + m] = d;
}

struct RawRing {
  uint64_t* bar;  // completion of a piece's copies
  uint32_t phase;
  int issued, waited;  // pieces (thread 0's counts, for the drain after a failure)
};

template <int MT, bool FUSED>
__device__ __forceinline__ void stage_act(const Args& a, uint8_t* aq, float* ad, int rsb, uint8_t* raw, int b0,
                                          int nblk, RawRing& rr, volatile int* misc) {
  constexpr int BAR_CONSUMERS = 1;
  if (a.img != nullptr) {
    // the K range's staged image, prepared once for every CTA: one bulk copy
    named_bar_sync(BAR_CONSUMERS, NT);  // the staged blocks are free
    const uint32_t bytes = (uint32_t)act_bytes<MT>(a.UB);
    if (threadIdx.x == 0 && misc[0] == 0) {
      mbar_arrive_expect_tx(rr.bar, bytes);
      bulk_g2s_nohint(aq, a.img + (size_t)(b0 / a.UB) * bytes, bytes, rr.bar);
      ++rr.issued;
    }
    if (misc[0] == 0) {
      const bool got = mbar_wait_bounded(rr.bar, rr.phase, a.wait_ns);
      if (!got) {
        atomicOr(a.err, ERR_CONSUMER_WAIT);
        misc[0] = 1;
      } else if (threadIdx.x == 0) {
        ++rr.waited;
      }
    }
    rr.phase ^= 1u;
    return;  // every consumer waited for the copy itself
  }
  constexpr int BPP = NT / 8;  // blocks per pass
  constexpr int BATCH = FUSED ? 4 : 8;
  const int64_t K = (int64_t)a.NB * QK;
  const int row_bytes = a.raw_bytes / a.M / 16 * 16;  // raw bytes per activation row and piece
  const int PB = FUSED ? row_bytes / 128 : (row_bytes - 32) / BLOCK_BYTES;
  const int sub = threadIdx.x & 7, slot = threadIdx.x >> 3;
  for (int p0 = 0; p0 < nblk; p0 += PB) {
    const int pb = min(PB, nblk - p0);
    named_bar_sync(BAR_CONSUMERS, NT);  // the raw area and the staged blocks are free
    // warp 0 fills the raw area: lane 0 announces the bytes and issues the
    // bulk copies, then (unfused) lane m copies row m's unaligned head and
    // tail with 16-bit loads, and lane 0 arrives once all lanes are done
    if (threadIdx.x < 32) {
      const bool go = __shfl_sync(0xffffffffu, misc[0] == 0 ? 1 : 0, 0) != 0;
      if (go) {
        const int lane = threadIdx.x;
        if (lane == 0) {
          uint32_t total = 0;
          for (int m = 0; m < a.M; ++m) {
            if constexpr (FUSED) {
              total += (uint32_t)pb * 128u;
            } else {
              const uintptr_t s0 = reinterpret_cast<uintptr_t>(a.A + ((int64_t)m * a.NB + b0 + p0) * BLOCK_BYTES);
              const uintptr_t e0 = s0 + (uintptr_t)pb * BLOCK_BYTES;
              const uintptr_t lo = (s0 + 15) & ~(uintptr_t)15, hi = e0 & ~(uintptr_t)15;
              if (hi > lo) total += (uint32_t)(hi - lo);
            }
          }
          mbar_expect_tx(rr.bar, total);
          for (int m = 0; m < a.M; ++m) {
            uint8_t* dst = raw + (size_t)m * row_bytes;
            if constexpr (FUSED) {
              bulk_g2s_nohint(dst, a.x + (int64_t)m * K + (int64_t)(b0 + p0) * QK, (uint32_t)pb * 128u, rr.bar);
            } else {
              const uintptr_t s0 = reinterpret_cast<uintptr_t>(a.A + ((int64_t)m * a.NB + b0 + p0) * BLOCK_BYTES);
              const uintptr_t e0 = s0 + (uintptr_t)pb * BLOCK_BYTES;
              const uintptr_t lo = (s0 + 15) & ~(uintptr_t)15, hi = e0 & ~(uintptr_t)15;
              if (hi > lo)
                bulk_g2s_nohint(dst + (s0 & 15) + (lo - s0), reinterpret_cast<const void*>(lo), (uint32_t)(hi - lo),
                                rr.bar);
            }
          }
        }
        if constexpr (!FUSED) {
          // block bytes start 2-byte aligned, so heads and tails are whole 16-bit words
          for (int m = lane; m < a.M; m += 32) {
            const uintptr_t s0 = reinterpret_cast<uintptr_t>(a.A + ((int64_t)m * a.NB + b0 + p0) * BLOCK_BYTES);
            const uintptr_t e0 = s0 + (uintptr_t)pb * BLOCK_BYTES;
            const uintptr_t lo = (s0 + 15) & ~(uintptr_t)15, hi = e0 & ~(uintptr_t)15;
            unsigned short* d0 = reinterpret_cast<unsigned short*>(raw + (size_t)m * row_bytes + (s0 & 15));
            if (hi > lo) {
              // head [s0, lo) and tail [hi, e0): at most 7 words each, all
              // loads in flight before the stores
              unsigned short hw[7], tw[7];
#pragma unroll
              for (int k = 0; k < 7; ++k) {
                const uintptr_t qh = s0 + 2 * k, qt = hi + 2 * k;
                hw[k] = qh < lo ? __ldcg(reinterpret_cast<const unsigned short*>(qh)) : (unsigned short)0;
                tw[k] = qt < e0 ? __ldcg(reinterpret_cast<const unsigned short*>(qt)) : (unsigned short)0;
              }
#pragma unroll
              for (int k = 0; k < 7; ++k) {
                if (s0 + 2 * k < lo) d0[k] = hw[k];
                if (hi + 2 * k < e0) d0[((hi - s0) >> 1) + k] = tw[k];
              }
            } else {  // no aligned body: the whole piece of this row (< 32 bytes) by plain loads
              unsigned short w[16];
#pragma unroll
              for (int k = 0; k < 16; ++k)
                w[k] = s0 + 2 * k < e0 ? __ldcg(reinterpret_cast<const unsigned short*>(s0 + 2 * k)) : (unsigned short)0;
#pragma unroll
              for (int k = 0; k < 16; ++k)
                if (s0 + 2 * k < e0) d0[k] = w[k];
            }
          }
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(rr.bar);
          ++rr.issued;
        }
      }
    }
    bool got = false;
    if (misc[0] == 0) {
      got = mbar_wait_bounded(rr.bar, rr.phase, a.wait_ns);
      if (!got) {
        atomicOr(a.err, ERR_CONSUMER_WAIT);
        misc[0] = 1;
      }
    }
    rr.phase ^= 1u;
    if (got && threadIdx.x == 0) ++rr.waited;
    // Block i of the piece (row-major over rows m < M and blocks kk < pb) is
    // taken by lane group i % 32 in pass i / 32: each thread starts at
    // i = slot with one division per piece and steps by 32 in constant time.
    // Trip counts are uniform across the CTA (the shuffles of the fused
    // quantization see full warps), and a batch issues all its loads before
    // any store.
    const int total_blocks = a.M * pb;
    const int q32 = BPP / pb, r32 = BPP - (BPP / pb) * pb;
    int m_cur = slot / pb, k_cur = slot - (slot / pb) * pb;
    const uintptr_t a_row0 = FUSED ? 0 : reinterpret_cast<uintptr_t>(a.A + (int64_t)(b0 + p0) * BLOCK_BYTES);
    const uintptr_t a_rstride = (uintptr_t)a.NB * BLOCK_BYTES;
    for (int base = 0; base < total_blocks; base += BPP * BATCH) {
      int mm[BATCH], kk[BATCH];
      bool on[BATCH];
#pragma unroll
      for (int q = 0; q < BATCH; ++q) {
        on[q] = got && base + q * BPP + slot < total_blocks;
        mm[q] = m_cur;
        kk[q] = k_cur;
        k_cur += r32;
        m_cur += q32;
        if (k_cur >= pb) {
          k_cur -= pb;
          ++m_cur;
        }
      }
      if constexpr (FUSED) {
        float4 v[BATCH];
#pragma unroll
        for (int q = 0; q < BATCH; ++q)
          v[q] = on[q] ? *reinterpret_cast<const float4*>(raw + (size_t)mm[q] * row_bytes + kk[q] * 128 + sub * 16)
                       : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        uint32_t w[BATCH];
        float d[BATCH];
        quantize_group8<BATCH>(v, w, d);
#pragma unroll
        for (int q = 0; q < BATCH; ++q)
          if (on[q]) put_block<MT>(aq, ad, rsb, mm[q], p0 + kk[q], sub, w[q], d[q]);
      } else {
        uint32_t w[BATCH];
        unsigned short dbits[BATCH];
#pragma unroll
        for (int q = 0; q < BATCH; ++q) {
          w[q] = 0u;
          dbits[q] = 0;
          if (on[q]) {
            // row m's bytes sit at the offset they have modulo 16 in global memory
            const uintptr_t delta = (a_row0 + (uintptr_t)mm[q] * a_rstride) & 15;
            const unsigned short* blk = reinterpret_cast<const unsigned short*>(
                raw + (size_t)mm[q] * row_bytes + delta + kk[q] * BLOCK_BYTES);
            w[q] = (uint32_t)blk[1 + 2 * sub] | ((uint32_t)blk[2 + 2 * sub] << 16);
            dbits[q] = blk[0];
          }
        }
#pragma unroll
        for (int q = 0; q < BATCH; ++q)
          if (on[q]) put_block<MT>(aq, ad, rsb, mm[q], p0 + kk[q], sub, w[q], __half2float(__ushort_as_half(dbits[q])));
      }
    }
  }
  named_bar_sync(BAR_CONSUMERS, NT);  // staged blocks visible to every consumer
}

// Fused path: the CTAs that own virtual tile 0 publish the quantized
// activations of their K range (every K range is covered once by tile 0),
// converted back from the staged fp16 quants and fp32 scales (both exact).
template <int MT>
__device__ __forceinline__ void write_act_out(const Args& a, const uint8_t* aq, const float* ad, int rsb, int b0,
                                              int nblk) {
  const int total = a.M * nblk * 8;
  for (int idx = threadIdx.x; idx < total; idx += NT) {
    const int sub = idx & 7, blkm = idx >> 3;
    const int m = blkm / nblk, blk = blkm - m * nblk;
    const uint2 h = lds64(aq + (size_t)m * rsb + blk * 64 + sub * 8);
    const __half2 lo = *reinterpret_cast<const __half2*>(&h.x), hi = *reinterpret_cast<const __half2*>(&h.y);
    const uint32_t q0 = (uint32_t)(__half2int_rn(__low2half(lo)) & 0xff), q1 = (uint32_t)(__half2int_rn(__high2half(lo)) & 0xff);
    const uint32_t q2 = (uint32_t)(__half2int_rn(__low2half(hi)) & 0xff), q3 = (uint32_t)(__half2int_rn(__high2half(hi)) & 0xff);
    unsigned short* o16 = reinterpret_cast<unsigned short*>(a.A_out + ((int64_t)m * a.NB + b0 + blk) * BLOCK_BYTES);
    o16[1 + 2 * sub] = (unsigned short)(q0 | (q1 << 8));
    o16[2 + 2 * sub] = (unsigned short)(q2 | (q3 << 8));
    if (sub == 0) o16[0] = __half_as_ushort(__float2half_rn(ad[blk * Cfg<MT>::MP + m]));
  }
}

// ---- block terms of one warp's 16-row slice ----------------------------------
// t[nt][0]: rows rloc + g, t[nt][1]: rows rloc + g + 8 of the tile, each a
// pair for activation rows 8nt + 2tig and 8nt + 2tig + 1; g = lane / 4,
// tig = lane % 4.  cq: the chunk of this tile (r rows, packed layout), sc:
// its scales, j: the block in the chunk, blk: the block in the unit's
// staged activations.
template <int MT>
__device__ __forceinline__ void block_terms(const uint8_t* cq, const uint8_t* sc, int r, int rloc, int j,
                                            const uint8_t* aq, const float* ad, int rsb, int blk,
                                            uint64_t (&t)[Cfg<MT>::NTL][2]) {
  constexpr int NTL = Cfg<MT>::NTL;
  const int lane = threadIdx.x & 31, g = lane >> 2, tig = lane & 3;
  float acc[NTL][4];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t af[4];
    i8x4_to_h2x2(lds32(cq + ((2 * j + h) * r + rloc + g) * 16 + 4 * tig), af[0], af[2]);
    i8x4_to_h2x2(lds32(cq + ((2 * j + h) * r + rloc + g + 8) * 16 + 4 * tig), af[1], af[3]);
#pragma unroll
    for (int nt = 0; nt < NTL; ++nt) {
      const uint2 b = lds64(aq + (size_t)(8 * nt + g) * rsb + blk * 64 + h * 32 + tig * 8);
      if (h == 0) {
        mma_16816_c0(acc[nt], af, b.x, b.y);
      } else {
        mma_16816_acc(acc[nt], af, b.x, b.y);
      }
    }
  }
  const float dw0 =
      __half2float(__ushort_as_half(*reinterpret_cast<const unsigned short*>(sc + (j * r + rloc + g) * 2)));
  const float dw1 =
      __half2float(__ushort_as_half(*reinterpret_cast<const unsigned short*>(sc + (j * r + rloc + g + 8) * 2)));
  const uint64_t w0 = f2_pack(dw0, dw0), w1 = f2_pack(dw1, dw1);
#pragma unroll
  for (int nt = 0; nt < NTL; ++nt) {
    // d_a of the thread's two activation rows: one 8-byte load
    const uint64_t da = *reinterpret_cast<const uint64_t*>(ad + blk * Cfg<MT>::MP + 8 * nt + 2 * tig);
    // t_b = float(isum) * (d_w * d_a), each product rounded once
    t[nt][0] = f2_mul(f2_pack(acc[nt][0], acc[nt][1]), f2_mul(w0, da));
    t[nt][1] = f2_mul(f2_pack(acc[nt][2], acc[nt][3]), f2_mul(w1, da));
  }
}

// The 8-block pairwise tree of one chunk (kb <= 8 blocks; terms of blocks at
// or past kb are zero).  All 8 blocks run in straight-line code: reads past
// kb stay inside the stage slot and the staged activations.
template <int MT>
__device__ __forceinline__ void chunk_value(const uint8_t* cq, int r, int kb, int rloc, const uint8_t* aq,
                                            const float* ad, int rsb, int blk0, uint64_t (&v)[Cfg<MT>::NTL][2]) {
  constexpr int NTL = Cfg<MT>::NTL;
  const uint8_t* sc = cq + kb * r * 32;
  uint64_t q[2][NTL][2];
#pragma unroll
  for (int h4 = 0; h4 < 2; ++h4) {
    uint64_t p2[2][NTL][2];
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      uint64_t ta[NTL][2], tb[NTL][2];
      const int j = 4 * h4 + 2 * h2;
      block_terms<MT>(cq, sc, r, rloc, j, aq, ad, rsb, blk0 + j, ta);
      block_terms<MT>(cq, sc, r, rloc, j + 1, aq, ad, rsb, blk0 + j + 1, tb);
#pragma unroll
      for (int nt = 0; nt < NTL; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          ta[nt][e] = (j < kb) ? ta[nt][e] : 0ull;  // +0.0f in both halves
          tb[nt][e] = (j + 1 < kb) ? tb[nt][e] : 0ull;
          p2[h2][nt][e] = f2_add(ta[nt][e], tb[nt][e]);
        }
    }
#pragma unroll
    for (int nt = 0; nt < NTL; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) q[h4][nt][e] = f2_add(p2[0][nt][e], p2[1][nt][e]);
  }
#pragma unroll
  for (int nt = 0; nt < NTL; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) v[nt][e] = f2_add(q[0][nt][e], q[1][nt][e]);
}

template <int MT, bool FUSED>
__global__ void __launch_bounds__(THREADS, 1) gemv_vt_kernel(const Args a) {
  constexpr int NTL = Cfg<MT>::NTL;
  constexpr int LV = Cfg<MT>::LV;
  constexpr int BAR_CONSUMERS = 1;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* stage_buf = smem;
  uint8_t* aq = smem + (size_t)STAGES * STAGE_BYTES;
  const int rsb = act_rsb(a.UB);
  float* ad = reinterpret_cast<float*>(aq + (size_t)Cfg<MT>::MP * rsb);
  uint8_t* raw = aq + act_bytes<MT>(a.UB);
  uint64_t* full = reinterpret_cast<uint64_t*>(raw + a.raw_bytes);
  uint64_t* empty = full + STAGES;
  uint64_t* abar = empty + STAGES;
  uint64_t* pready = abar + 1;  // cluster: the partials of every CTA of the cluster are in place
  uint64_t* pdone = abar + 2;   // cluster: every CTA of the cluster has read this CTA's partials
  volatile int* misc = reinterpret_cast<volatile int*>(abar + 3);
  // misc[0]: abort flag, misc[1]: "this CTA combines the tile", misc[2]: rounds issued
  // In a cluster, a unit's partials [M][VR] sit in the raw area: the CTA
  // stages its one K range before its first unit and never again.
  float* pbuf = reinterpret_cast<float*>(raw);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NCW);
    }
    mbar_init(abar, 1);
    if (a.cl > 1) {
      mbar_init(pready, a.cl);
      mbar_init(pdone, a.cl);
    }
    misc[0] = 0;
    misc[1] = 0;
    misc[2] = 0;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_dependents();
  // In a cluster every thread arrives on the cluster barrier now (the
  // mbarriers above are initialised) and waits before its first access to
  // another CTA: the consumers before their first remote arrival, the
  // producer lane inside produce(); lanes 1-31 of the producer warp wait and
  // exit.
  const bool clu = a.cl > 1;
  if (warp == NCW) {
    if (clu) {
      __syncwarp();
      cluster_arrive_aligned();
      if (lane != 0) {
        asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
        return;
      }
    }
    if (lane == 0) produce(a, stage_buf, full, empty, misc);
    return;
  }
  if (clu) cluster_arrive_aligned();
  bool cl_synced = !clu;
  int ncomb = 0;  // cluster combines done (phase parity of pready and pdone)
  const int crank = clu ? (int)blockIdx.x % a.cl : 0;
  RawRing rr{abar, 0u, 0, 0};

  const int g = lane >> 2, tig = lane & 3;
  const int row0v = 16 * warp;          // first row of this warp's slice in the virtual tile
  const int gsl = row0v / a.R;          // tile of the virtual tile
  const int rloc = row0v - gsl * a.R;   // first row inside that tile
  int stage = 0;
  uint32_t phase = 0;
  int consumed = 0;
  bool ok = true;
  bool waited = false;
  int staged_s = -1;

  const UnitRange ur = unit_range(a);
  for (int u = ur.first; u < ur.end; u += ur.step) {
    const int s = u / a.TV, tv = u - s * a.TV;
    const int c0 = s * a.RU;
    const int nr = min(a.RU, a.nch - c0);
    const int b0 = c0 * CHUNK_BLOCKS;
    const int nblk = min(a.UB, a.NB - b0);
    const int t = tv * a.G + gsl;
    const int r = t < a.T ? tile_rows(t, a.N, a.R) : 0;
    const bool live = rloc < r;  // warp-uniform

    if (!waited) {
      pdl_wait();
      waited = true;
    }
    // After an abort (misc[0]) every consumer still runs the same barrier
    // sequence to the end, skipping the work: no thread leaves early, so no
    // barrier waits for one that did.
    if (s != staged_s) {  // units with the same K range reuse the staged blocks
      stage_act<MT, FUSED>(a, aq, ad, rsb, raw, b0, nblk, rr, misc);
      staged_s = s;
    }
    if constexpr (FUSED) {
      if (a.A_out != nullptr && tv == 0) write_act_out<MT>(a, aq, ad, rsb, b0, nblk);
    }

    uint64_t slot[LV][NTL][2];
#pragma unroll
    for (int l = 0; l < LV; ++l)
#pragma unroll
      for (int nt = 0; nt < NTL; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) slot[l][nt][e] = 0ull;

    for (int rho = 0; rho < nr; ++rho) {
      // once aborted, no more waits; a stage is released only when its round
      // was received, so after a failure no stage with a copy in flight is
      // reused and the drain below can wait for each of them
      bool got = false;
      if (misc[0] == 0) {
        got = mbar_wait_bounded(&full[stage], phase, a.wait_ns);
        if (!got) {
          atomicOr(a.err, ERR_CONSUMER_WAIT);
          misc[0] = 1;
        }
      }
      if (!got) ok = false;
      uint64_t v[NTL][2];
#pragma unroll
      for (int nt = 0; nt < NTL; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) v[nt][e] = 0ull;
      if (got && live) {
        const uint8_t* cq = stage_buf + (size_t)stage * STAGE_BYTES + (size_t)gsl * a.R * SLOT_UNIT;
        chunk_value<MT>(cq, r, chunk_blocks(c0 + rho, a.NB), rloc, aq, ad, rsb, rho * CHUNK_BLOCKS, v);
      }
      __syncwarp();
      if (got) {
        if (lane == 0) mbar_arrive(&empty[stage]);
        ++consumed;
      }
      if (++stage == STAGES) {
        stage = 0;
        phase ^= 1u;
      }
      // binary counter over the round subtrees
      bool placed = false;
#pragma unroll
      for (int l = 0; l < LV; ++l) {
        if (!placed) {
          if ((rho >> l) & 1) {
#pragma unroll
            for (int nt = 0; nt < NTL; ++nt)
#pragma unroll
              for (int e = 0; e < 2; ++e) v[nt][e] = f2_add(slot[l][nt][e], v[nt][e]);
          } else {
#pragma unroll
            for (int nt = 0; nt < NTL; ++nt)
#pragma unroll
              for (int e = 0; e < 2; ++e) slot[l][nt][e] = v[nt][e];
            placed = true;
          }
        }
      }
    }
    // what is left merges from the lowest level up (= zero padding)
    uint64_t pv2[NTL][2];
    bool have = false;
#pragma unroll
    for (int nt = 0; nt < NTL; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) pv2[nt][e] = 0ull;
#pragma unroll
    for (int l = 0; l < LV; ++l) {
      if ((nr >> l) & 1) {
#pragma unroll
        for (int nt = 0; nt < NTL; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) pv2[nt][e] = have ? f2_add(slot[l][nt][e], pv2[nt][e]) : slot[l][nt][e];
        have = true;
      }
    }
    // pv[nt][e]: rows rloc + g + (e >> 1) * 8, activation row 8nt + 2tig + (e & 1)
    float pv[NTL][4];
#pragma unroll
    for (int nt = 0; nt < NTL; ++nt) {
      f2_unpack(pv2[nt][0], pv[nt][0], pv[nt][1]);
      f2_unpack(pv2[nt][1], pv[nt][2], pv[nt][3]);
    }

    const int64_t n0 = (int64_t)t * a.R + rloc;  // output row of this slice's row 0
    if (a.S == 1) {
      if (ok && live && misc[0] == 0) {
#pragma unroll
        for (int nt = 0; nt < NTL; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int m = 8 * nt + 2 * tig + (e & 1);
            const int row = g + (e >> 1) * 8;
            if (m < a.M && rloc + row < r) a.y[(int64_t)m * a.N + n0 + row] = pv[nt][e];
          }
      }
      continue;
    }

    if (clu) {
      // split along K inside the cluster: every CTA puts its unit value into
      // its own shared memory, and CTA rank k combines the k-th share of the
      // tile's outputs from the partials of all ranks (distributed shared
      // memory), in split order as below
      // (one thread waits on each mbarrier and a CTA barrier passes the
      // phase on; the arrivals on the cl CTAs are issued by cl lanes at once)
      if (ncomb > 0) {  // the previous unit's partials are read by every CTA
        if (threadIdx.x == 0 && misc[0] == 0 &&
            !mbar_wait_bounded<true>(pdone, (uint32_t)((ncomb - 1) & 1), a.wait_ns)) {
          atomicOr(a.err, ERR_CONSUMER_WAIT);
          misc[0] = 1;
        }
        named_bar_sync(BAR_CONSUMERS, NT);
      }
      if (!cl_synced) {  // every CTA's mbarriers are initialised
        cluster_wait_aligned();
        cl_synced = true;
      }
      if (ok && live && misc[0] == 0) {
#pragma unroll
        for (int nt = 0; nt < NTL; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int m = 8 * nt + 2 * tig + (e & 1);
            const int row = g + (e >> 1) * 8;
            if (m < a.M) pbuf[m * VR + row0v + row] = pv[nt][e];
          }
      }
      named_bar_sync(BAR_CONSUMERS, NT);
      if ((int)threadIdx.x < a.cl) mbar_arrive_remote(mapa_shared(smem_u32(pready), threadIdx.x));
      if (threadIdx.x == 0 && misc[0] == 0 && !mbar_wait_bounded<true>(pready, (uint32_t)(ncomb & 1), a.wait_ns)) {
        atomicOr(a.err, ERR_CONSUMER_WAIT);
        misc[0] = 1;
      }
      named_bar_sync(BAR_CONSUMERS, NT);  // every partial of the cluster is visible
      {
        const int64_t nbase = (int64_t)tv * VR;
        const int nrows = (int)min((int64_t)VR, a.N - nbase);
        const int quads = a.M * (VR / 4);
        const int share = (quads + a.cl - 1) / a.cl;
        const int qa = crank * share, qb = min(quads, qa + share);
        const uint32_t pb0 = smem_u32(pbuf);
        for (int qd = qa + (int)threadIdx.x; qd < qb; qd += NT) {
          const int m = qd / (VR / 4), n4 = (qd - m * (VR / 4)) * 4;
          const uint32_t off = pb0 + (uint32_t)(m * VR + n4) * 4u;
          float4 pk[8];
#pragma unroll
          for (int k = 0; k < 8; ++k)
            pk[k] = k < a.cl ? ld_cluster_f4(mapa_shared(off, (uint32_t)k)) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
          float sl[SPLIT_LV][4];
#pragma unroll
          for (int l = 0; l < SPLIT_LV; ++l)
#pragma unroll
            for (int e = 0; e < 4; ++e) sl[l][e] = 0.0f;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            if (k < a.cl) {
              float vv[4] = {pk[k].x, pk[k].y, pk[k].z, pk[k].w};
              bool placed = false;
#pragma unroll
              for (int l = 0; l < SPLIT_LV; ++l) {
                if (!placed) {
                  if ((k >> l) & 1) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) vv[e] = tadd(sl[l][e], vv[e]);
                  } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) sl[l][e] = vv[e];
                    placed = true;
                  }
                }
              }
            }
          }
          float out[4] = {0.0f, 0.0f, 0.0f, 0.0f};
          bool h = false;
#pragma unroll
          for (int l = 0; l < SPLIT_LV; ++l) {
            if ((a.cl >> l) & 1) {
#pragma unroll
              for (int e = 0; e < 4; ++e) out[e] = h ? tadd(sl[l][e], out[e]) : sl[l][e];
              h = true;
            }
          }
          if (misc[0] == 0) {
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (n4 + e < nrows) a.y[(int64_t)m * a.N + nbase + n4 + e] = out[e];
          }
        }
      }
      named_bar_sync(BAR_CONSUMERS, NT);  // this CTA's reads of the partials are done
      if ((int)threadIdx.x < a.cl) mbar_arrive_remote(mapa_shared(smem_u32(pdone), threadIdx.x));
      ++ncomb;
      continue;
    }

    // split along K: publish the unit value, take a ticket, the last one combines
    if (ok && live && misc[0] == 0) {
#pragma unroll
      for (int nt = 0; nt < NTL; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int m = 8 * nt + 2 * tig + (e & 1);
          const int row = g + (e >> 1) * 8;
          if (m < a.M && rloc + row < r) a.ws_part[((int64_t)s * a.M + m) * a.Np + n0 + row] = pv[nt][e];
        }
    }
    // the barrier orders every consumer's partial stores before thread 0's
    // fence and ticket (the pattern of a grid-wide barrier)
    named_bar_sync(BAR_CONSUMERS, NT);
    if (threadIdx.x == 0) {
      const bool any_abort = misc[0] != 0;
      __threadfence();
      const unsigned prev = any_abort ? 0u : atomicAdd(&a.ws_cnt[tv], 1u);
      misc[1] = (!any_abort && prev == (unsigned)(a.S - 1)) ? 1 : 0;
    }
    named_bar_sync(BAR_CONSUMERS, NT);
    if (misc[1]) {
      __threadfence();
      // this virtual tile's outputs, 4 consecutive rows (a quad) per thread;
      // CQ quads per pass with all their partial loads in flight, merged
      // with a binary counter over the split index
      constexpr int CQ = 2;
      const int64_t nbase = (int64_t)tv * VR;
      const int nrows = (int)min((int64_t)VR, a.N - nbase);
      const int quads = a.M * (VR / 4);
      const int64_t sstride = (int64_t)a.M * a.Np;
      for (int q0 = threadIdx.x; q0 < quads; q0 += NT * CQ) {  // the same trip count in every thread
        float sl[CQ][SPLIT_LV][4];
#pragma unroll
        for (int c = 0; c < CQ; ++c)
#pragma unroll
          for (int l = 0; l < SPLIT_LV; ++l)
#pragma unroll
            for (int k = 0; k < 4; ++k) sl[c][l][k] = 0.0f;
        const float* part[CQ];
        bool on[CQ];
#pragma unroll
        for (int c = 0; c < CQ; ++c) {
          const int qd = q0 + c * NT;
          const int m = qd / (VR / 4), n4 = (qd - m * (VR / 4)) * 4;
          on[c] = qd < quads && n4 < nrows;
          part[c] = a.ws_part + (int64_t)m * a.Np + nbase + n4;
        }
        for (int s0 = 0; s0 < a.S; s0 += 8) {
          float4 pv8[CQ][8];
#pragma unroll
          for (int c = 0; c < CQ; ++c)
#pragma unroll
            for (int k = 0; k < 8; ++k)
              pv8[c][k] = (on[c] && s0 + k < a.S)
                              ? __ldcg(reinterpret_cast<const float4*>(part[c] + (int64_t)(s0 + k) * sstride))
                              : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
          for (int c = 0; c < CQ; ++c)
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const int ss = s0 + k;
              if (ss < a.S) {
                float vv[4] = {pv8[c][k].x, pv8[c][k].y, pv8[c][k].z, pv8[c][k].w};
                bool placed = false;
#pragma unroll
                for (int l = 0; l < SPLIT_LV; ++l) {
                  if (!placed) {
                    if ((ss >> l) & 1) {
#pragma unroll
                      for (int e = 0; e < 4; ++e) vv[e] = tadd(sl[c][l][e], vv[e]);
                    } else {
#pragma unroll
                      for (int e = 0; e < 4; ++e) sl[c][l][e] = vv[e];
                      placed = true;
                    }
                  }
                }
              }
            }
        }
#pragma unroll
        for (int c = 0; c < CQ; ++c) {
          if (!on[c]) continue;
          const int qd = q0 + c * NT;
          const int m = qd / (VR / 4), n4 = (qd - m * (VR / 4)) * 4;
          float out[4] = {0.0f, 0.0f, 0.0f, 0.0f};
          bool h = false;
#pragma unroll
          for (int l = 0; l < SPLIT_LV; ++l) {
            if ((a.S >> l) & 1) {
#pragma unroll
              for (int e = 0; e < 4; ++e) out[e] = h ? tadd(sl[c][l][e], out[e]) : sl[c][l][e];
              h = true;
            }
          }
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (n4 + e < nrows) a.y[(int64_t)m * a.N + nbase + n4 + e] = out[e];
        }
      }
      if (threadIdx.x == 0) a.ws_cnt[tv] = 0u;
    }
  }

  if (clu) {
    if (!cl_synced) cluster_wait_aligned();
    // no other CTA of the cluster reads this one's shared memory any more
    // (the full bound, whatever the other waits had)
    if (threadIdx.x == 0 && ncomb > 0 &&
        !mbar_wait_bounded<true>(pdone, (uint32_t)((ncomb - 1) & 1), WAIT_LIMIT_NS))
      atomicOr(a.err, ERR_DRAIN_WAIT);
  }
  // After a failed wait: let copies that were issued but not received by
  // warp 0 land before the CTA's shared memory goes away.  Those stages were
  // never released, so each has at most one copy in flight; the drain keeps
  // the full bound whatever limit the other waits had.
  if (threadIdx.x == 0 && misc[0]) {
    if (rr.issued > rr.waited)  // the last piece's copies (at most one piece in flight)
      if (!mbar_wait_bounded(abar, (uint32_t)(rr.waited & 1), WAIT_LIMIT_NS)) atomicOr(a.err, ERR_DRAIN_WAIT);
    for (int k = consumed; k < misc[2]; ++k) {
      if (!mbar_wait_bounded(&full[k % STAGES], (uint32_t)((k / STAGES) & 1), WAIT_LIMIT_NS)) {
        atomicOr(a.err, ERR_DRAIN_WAIT);
        break;
      }
    }
  }
}

// ---- host side ---------------------------------------------------------------
template <int MT>
cudaError_t launch_m(const Args& a, bool fused, int grid, bool pdl, cudaStream_t s);
template <int MT>
cudaError_t attributes_m(bool fused);
template <int MT>
int max_clusters_m(bool fused, int cl);

template <int MT, bool FUSED>
cudaError_t set_attributes() {
  cudaError_t e = cudaFuncSetAttribute(gemv_vt_kernel<MT, FUSED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem_bytes());
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(gemv_vt_kernel<MT, FUSED>, cudaFuncAttributePreferredSharedMemoryCarveout,
                              (int)cudaSharedmemCarveoutMaxShared);
}

template <int MT, bool FUSED>
cudaError_t launch_t(const Args& args, int grid, bool pdl, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = smem_bytes();
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (args.cl > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = args.cl;
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
  return cudaLaunchKernelEx(&cfg, gemv_vt_kernel<MT, FUSED>, args);
}

// Clusters of `cl` CTAs of this kernel that can be resident at once (0 when
// none can).
template <int MT, bool FUSED>
int max_clusters_t(int cl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cl);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = smem_bytes();
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, gemv_vt_kernel<MT, FUSED>, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return n;
}

// Per-row-count translation units instantiate the launch and the attribute
// setting for both the fused and the unfused kernel.
#define Q8_VT_INSTANTIATE(MT)                                                                           \
  template <>                                                                                           \
  cudaError_t launch_m<MT>(const Args& a, bool fused, int grid, bool pdl, cudaStream_t s) {             \
    return fused ? launch_t<MT, true>(a, grid, pdl, s) : launch_t<MT, false>(a, grid, pdl, s);          \
  }                                                                                                     \
  template <>                                                                                           \
  cudaError_t attributes_m<MT>(bool fused) {                                                            \
    return fused ? set_attributes<MT, true>() : set_attributes<MT, false>();                            \
  }                                                                                                     \
  template <>                                                                                           \
  int max_clusters_m<MT>(bool fused, int cl) {                                                          \
    return fused ? max_clusters_t<MT, true>(cl) : max_clusters_t<MT, false>(cl);                        \
  }

}  // namespace vt
}  // namespace q8
