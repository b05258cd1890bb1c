// q8_gemv.cu -- the Q8_0 decode GEMV (int8 dot products on the DP4A path).
//
// One persistent CTA per SM slot walks a list of work units.  A unit is one
// 128-row tile of W times C consecutive blocks along K (C = 8 * 2^k, aligned
// to C).  Warp 4 of the CTA is the producer: one lane streams the unit's
// 34,816-byte chunks (128 rows x 8 blocks, contiguous in the packed layout)
// into a ring of shared-memory stages with cp.async.bulk, completing on
// mbarriers.  Warps 0-3 are the consumers: thread i owns row i of the tile,
// reads its quants and scale from shared memory, and for each activation row
// computes the exact int32 block dot with __dp4a, the canonical term
// t_b = float(isum) * (d_w * d_a) and the fixed pairwise tree over b.
//
// Reduction order.  The canonical sum over blocks b is the pairwise tree over
// b padded with zeros to a power of two.  A chunk (8 aligned blocks) is a
// subtree; chunk values are merged with a binary counter (merge with the left
// sibling while the index bit is 1), and what is left at the end is merged
// from the lowest level up, which is what zero padding gives.  A unit (C
// aligned blocks) is again a subtree, and the K-split combine merges unit
// values the same way.  The result is therefore independent of C, of the
// number of splits, of M and of the row's position in the batch.
//
// Split-K.  When a tile is split into S > 1 units, each unit writes its
// partial row values to the workspace, then takes a ticket on the tile's
// counter; the CTA holding the last ticket merges the S partials in index
// order, writes y and resets the counter to zero.  No CTA waits for another.
//
// Programmatic dependent launch.  The producer never waits for the previous
// grid: W is immutable, so streaming starts at once.  The consumers execute
// griddepcontrol.wait before reading activations or writing anything.
#include <cuda_runtime.h>

#include "q8_device.cuh"
#include "q8_internal.h"

namespace q8 {
namespace {

constexpr int NCW = 4;                      // consumer warps: 128 threads = 128 rows
constexpr int GEMV_THREADS = (NCW + 1) * 32;
constexpr int STAGES = 3;
constexpr int ACT_SMEM_BUDGET = 36864;      // bytes for one unit's activation blocks
constexpr int MAX_SPLITS = 128;
constexpr int SPLIT_LEVELS = 8;             // binary counter levels for S <= 128
// Workspace layout: a fixed prefix of tile tickets, then the partials.  The
// prefix has the same size for every call, so partials written by one call
// never land on the tickets of another call that shares the workspace.
constexpr int MAX_SPLIT_TILES = 4096;       // split along K only when T <= 4096
constexpr size_t TICKET_BYTES = (size_t)MAX_SPLIT_TILES * 4;

template <int MT>
struct MtCfg {
  // largest blocks-per-unit (8 * 2^k) whose activations (36 B per block per
  // row in shared memory) fit the budget, capped at 256
  static constexpr int raw = ACT_SMEM_BUDGET / (MT * 36);
  static constexpr int C_MAX = raw >= 256 ? 256 : raw >= 128 ? 128 : raw >= 64 ? 64 : raw >= 32 ? 32 : raw >= 16 ? 16 : 8;
  static constexpr int LV = C_MAX == 256 ? 6 : C_MAX == 128 ? 5 : C_MAX == 64 ? 4 : C_MAX == 32 ? 3 : C_MAX == 16 ? 2 : 1;
};

__device__ unsigned int g_gemv_error;  // 0 = fine; bit flags of failed waits

enum : unsigned { ERR_PRODUCER_WAIT = 1u, ERR_CONSUMER_WAIT = 2u, ERR_DRAIN_WAIT = 4u };

struct GemvArgs {
  const uint8_t* W;
  const uint8_t* A;     // activation blocks [M][NB] (unfused)
  const float* x;       // fp32 activations [M][K] (fused)
  uint8_t* A_out;       // fused: optional activation blocks out
  float* y;             // [M][N]
  float* ws_part;       // [S][M][N] partials (S > 1)
  unsigned* ws_cnt;     // [T] tickets (S > 1)
  int64_t N;
  int NB, T, M, C, S, units;
};

template <int MT>
constexpr size_t gemv_smem_bytes() {
  return (size_t)STAGES * CHUNK_FULL_BYTES + (size_t)MT * MtCfg<MT>::C_MAX * 36 +
         2 * STAGES * sizeof(uint64_t) + 4 * sizeof(int);
}

// ---- producer: one lane streams every chunk of every unit of this CTA ----
__device__ __forceinline__ void produce(const GemvArgs& a, uint8_t* stage_buf, uint64_t* full,
                                        uint64_t* empty, volatile int* misc) {
  const uint64_t pol = l2_policy_evict_first();
  int stage = 0;
  uint32_t phase = 0;
  int issued = 0;
  for (int u = blockIdx.x; u < a.units; u += gridDim.x) {
    const int t = u / a.S, s = u % a.S;
    const int r = tile_rows(t, a.N);
    const int kb0 = s * a.C;
    const int kb1 = min(kb0 + a.C, a.NB);
    for (int cb = kb0; cb < kb1; cb += CHUNK_BLOCKS) {
      const int kb = min(CHUNK_BLOCKS, kb1 - cb);
      if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, WAIT_LIMIT_NS)) {
        atomicOr(&g_gemv_error, ERR_PRODUCER_WAIT);
        misc[0] = 1;
        return;
      }
      if (misc[0]) return;
      const uint8_t* src = a.W + chunk_offset(t, cb / CHUNK_BLOCKS, r, a.NB);
      uint8_t* dst = stage_buf + (size_t)stage * CHUNK_FULL_BYTES;
      const uint32_t bytes = (uint32_t)(kb * r * BLOCK_BYTES);
      const uint32_t bulk = bytes & ~15u;
      for (uint32_t k = bulk; k < bytes; ++k) dst[k] = src[k];  // ragged tail < 16 B
      mbar_arrive_expect_tx(&full[stage], bulk);
      bulk_g2s(dst, src, bulk, &full[stage], pol);
      misc[2] = ++issued;
      if (++stage == STAGES) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
}

// ---- activation staging for one unit: blocks [kb0, kb0 + nblk) of rows < M ----
template <int MT, bool FUSED>
__device__ __forceinline__ void stage_activations(const GemvArgs& a, int t, int kb0, int nblk,
                                                  uint8_t* act_q, float* act_d) {
  constexpr int C_MAX = MtCfg<MT>::C_MAX;
  if constexpr (!FUSED) {
    const int total = a.M * nblk;
    for (int idx = threadIdx.x; idx < total; idx += NCW * 32) {
      const int m = idx / nblk, blk = idx - m * nblk;
      const uint8_t* src = a.A + ((int64_t)m * a.NB + kb0 + blk) * BLOCK_BYTES;
      uint4 q0, q1;
      load_block_quants_u16(src, q0, q1);
      const uint16_t d16 = load_block_scale_bits(src);
      uint8_t* dst = act_q + (m * C_MAX + blk) * 32;
      *reinterpret_cast<uint4*>(dst) = q0;
      *reinterpret_cast<uint4*>(dst + 16) = q1;
      act_d[m * C_MAX + blk] = __half2float(__ushort_as_half(d16));
    }
  } else {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int total = a.M * nblk;
    const int64_t K = (int64_t)a.NB * QK;
    for (int idx = warp; idx < total; idx += NCW) {
      const int m = idx / nblk, blk = idx - m * nblk;
      const float v = __ldcg(a.x + (int64_t)m * K + (int64_t)(kb0 + blk) * QK + lane);
      const LaneQuant lq = quantize_lane(v);
      act_q[(m * C_MAX + blk) * 32 + lane] = (uint8_t)(lq.q & 0xff);
      if (lane == 0) act_d[m * C_MAX + blk] = lq.d_stored;
      if (a.A_out != nullptr && t == 0) {
        uint8_t* ob = a.A_out + ((int64_t)m * a.NB + kb0 + blk) * BLOCK_BYTES;
        ob[2 + lane] = (uint8_t)(lq.q & 0xff);
        if (lane < 2) ob[lane] = (uint8_t)(lane == 0 ? (lq.d16 & 0xff) : (lq.d16 >> 8));
      }
    }
  }
}

// ---- one chunk (kb <= 8 blocks) of row i: the 8-leaf pairwise tree per m ----
template <int MT>
__device__ __forceinline__ void chunk_value(const uint8_t* cq, int r, int kb, int i,
                                            const uint8_t* aq, const float* ad, int M,
                                            float (&v)[MT]) {
  constexpr int C_MAX = MtCfg<MT>::C_MAX;
  const uint8_t* sc = cq + kb * r * 32;
  float l0[MT], l1[MT], l2[MT];
#pragma unroll
  for (int j = 0; j < CHUNK_BLOCKS; ++j) {
    float tj[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) tj[m] = 0.0f;
    if (j < kb) {
      const uint4 w0 = lds128(cq + ((2 * j) * r + i) * 16);
      const uint4 w1 = lds128(cq + ((2 * j + 1) * r + i) * 16);
      const float dw =
          __half2float(__ushort_as_half(*reinterpret_cast<const unsigned short*>(sc + (j * r + i) * 2)));
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        if (m < M) {
          const uint8_t* am = aq + (m * C_MAX + j) * 32;
          tj[m] = block_term(dot_block(w0, w1, lds128(am), lds128(am + 16)), dw, ad[m * C_MAX + j]);
        }
      }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      if ((j & 1) == 0) {
        l0[m] = tj[m];
      } else {
        const float p = tadd(l0[m], tj[m]);        // 2 leaves
        if ((j & 2) == 0) {
          l1[m] = p;
        } else {
          const float q = tadd(l1[m], p);          // 4 leaves
          if ((j & 4) == 0) l2[m] = q;
          else v[m] = tadd(l2[m], q);              // 8 leaves
        }
      }
    }
  }
}

template <int MT, bool FUSED>
__global__ void __launch_bounds__(GEMV_THREADS, 1) gemv_kernel(const GemvArgs a) {
  constexpr int C_MAX = MtCfg<MT>::C_MAX;
  constexpr int LV = MtCfg<MT>::LV;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* stage_buf = smem;
  uint8_t* act_q = smem + (size_t)STAGES * CHUNK_FULL_BYTES;
  float* act_d = reinterpret_cast<float*>(act_q + MT * C_MAX * 32);
  uint64_t* full = reinterpret_cast<uint64_t*>(act_d + MT * C_MAX);
  uint64_t* empty = full + STAGES;
  volatile int* misc = reinterpret_cast<volatile int*>(empty + STAGES);
  // misc[0]: abort flag, misc[1]: "this CTA combines the tile", misc[2]: chunks issued

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NCW);
    }
    misc[0] = 0;
    misc[1] = 0;
    misc[2] = 0;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  if (warp == NCW) {
    if (lane == 0) produce(a, stage_buf, full, empty, misc);
    return;
  }

  const int i = threadIdx.x;  // row inside the tile
  int stage = 0;
  uint32_t phase = 0;
  int consumed = 0;
  bool ok = true;
  bool waited = false;

  for (int u = blockIdx.x; u < a.units; u += gridDim.x) {
    const int t = u / a.S, s = u % a.S;
    const int r = tile_rows(t, a.N);
    const int kb0 = s * a.C;
    const int nblk = min(a.C, a.NB - kb0);
    const int nchunks = (nblk + CHUNK_BLOCKS - 1) / CHUNK_BLOCKS;
    const int64_t n = (int64_t)t * TILE_ROWS + i;

    if (!waited) {
      pdl_wait();
      waited = true;
    }
    named_bar_sync(1, NCW * 32);  // every consumer is done with the previous unit
    stage_activations<MT, FUSED>(a, t, kb0, nblk, act_q, act_d);
    named_bar_sync(1, NCW * 32);

    float slot[MT][LV];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int l = 0; l < LV; ++l) slot[m][l] = 0.0f;

    for (int ci = 0; ci < nchunks; ++ci) {
      if (ok && misc[0]) ok = false;
      if (!ok) break;
      if (!mbar_wait_bounded(&full[stage], phase, WAIT_LIMIT_NS)) {
        atomicOr(&g_gemv_error, ERR_CONSUMER_WAIT);
        misc[0] = 1;
        ok = false;
        break;
      }
      const int kb = min(CHUNK_BLOCKS, nblk - ci * CHUNK_BLOCKS);
      float v[MT];
      chunk_value<MT>(stage_buf + (size_t)stage * CHUNK_FULL_BYTES, r, kb, i,
                      act_q + ci * CHUNK_BLOCKS * 32, act_d + ci * CHUNK_BLOCKS, a.M, v);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
      ++consumed;
      if (++stage == STAGES) {
        stage = 0;
        phase ^= 1u;
      }
      // binary counter over chunk subtrees
      bool placed = false;
#pragma unroll
      for (int l = 0; l < LV; ++l) {
        if (!placed) {
          if ((ci >> l) & 1) {
#pragma unroll
            for (int m = 0; m < MT; ++m) v[m] = tadd(slot[m][l], v[m]);
          } else {
#pragma unroll
            for (int m = 0; m < MT; ++m) slot[m][l] = v[m];
            placed = true;
          }
        }
      }
    }

    // what is left merges from the lowest level up (= zero padding)
    float res[MT];
    bool have = false;
#pragma unroll
    for (int m = 0; m < MT; ++m) res[m] = 0.0f;
#pragma unroll
    for (int l = 0; l < LV; ++l) {
      if ((nchunks >> l) & 1) {
#pragma unroll
        for (int m = 0; m < MT; ++m) res[m] = have ? tadd(slot[m][l], res[m]) : slot[m][l];
        have = true;
      }
    }

    if (a.S == 1) {
      if (ok && i < r) {
#pragma unroll
        for (int m = 0; m < MT; ++m)
          if (m < a.M) a.y[(int64_t)m * a.N + n] = res[m];
      }
      continue;
    }

    // split along K: publish the partial, take a ticket, last one combines
    if (ok && i < r) {
#pragma unroll
      for (int m = 0; m < MT; ++m)
        if (m < a.M) a.ws_part[((int64_t)s * a.M + m) * a.N + n] = res[m];
    }
    __threadfence();
    named_bar_sync(1, NCW * 32);
    if (threadIdx.x == 0) {
      const bool any_abort = misc[0] != 0;
      const unsigned prev = any_abort ? 0u : atomicAdd(&a.ws_cnt[t], 1u);
      misc[1] = (!any_abort && prev == (unsigned)(a.S - 1)) ? 1 : 0;
    }
    named_bar_sync(1, NCW * 32);
    if (misc[1]) {
      __threadfence();
      if (i < r) {
        for (int m = 0; m < a.M; ++m) {
          float sl[SPLIT_LEVELS];
#pragma unroll
          for (int l = 0; l < SPLIT_LEVELS; ++l) sl[l] = 0.0f;
          for (int ss = 0; ss < a.S; ++ss) {
            float v = __ldcg(&a.ws_part[((int64_t)ss * a.M + m) * a.N + n]);
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

  // After a failed wait: let copies that were issued but not consumed land
  // before the CTA's shared memory goes away (bounded as well).
  if (threadIdx.x == 0 && misc[0]) {
    for (int k = consumed; k < misc[2]; ++k) {
      if (!mbar_wait_bounded(&full[k % STAGES], (uint32_t)((k / STAGES) & 1), WAIT_LIMIT_NS / 4)) {
        atomicOr(&g_gemv_error, ERR_DRAIN_WAIT);
        break;
      }
    }
  }
}

template <int MT, bool FUSED>
cudaError_t prepare_kernel() {
  static bool done = false;  // per device handled by callers setting the attribute each time
  (void)done;
  return cudaFuncSetAttribute(gemv_kernel<MT, FUSED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)gemv_smem_bytes<MT>());
}

template <int MT, bool FUSED>
int occupancy_of() {
  if (prepare_kernel<MT, FUSED>() != cudaSuccess) return 0;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, gemv_kernel<MT, FUSED>, GEMV_THREADS,
                                                    gemv_smem_bytes<MT>()) != cudaSuccess)
    return 0;
  return occ;
}

int occupancy(int MT, bool fused) {
  switch (MT) {
    case 1: return fused ? occupancy_of<1, true>() : occupancy_of<1, false>();
    case 2: return fused ? occupancy_of<2, true>() : occupancy_of<2, false>();
    case 4: return fused ? occupancy_of<4, true>() : occupancy_of<4, false>();
    case 8: return fused ? occupancy_of<8, true>() : occupancy_of<8, false>();
    default: return fused ? occupancy_of<16, true>() : occupancy_of<16, false>();
  }
}

int c_max_of(int MT) {
  switch (MT) {
    case 1: return MtCfg<1>::C_MAX;
    case 2: return MtCfg<2>::C_MAX;
    case 4: return MtCfg<4>::C_MAX;
    case 8: return MtCfg<8>::C_MAX;
    default: return MtCfg<16>::C_MAX;
  }
}

size_t smem_of(int MT) {
  switch (MT) {
    case 1: return gemv_smem_bytes<1>();
    case 2: return gemv_smem_bytes<2>();
    case 4: return gemv_smem_bytes<4>();
    case 8: return gemv_smem_bytes<8>();
    default: return gemv_smem_bytes<16>();
  }
}

template <int MT, bool FUSED>
cudaError_t launch_one(const GemvPlan& p, const GemvArgs& args, bool pdl, cudaStream_t s) {
  cudaError_t e = prepare_kernel<MT, FUSED>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(GEMV_THREADS);
  cfg.dynamicSmemBytes = gemv_smem_bytes<MT>();
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, gemv_kernel<MT, FUSED>, args);
}

}  // namespace

bool plan_gemv(const DeviceInfo& dev, int64_t N, int64_t K, int M, bool fused, GemvPlan* p) {
  GemvPlan q;
  q.N = N;
  q.K = K;
  q.NB = K / QK;
  q.M = M;
  const int Mp = M > 16 ? 16 : M;  // rows per launch
  q.MT = Mp <= 1 ? 1 : Mp <= 2 ? 2 : Mp <= 4 ? 4 : Mp <= 8 ? 8 : 16;
  const int64_t T = (N + TILE_ROWS - 1) / TILE_ROWS;
  if (T > (int64_t)1 << 30) return false;
  q.T = (int)T;
  const int cmax = c_max_of(q.MT);
  int occ = occupancy(q.MT, fused);
  if (occ < 1) occ = 1;
  const int64_t target = (int64_t)dev.sm_count * occ;
  int chosen = 0, smallest_valid = 0;
  for (int c = cmax; c >= CHUNK_BLOCKS; c >>= 1) {
    const int64_t S = (q.NB + c - 1) / c;
    if (S > MAX_SPLITS) break;
    smallest_valid = c;
    if (chosen == 0 && T * S >= target) chosen = c;
  }
  if (smallest_valid == 0) return false;  // K too large for the split limit
  if (chosen == 0) chosen = smallest_valid;
  // no unit needs more blocks than K has
  while (chosen > CHUNK_BLOCKS && chosen / 2 >= q.NB) chosen >>= 1;
  q.C = chosen;
  q.S = (int)((q.NB + q.C - 1) / q.C);
  if (q.S > 1 && T > MAX_SPLIT_TILES) {
    // prefer no split for very tall matrices; impossible only when one
    // unit's activations cannot fit shared memory
    if ((q.NB + cmax - 1) / cmax > 1) return false;
    q.C = cmax;
    while (q.C > CHUNK_BLOCKS && q.C / 2 >= q.NB) q.C >>= 1;
    q.S = 1;
  }
  const int64_t units = T * q.S;
  if (units > ((int64_t)1 << 31) - 1) return false;
  q.units = (int)units;
  q.grid = (int)(units < target ? units : target);
  q.smem = smem_of(q.MT);
  q.ws_bytes = q.S > 1 ? TICKET_BYTES + (size_t)q.S * Mp * N * 4 : 0;
  *p = q;
  return true;
}

cudaError_t launch_gemv(const GemvPlan& p, const uint8_t* W, const uint8_t* A, const float* x,
                        uint8_t* A_out, float* y, void* workspace, bool pdl, cudaStream_t s) {
  const bool fused = (x != nullptr);
  const size_t cnt_bytes = TICKET_BYTES;
  for (int m0 = 0; m0 < p.M; m0 += 16) {
    const int Mp = (p.M - m0) < 16 ? (p.M - m0) : 16;
    GemvArgs args;
    args.W = W;
    args.A = A ? A + (size_t)m0 * p.NB * BLOCK_BYTES : nullptr;
    args.x = x ? x + (size_t)m0 * p.K : nullptr;
    args.A_out = A_out ? A_out + (size_t)m0 * p.NB * BLOCK_BYTES : nullptr;
    args.y = y + (size_t)m0 * p.N;
    args.ws_cnt = p.S > 1 ? reinterpret_cast<unsigned*>(workspace) : nullptr;
    args.ws_part = p.S > 1 ? reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(workspace) + cnt_bytes)
                           : nullptr;
    args.N = p.N;
    args.NB = (int)p.NB;
    args.T = p.T;
    args.M = Mp;
    args.C = p.C;
    args.S = p.S;
    args.units = p.units;
    const int MT = Mp <= 1 ? 1 : Mp <= 2 ? 2 : Mp <= 4 ? 4 : Mp <= 8 ? 8 : 16;
    // a pass with fewer rows than the plan's MT reuses the plan's unit sizes
    // (C fits the larger MT, so it fits a smaller one too)
    GemvPlan pp = p;
    cudaError_t e;
    switch (MT) {
      case 1: e = fused ? launch_one<1, true>(pp, args, pdl, s) : launch_one<1, false>(pp, args, pdl, s); break;
      case 2: e = fused ? launch_one<2, true>(pp, args, pdl, s) : launch_one<2, false>(pp, args, pdl, s); break;
      case 4: e = fused ? launch_one<4, true>(pp, args, pdl, s) : launch_one<4, false>(pp, args, pdl, s); break;
      case 8: e = fused ? launch_one<8, true>(pp, args, pdl, s) : launch_one<8, false>(pp, args, pdl, s); break;
      default: e = fused ? launch_one<16, true>(pp, args, pdl, s) : launch_one<16, false>(pp, args, pdl, s); break;
    }
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t read_and_clear_gemv_error(unsigned* code) {
  unsigned v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_gemv_error, sizeof(v));
  if (e != cudaSuccess) return e;
  *code = v;
  const unsigned zero = 0;
  return cudaMemcpyToSymbol(g_gemv_error, &zero, sizeof(zero));
}

}  // namespace q8
