// q8_gemv.cu -- launch planning and dispatch for the GEMV kernels
// (the kernel itself is in q8_gemv_impl.cuh, instantiated per tile height
// in q8_gemv_r*.cu).
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "q8_gemv_impl.cuh"
#include "q8_internal.h"

namespace q8 {

template <int R>
cudaError_t launch_gemv_r(const GemvArgs& args, int MT, bool fused, int var, int grid, int cluster, bool pdl,
                         cudaStream_t s);
template <int R>
int occupancy_r(int MT, bool fused, int var);
template <int R>
bool cluster_fits_r(int MT, bool fused, int var, int cluster);

namespace {

__device__ unsigned int g_gemv_error;  // 0 = fine; bit flags of failed waits

constexpr int MAX_DEVICES = 64;
std::mutex g_mu;
unsigned* g_err_ptr[MAX_DEVICES] = {};

cudaError_t error_word(int dev, unsigned** out) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_err_ptr[dev] == nullptr) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_gemv_error);
    if (e != cudaSuccess) return e;
    g_err_ptr[dev] = static_cast<unsigned*>(p);
  }
  *out = g_err_ptr[dev];
  return cudaSuccess;
}

int occupancy(int R, int MT, bool fused, bool u5) {
  switch (R) {
    case 16: return occupancy_r<16>(MT, fused, u5 ? VAR_TCGEN05 : VAR_DEFAULT);
    case 32: return occupancy_r<32>(MT, fused, u5 ? VAR_TCGEN05 : VAR_DEFAULT);
    case 64: return occupancy_r<64>(MT, fused, u5 ? VAR_TCGEN05 : VAR_DEFAULT);
    default: return occupancy_r<128>(MT, fused, u5 ? VAR_TCGEN05 : VAR_DEFAULT);
  }
}

// cluster feasibility per (R, MT, fused, size), cached
std::mutex g_cl_mu;
signed char g_cl_cache[4][5][2][2][4];  // 0 unknown, 1 fits, -1 does not
bool cluster_fits(int R, int MT, bool fused, bool u5, int c) {
  const int ri = R == 16 ? 0 : R == 32 ? 1 : R == 64 ? 2 : 3;
  const int mi = MT == 1 ? 0 : MT == 2 ? 1 : MT == 4 ? 2 : MT == 8 ? 3 : 4;
  const int ci = c == 2 ? 0 : c == 4 ? 1 : c == 8 ? 2 : 3;
  std::lock_guard<std::mutex> lk(g_cl_mu);
  signed char& v = g_cl_cache[ri][mi][fused ? 1 : 0][u5 ? 1 : 0][ci];
  if (v == 0) {
    bool ok;
    switch (R) {
      case 16: ok = cluster_fits_r<16>(MT, fused, u5 ? VAR_TCGEN05 : VAR_DEFAULT, c); break;
      case 32: ok = cluster_fits_r<32>(MT, fused, u5 ? VAR_TCGEN05 : VAR_DEFAULT, c); break;
      case 64: ok = cluster_fits_r<64>(MT, fused, u5 ? VAR_TCGEN05 : VAR_DEFAULT, c); break;
      default: ok = cluster_fits_r<128>(MT, fused, u5 ? VAR_TCGEN05 : VAR_DEFAULT, c); break;
    }
    v = ok ? 1 : -1;
  }
  return v > 0;
}

int mt_of(int M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : M <= 8 ? 8 : 16; }
int stage_target_of(int MT) {
  switch (MT) {
    case 1: return MCfg<1>::STAGE_TARGET;
    case 2: return MCfg<2>::STAGE_TARGET;
    case 4: return MCfg<4>::STAGE_TARGET;
    case 8: return MCfg<8>::STAGE_TARGET;
    default: return MCfg<16>::STAGE_TARGET;
  }
}
int budget_of(int R, int MT, bool u5) {
  if (u5 && R == 128 && MT == 16) return act_budget<128, 16, VAR_TCGEN05>();  // the tcgen05 path's smaller area
  switch (MT) {
    case 1: return MCfg<1>::ACT_BUDGET;
    case 2: return MCfg<2>::ACT_BUDGET;
    case 4: return MCfg<4>::ACT_BUDGET;
    case 8: return MCfg<8>::ACT_BUDGET;
    default: return MCfg<16>::ACT_BUDGET;
  }
}

}  // namespace

cudaError_t device_error_word(int dev, unsigned** out) { return error_word(dev, out); }

namespace {
std::atomic<uint64_t> g_wait_limit{WAIT_LIMIT_NS};
}  // namespace
void set_gemv_wait_limit_ns(uint64_t ns) { g_wait_limit.store(ns == 0 ? WAIT_LIMIT_NS : ns); }
uint64_t gemv_wait_limit_ns() { return g_wait_limit.load(); }

// Row counts from which a launch takes the virtual-tile kernel (4 to 32 rows
// per pass); fewer rows take the one-tile-per-unit kernel below.
#ifndef Q8_VT_MIN_M
#define Q8_VT_MIN_M 9
#endif

bool plan_gemv(const DeviceInfo& dev, int64_t N, int64_t K, int M, bool fused, bool tcgen05, GemvPlan* out,
               bool allow_vt, bool allow_image) {
  // (shapes the virtual-tile plan cannot take, e.g. K beyond what its splits
  // cover, fall back to the kernel below: the bits are the same)
  if (allow_vt && !tcgen05 && M >= Q8_VT_MIN_M && plan_vt(dev, N, K, M, fused, allow_image, out)) return true;
  GemvPlan q;
  q.N = N;
  q.K = K;
  q.NB = K / QK;
  q.M = M;
  const int Mp = M > 16 ? 16 : M;  // rows per launch
  q.MT = mt_of(Mp);
  q.R = layout_tile_rows(N);
  const int P = 128 / q.R;
  const int64_t T = (N + q.R - 1) / q.R;
  const int64_t nch = (q.NB + CHUNK_BLOCKS - 1) / CHUNK_BLOCKS;
  if (T > ((int64_t)1 << 30) || nch > ((int64_t)1 << 24)) return false;
  q.T = (int)T;
  q.nch = (int)nch;
  // the tcgen05 kernel serves 128-row tiles with 16 rows per pass
  q.u5 = tcgen05 && q.R == 128 && q.MT == 16;
  if (occupancy(q.R, q.MT, fused, q.u5) < 1) return false;  // also sets the smem attribute
  // rounds of P chunks; a unit is RU rounds (a power of two)
  const int64_t nrounds_all = (nch + P - 1) / P;
  int64_t ru = 1;
  while (ru < nrounds_all && ru < MAX_ROUNDS_PER_UNIT) ru <<= 1;
  // sized for MT rows: the kernel's reduction depth is fixed by MT, not M
  const int budget = budget_of(q.R, q.MT, q.u5);
  while (ru > 1 && act_bytes(q.MT, P, (int)ru) > budget) ru >>= 1;
  if (act_bytes(q.MT, P, (int)ru) > budget) return false;
  int64_t S = (nrounds_all + ru - 1) / ru;
  // too few tiles to occupy the GPU: split along K while that helps
  while (T * S < dev.sm_count / 2 && ru > 1) {
    ru >>= 1;
    S = (nrounds_all + ru - 1) / ru;
  }
  if (S > MAX_SPLITS) return false;
  if (S > 1 && T > MAX_SPLIT_TILES) return false;
  q.RU = (int)ru;
  q.S = (int)S;
  const int64_t units = T * S;
  if (units > ((int64_t)1 << 31) - 1) return false;
  q.units = (int)units;
  // one persistent CTA per SM; SMs this kernel leaves free take the next
  // kernel's CTAs early (PDL), which stream their first weights at once
  q.grid = (int)(units < dev.sm_count ? units : dev.sm_count);
  // When every unit covers all of K and every CTA has exactly one unit, the
  // CTAs stage the same activation blocks on the critical path.  If one CTA
  // would stage more than one batch of them (MCfg::STAGE_TARGET), clusters
  // of 2 or 4 CTAs share the work (each stages 1/c and writes it to all,
  // then a cluster barrier); otherwise each CTA stages everything itself, which is cheaper
  // than the barrier.  CTAs that loop over several units stage once and
  // amortize it, so they run unclustered (no co-scheduling constraint).  The
  // grid is rounded down to a multiple of the cluster size (persistent CTAs
  // pick up the remaining units).
  q.cluster = 1;
  if (q.S == 1 && units <= dev.sm_count) {
    const int64_t blocks = (int64_t)Mp * q.NB;
#if defined(Q8_MAX_CLUSTER)
    const int cmax = Q8_MAX_CLUSTER;
#else
    const int cmax = 4;
#endif
    int want = 1;
    const int target = stage_target_of(q.MT);
    while (want < cmax && (blocks + want - 1) / want > target) want <<= 1;
    for (int c = want; c >= 2; c >>= 1) {
      if (q.grid >= c && cluster_fits(q.R, q.MT, fused, q.u5, c)) {
        q.cluster = c;
        q.grid = q.grid / c * c;
        break;
      }
    }
  }
  q.ws_bytes = q.S > 1 ? TICKET_BYTES + (size_t)q.S * Mp * N * 4 : 0;
  *out = q;
  return true;
}

cudaError_t launch_gemv(const GemvPlan& p, const uint8_t* W, const uint8_t* A, const float* x,
                        uint8_t* A_out, float* y, void* workspace, bool pdl, cudaStream_t s,
                        uint8_t* h_blocks) {
  if (p.vt) {
    if (h_blocks != nullptr) return cudaErrorInvalidValue;  // the SwiGLU epilogue is planned without vt
    return launch_vt(p, W, A, x, A_out, y, workspace, pdl, s);
  }
  const bool fused = (x != nullptr);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  unsigned* err = nullptr;
  if ((e = error_word(dev, &err)) != cudaSuccess) return e;
  for (int m0 = 0; m0 < p.M; m0 += 16) {
    const int Mp = (p.M - m0) < 16 ? (p.M - m0) : 16;
    GemvArgs args;
    args.W = W;
    args.A = A ? A + (size_t)m0 * p.NB * BLOCK_BYTES : nullptr;
    args.x = x ? x + (size_t)m0 * p.K : nullptr;
    args.A_out = A_out ? A_out + (size_t)m0 * p.NB * BLOCK_BYTES : nullptr;
    args.y = y != nullptr ? y + (size_t)m0 * p.N : nullptr;
    args.h_blocks = h_blocks != nullptr ? h_blocks + (size_t)m0 * (p.N / 64) * BLOCK_BYTES : nullptr;
    args.ws_cnt = p.S > 1 ? reinterpret_cast<unsigned*>(workspace) : nullptr;
    args.ws_part = p.S > 1 ? reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(workspace) + TICKET_BYTES)
                           : nullptr;
    args.err = err;
    args.wait_ns = gemv_wait_limit_ns();
    args.N = p.N;
    args.NB = (int)p.NB;
    args.nch = p.nch;
    args.T = p.T;
    args.M = Mp;
    args.RU = p.RU;
    args.S = p.S;
    args.units = p.units;
    // A last pass with fewer rows (M > 16) may use a smaller MT.  A unit
    // sized for 16 rows fits MT 4 and 8 (fewer rows, no smaller budget per
    // row); MT 1 and 2 have a smaller budget, so such a pass runs with MT 4.
    int MT = p.MT;
    if (Mp < 16 && p.MT == 16) {
      MT = mt_of(Mp);
      if (MT <= 2) MT = 4;
    }
    // shared memory for the unit's staged activations only (a launch with a
    // short K range does not reserve the whole budget)
    args.act_smem = (act_bytes(MT, 128 / p.R, p.RU) + 15) / 16 * 16;
    // kernel variant: the SwiGLU epilogue when h_blocks is given, the tcgen05
    // block dots when the plan asks for them (16-row passes), else the default
    const int var = h_blocks != nullptr ? VAR_SWIGLU : (p.u5 && MT == 16) ? VAR_TCGEN05 : VAR_DEFAULT;
    switch (p.R) {
      case 16: e = launch_gemv_r<16>(args, MT, fused, var, p.grid, p.cluster, pdl, s); break;
      case 32: e = launch_gemv_r<32>(args, MT, fused, var, p.grid, p.cluster, pdl, s); break;
      case 64: e = launch_gemv_r<64>(args, MT, fused, var, p.grid, p.cluster, pdl, s); break;
      default: e = launch_gemv_r<128>(args, MT, fused, var, p.grid, p.cluster, pdl, s); break;
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
