// q8_gemv_vt.cu -- launch planning and dispatch of the virtual-tile decode
// GEMV (q8_gemv_vt.cuh; instantiated per row count in q8_gemv_vt_m*.cu).
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "q8_gemv_vt.cuh"
#include "q8_internal.h"

namespace q8 {
namespace vt {


namespace {

int mt_of(int M) { return M <= 4 ? 4 : M <= 8 ? 8 : M <= 16 ? 16 : 32; }
int mi_of(int MT) { return MT == 4 ? 0 : MT == 8 ? 1 : MT == 16 ? 2 : 3; }

int ub_max_of(int MT) {
  switch (MT) {
    case 4: return Cfg<4>::UB_MAX;
    case 8: return Cfg<8>::UB_MAX;
    case 16: return Cfg<16>::UB_MAX;
    default: return Cfg<32>::UB_MAX;
  }
}
int raw_of(int MT, int UB) {
  switch (MT) {
    case 4: return raw_bytes<4>(UB);
    case 8: return raw_bytes<8>(UB);
    case 16: return raw_bytes<16>(UB);
    default: return raw_bytes<32>(UB);
  }
}

constexpr int MAX_DEVICES = 64;

// Kernel attributes (shared-memory size and carveout) are set once per
// instantiation and device, not on every launch.
std::mutex g_attr_mu;
bool g_attr_done[MAX_DEVICES][4][2] = {};
cudaError_t ensure_attributes(int dev, int MT, bool fused) {
  std::lock_guard<std::mutex> lk(g_attr_mu);
  bool& done = g_attr_done[dev][mi_of(MT)][fused ? 1 : 0];
  if (done) return cudaSuccess;
  cudaError_t e;
  switch (MT) {
    case 4: e = attributes_m<4>(fused); break;
    case 8: e = attributes_m<8>(fused); break;
    case 16: e = attributes_m<16>(fused); break;
    default: e = attributes_m<32>(fused); break;
  }
  if (e == cudaSuccess) done = true;
  return e;
}

// A fused call with at least this many rows per pass quantizes x once (the
// quantize kernel, into A_blocks_out or the workspace) and runs the GEMV on
// the blocks: every CTA quantizing all of its K range costs more than the
// extra launch once the rows are many.
constexpr int QUANT_FIRST_MT = 16;

// Workspace of a plan: the tickets (always reserved: one workspace serves
// every call, and a split call needs them zero), the partials when split
// along K, then the quantized activations of a quantize-first fused call.
size_t act_offset(const GemvPlan& q, int Mp) {
  const size_t part = TICKET_BYTES + (q.S > 1 ? (size_t)q.S * Mp * q.Np * 4 : 0);
  return (part + 15) & ~(size_t)15;
}

int64_t pow2_floor(int64_t v) {
  int64_t p = 1;
  while (p * 2 <= v) p *= 2;
  return p;
}

}  // namespace
}  // namespace vt

// Plan of the virtual-tile kernel for M rows (passes of at most 32 rows).
bool plan_vt(const DeviceInfo& dev, int64_t N, int64_t K, int M, bool fused, GemvPlan* out) {
  using namespace vt;
  if (dev.device < 0 || dev.device >= MAX_DEVICES) return false;
  GemvPlan q;
  q.vt = true;
  q.N = N;
  q.K = K;
  q.NB = K / QK;
  q.M = M;
  const int Mp = M > 32 ? 32 : M;  // rows per launch
  q.MT = mt_of(Mp);
  q.R = layout_tile_rows(N);
  const int64_t T = (N + q.R - 1) / q.R;
  const int64_t TV = (N + VR - 1) / VR;
  const int64_t nch = (q.NB + CHUNK_BLOCKS - 1) / CHUNK_BLOCKS;
  if (T > ((int64_t)1 << 30) || nch > ((int64_t)1 << 24)) return false;
  q.T = (int)T;
  q.TV = (int)TV;
  q.nch = (int)nch;
  if (ensure_attributes(dev.device, q.MT, fused) != cudaSuccess) return false;
  // rounds per unit: all of K when the unit's activations fit, else the
  // largest power of two that does (split units must be aligned subtrees)
  const int64_t ru_max = ub_max_of(q.MT) / CHUNK_BLOCKS;
  int64_t ru = nch <= ru_max ? nch : pow2_floor(ru_max);
  int64_t S = (nch + ru - 1) / ru;
  // too few virtual tiles to occupy the GPU: split along K while that helps
  while (TV * S < dev.sm_count / 2 && ru > 1) {
    ru = (S == 1 && pow2_floor(ru) < ru) ? pow2_floor(ru) : ru / 2;
    S = (nch + ru - 1) / ru;
  }
  if (S > MAX_SPLITS) return false;
  if (S > 1 && TV > MAX_TILES_SPLIT) return false;
  const int64_t units = TV * S;
  if (units > ((int64_t)1 << 31) - 1) return false;
  q.RU = (int)ru;
  q.S = (int)S;
  q.UB = (int)(ru * CHUNK_BLOCKS);
  q.units = (int)units;
  q.grid = (int)(units < dev.sm_count ? units : dev.sm_count);
  q.Np = (int)((N + 3) / 4 * 4);
  q.cluster = 1;
  q.ws_bytes = q.S > 1 ? TICKET_BYTES + (size_t)q.S * Mp * q.Np * 4 : 0;
  if (fused && q.MT >= QUANT_FIRST_MT) q.ws_bytes = act_offset(q, Mp) + (size_t)M * q.NB * BLOCK_BYTES;
  *out = q;
  return true;
}

cudaError_t launch_vt(const GemvPlan& p, const uint8_t* W, const uint8_t* A, const float* x, uint8_t* A_out,
                      float* y, void* workspace, bool pdl, cudaStream_t s) {
  using namespace vt;
  bool fused = (x != nullptr);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  unsigned* err = nullptr;
  if ((e = device_error_word(dev, &err)) != cudaSuccess) return e;
  if (fused && p.MT >= QUANT_FIRST_MT) {
    // quantize once (bit-exact with the in-kernel quantization), then the
    // GEMV on the blocks as a programmatic dependent of the quantize kernel
    uint8_t* blocks = A_out != nullptr ? A_out
                                       : reinterpret_cast<uint8_t*>(workspace) + act_offset(p, p.M > 32 ? 32 : p.M);
    if ((e = launch_quantize(x, p.M, p.K, blocks, pdl, s)) != cudaSuccess) return e;
    A = blocks;
    x = nullptr;
    A_out = nullptr;
    fused = false;
    pdl = true;
  }
  for (int m0 = 0; m0 < p.M; m0 += 32) {
    const int Mp = (p.M - m0) < 32 ? (p.M - m0) : 32;
    // a last pass with fewer rows runs a smaller instantiation: its blocks
    // per unit never exceed the plan's, which fit the largest
    const int MT = mt_of(Mp) < p.MT ? mt_of(Mp) : p.MT;
    if ((e = ensure_attributes(dev, MT, fused)) != cudaSuccess) return e;
    Args a;
    a.W = W;
    a.A = A ? A + (size_t)m0 * p.NB * BLOCK_BYTES : nullptr;
    a.x = x ? x + (size_t)m0 * p.K : nullptr;
    a.A_out = A_out ? A_out + (size_t)m0 * p.NB * BLOCK_BYTES : nullptr;
    a.y = y + (size_t)m0 * p.N;
    a.ws_cnt = p.S > 1 ? reinterpret_cast<unsigned*>(workspace) : nullptr;
    a.ws_part = p.S > 1 ? reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(workspace) + TICKET_BYTES) : nullptr;
    a.err = err;
    a.wait_ns = gemv_wait_limit_ns();
    a.N = p.N;
    a.NB = (int)p.NB;
    a.nch = p.nch;
    a.T = p.T;
    a.R = p.R;
    a.G = VR / p.R;
    a.TV = p.TV;
    a.M = Mp;
    a.RU = p.RU;
    a.S = p.S;
    a.units = p.units;
    a.UB = p.UB;
    a.Np = p.Np;
    a.raw_bytes = raw_of(MT, p.UB);
    switch (MT) {
      case 4: e = launch_m<4>(a, fused, p.grid, pdl, s); break;
      case 8: e = launch_m<8>(a, fused, p.grid, pdl, s); break;
      case 16: e = launch_m<16>(a, fused, p.grid, pdl, s); break;
      default: e = launch_m<32>(a, fused, p.grid, pdl, s); break;
    }
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace q8
