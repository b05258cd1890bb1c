// q8_gemv_vt.cu -- launch planning and dispatch of the virtual-tile decode
// GEMV (q8_gemv_vt.cuh; instantiated per row count in q8_gemv_vt_m*.cu).
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "q8_gemv_vt.cuh"
#include "q8_internal.h"

namespace q8 {
namespace vt {

// ---- the staged image of the activations (calls with many rows) ---------------
// Quantizes x [M][K] once, exactly as q8_quantize_act does (FROM_BLOCKS:
// reads the blocks A [M][NB] instead), and writes the staged layout of the
// virtual-tile kernel for each launch of 32 rows and each K range of UB
// blocks.  Launch p (rows 32p..) owns pass_stride bytes at
// img + p * pass_stride; its image s (act_bytes(UB) bytes for its MP staged
// rows, at s * act_bytes(UB) within) holds the fp16 quants of its row m,
// block bl at m * rsb + bl * 64 and the fp32 scale at MP * rsb + (bl * MP +
// m) * 4.  Every launch has MP_full staged rows except the last (MP_last).
// Optionally also writes the blocks themselves (A_out, quantizing only).
// Eight lanes per block; the trip counts are uniform across the CTA.
constexpr int IMG_THREADS = 256;
constexpr int IMG_B = 2;  // blocks per lane group in flight
template <bool FROM_BLOCKS>
__global__ void __launch_bounds__(IMG_THREADS) vt_image_kernel(const float* __restrict__ x,
                                                               const uint8_t* __restrict__ A, int M, int NB, int UB,
                                                               int MP_full, int MP_last, uint8_t* __restrict__ img,
                                                               int64_t pass_stride, uint8_t* __restrict__ A_out) {
  pdl_launch_dependents();
  pdl_wait();
  constexpr int B = IMG_B;
  const int sub = threadIdx.x & 7;
  const int rsb = act_rsb(UB);
  const int last_pass = (M - 1) >> 5;
  const int64_t total = (int64_t)M * NB;
  const int64_t groups = (int64_t)gridDim.x * (IMG_THREADS / 8);
  const int64_t g0 = (int64_t)blockIdx.x * (IMG_THREADS / 8) + (threadIdx.x >> 3);
  for (int64_t base = 0; base < total; base += groups * B) {
    int64_t blk[B];
    uint32_t w[B];
    float d[B];
    if constexpr (FROM_BLOCKS) {
      // a block is 34 bytes (2-byte aligned): the binary16 scale, then 32 quants
#pragma unroll
      for (int q = 0; q < B; ++q) {
        blk[q] = base + q * groups + g0;
        w[q] = 0u;
        d[q] = 0.0f;
        if (blk[q] < total) {
          const unsigned short* b16 = reinterpret_cast<const unsigned short*>(A + blk[q] * BLOCK_BYTES);
          w[q] = (uint32_t)__ldcg(b16 + 1 + 2 * sub) | ((uint32_t)__ldcg(b16 + 2 + 2 * sub) << 16);
          d[q] = __half2float(__ushort_as_half(__ldcg(b16)));
        }
      }
    } else {
      float4 v[B];
#pragma unroll
      for (int q = 0; q < B; ++q) {
        blk[q] = base + q * groups + g0;
        v[q] = blk[q] < total ? __ldcg(reinterpret_cast<const float4*>(x + blk[q] * QK) + sub)
                              : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      }
      quantize_group8<B>(v, w, d);
    }
#pragma unroll
    for (int q = 0; q < B; ++q) {
      if (blk[q] >= total) continue;
      const int m = (int)(blk[q] / NB), b = (int)(blk[q] - (int64_t)m * NB);
      const int pass = m >> 5, ml = m & 31;
      const int MP = pass == last_pass ? MP_last : MP_full;
      const int s = b / UB, bl = b - s * UB;
      uint8_t* im = img + pass * pass_stride + (int64_t)s * ((int64_t)MP * rsb + (int64_t)UB * MP * 4);
      uint32_t lo, hi;
      i8x4_to_h2x2(w[q], lo, hi);
      *reinterpret_cast<uint2*>(im + (size_t)ml * rsb + bl * 64 + sub * 8) = make_uint2(lo, hi);
      if (sub == 0) reinterpret_cast<float*>(im + (size_t)MP * rsb)[bl * MP + ml] = d[q];
      if (!FROM_BLOCKS && A_out != nullptr) store_block_lane(A_out + blk[q] * BLOCK_BYTES, sub, w[q], d[q]);
    }
  }
}


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

// Clusters of `cl` CTAs that can be resident at once, per device,
// instantiation and cluster size (queried once).
int g_max_clusters[MAX_DEVICES][4][2][9];
bool g_max_clusters_known[MAX_DEVICES][4][2][9] = {};
int max_clusters(int dev, int MT, bool fused, int cl) {
  std::lock_guard<std::mutex> lk(g_attr_mu);
  const int mi = mi_of(MT), fi = fused ? 1 : 0;
  if (!g_max_clusters_known[dev][mi][fi][cl]) {
    int n;
    switch (MT) {
      case 4: n = max_clusters_m<4>(fused, cl); break;
      case 8: n = max_clusters_m<8>(fused, cl); break;
      case 16: n = max_clusters_m<16>(fused, cl); break;
      default: n = max_clusters_m<32>(fused, cl); break;
    }
    g_max_clusters[dev][mi][fi][cl] = n;
    g_max_clusters_known[dev][mi][fi][cl] = true;
  }
  return g_max_clusters[dev][mi][fi][cl];
}

// A call with at least this many rows per pass stages its activations once
// (the image kernel: quantizes x into the workspace and A_blocks_out, or
// converts the blocks) and runs the GEMV on the staged images: every CTA
// quantizing or converting all of its K range costs more than the extra
// launch once the rows are many.
constexpr int QUANT_FIRST_MT = 16;

// Workspace of a plan: the tickets (always reserved: one workspace serves
// every call, and a split call needs them zero), the partials when split
// along K without a cluster, then the staged images of a quantize-first
// fused call.
size_t act_offset(const GemvPlan& q, int Mp) {
  const size_t part = TICKET_BYTES + (q.S > 1 && q.cluster == 1 ? (size_t)q.S * Mp * q.Np * 4 : 0);
  return (part + 15) & ~(size_t)15;
}

// Staged rows of an instantiation and the bytes of one staged image.
int mp_of(int MT) { return MT < 8 ? 8 : MT; }
size_t image_bytes(int MT, int UB) {
  const int MP = mp_of(MT);
  return (size_t)MP * act_rsb(UB) + (size_t)UB * MP * 4;
}
// Images of a call: every launch of 32 rows owns S images of the plan's
// largest instantiation.
size_t pass_stride(const GemvPlan& q) { return (size_t)q.S * image_bytes(q.MT, q.UB); }

int64_t pow2_floor(int64_t v) {
  int64_t p = 1;
  while (p * 2 <= v) p *= 2;
  return p;
}

}  // namespace
}  // namespace vt

// Plan of the virtual-tile kernel for M rows (passes of at most 32 rows).
bool plan_vt(const DeviceInfo& dev, int64_t N, int64_t K, int M, bool fused, bool image, GemvPlan* out) {
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
  // split along K: the S CTAs of a virtual tile form a cluster and combine
  // through distributed shared memory, when every virtual tile's cluster
  // can be resident at once (a CTA of a cluster waits for its peers before
  // it moves on, so a second wave would wait for the first)
  if (S > 1 && S <= MAX_CLUSTER) {
    const bool kfused = fused && !(image && q.MT >= QUANT_FIRST_MT);  // the instantiation launched
    if (ensure_attributes(dev.device, q.MT, kfused) != cudaSuccess) return false;
    if (TV <= max_clusters(dev.device, q.MT, kfused, (int)S)) {
      q.cluster = (int)S;
      q.grid = (int)(TV * S);
    }
  }
  q.ws_bytes = q.S > 1 ? act_offset(q, Mp) : 0;
  q.img = image && q.MT >= QUANT_FIRST_MT;
  if (q.img) q.ws_bytes = act_offset(q, Mp) + (size_t)((M + 31) / 32) * pass_stride(q);
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
  const uint8_t* img = nullptr;
  if (p.img) {
    // stage once into the images (bit-exact with the in-kernel staging),
    // then the GEMV on them as a programmatic dependent
    uint8_t* im = reinterpret_cast<uint8_t*>(workspace) + act_offset(p, p.M > 32 ? 32 : p.M);
    const int last = p.M - (p.M - 1) / 32 * 32;  // rows of the last launch
    const int mt_last = mt_of(last) < p.MT ? mt_of(last) : p.MT;
    const int64_t nblocks = (int64_t)p.M * p.NB;
    const int64_t per_cta = (int64_t)(IMG_THREADS / 8) * IMG_B;
    int64_t grid = (nblocks + per_cta - 1) / per_cta;
    if (grid > 8 * 1024) grid = 8 * 1024;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(IMG_THREADS);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    e = fused ? cudaLaunchKernelEx(&cfg, vt_image_kernel<false>, x, (const uint8_t*)nullptr, p.M, (int)p.NB,
                                   p.UB, mp_of(p.MT), mp_of(mt_last), im, (int64_t)pass_stride(p), A_out)
              : cudaLaunchKernelEx(&cfg, vt_image_kernel<true>, (const float*)nullptr, A, p.M, (int)p.NB, p.UB,
                                   mp_of(p.MT), mp_of(mt_last), im, (int64_t)pass_stride(p), (uint8_t*)nullptr);
    if (e != cudaSuccess) return e;
    img = im;
    A = nullptr;
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
    a.img = img ? img + (size_t)(m0 / 32) * pass_stride(p) : nullptr;
    a.cl = p.cluster;
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
