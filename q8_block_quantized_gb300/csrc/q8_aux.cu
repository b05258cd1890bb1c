// q8_aux.cu -- activation quantization, weight repack/unpack and the exact
// block-dot test hook.
#include <cuda_runtime.h>

#include "q8_device.cuh"
#include "q8_internal.h"

namespace q8 {
namespace {

constexpr int QUANT_THREADS = 256;  // 8 warps, one 32-value block per warp

// One warp per block.  Blocks of an [M][K] matrix are consecutive runs of 32
// floats, so block g reads x[32g .. 32g+31] and writes out[34g .. 34g+33].
__global__ void __launch_bounds__(QUANT_THREADS) quantize_kernel(const float* __restrict__ x,
                                                                int64_t nblocks,
                                                                uint8_t* __restrict__ out) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t)blockIdx.x * (QUANT_THREADS / 32) + (threadIdx.x >> 5);
  const int64_t nwarps = (int64_t)gridDim.x * (QUANT_THREADS / 32);
  for (int64_t g = warp; g < nblocks; g += nwarps) {
    const float v = __ldcg(x + g * QK + lane);
    const LaneQuant lq = quantize_lane(v);
    uint8_t* ob = out + g * BLOCK_BYTES;
    ob[2 + lane] = (uint8_t)(lq.q & 0xff);
    if (lane < 2) ob[lane] = (uint8_t)(lane == 0 ? (lq.d16 & 0xff) : (lq.d16 >> 8));
  }
}

// One thread per (row n, block b): 34 source bytes -> two 16-byte quant runs
// and one scale in the packed layout.  Row index fastest so packed writes of
// neighbouring threads are contiguous.
// `rows` holds [N][nb] row-contiguous blocks, `packed` the packed layout;
// inverse == false copies rows -> packed, inverse == true packed -> rows.
// R is the tile height: q8_packed_tile_rows(N) for weights, 128 for the
// activations of the prefill GEMM.
// zero, nzero: words to clear first (the prefill GEMM's split flags; none
// for the weights)
__global__ void repack_kernel(uint8_t* rows, int64_t N, int64_t nb, int R, uint8_t* packed, bool inverse,
                              unsigned* zero, int nzero) {
  pdl_launch_dependents();
  pdl_wait();  // (a no-op unless launched as a programmatic dependent)
  if (blockIdx.x == 0)
    for (int k = threadIdx.x; k < nzero; k += blockDim.x) zero[k] = 0u;
  const int64_t T = (N + R - 1) / R;
  const int64_t total = T * nb * R;
  for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < total;
       g += (int64_t)gridDim.x * blockDim.x) {
    const int i = (int)(g % R);
    const int64_t rest = g / R;
    const int64_t b = rest % nb;
    const int64_t t = rest / nb;
    const int r = tile_rows(t, N, R);
    if (i >= r) continue;
    const int64_t n = t * R + i;
    const int64_t c = b / CHUNK_BLOCKS;
    const int j = (int)(b % CHUNK_BLOCKS);
    const int kb = chunk_blocks(c, nb);
    uint8_t* chunk = packed + chunk_offset(t, c, r, R, nb);
    uint16_t* s16 = reinterpret_cast<uint16_t*>(rows + (n * nb + b) * BLOCK_BYTES);
    uint4* q0 = reinterpret_cast<uint4*>(chunk + chunk_quant_off(j, 0, i, r));
    uint4* q1 = reinterpret_cast<uint4*>(chunk + chunk_quant_off(j, 1, i, r));
    uint16_t* sc = reinterpret_cast<uint16_t*>(chunk + chunk_scale_off(j, i, r, kb));
    if (!inverse) {
      uint32_t w[8 * 2];
#pragma unroll
      for (int k = 0; k < 16; ++k) w[k] = s16[1 + k];
      uint32_t p[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) p[k] = w[2 * k] | (w[2 * k + 1] << 16);
      *q0 = make_uint4(p[0], p[1], p[2], p[3]);
      *q1 = make_uint4(p[4], p[5], p[6], p[7]);
      *sc = s16[0];
    } else {
      const uint4 a = *q0, bq = *q1;
      const uint32_t p[8] = {a.x, a.y, a.z, a.w, bq.x, bq.y, bq.z, bq.w};
      s16[0] = *sc;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        s16[1 + 2 * k] = (uint16_t)(p[k] & 0xffffu);
        s16[2 + 2 * k] = (uint16_t)(p[k] >> 16);
      }
    }
  }
}

// Test hook: isum[m][n][b] from packed W and row-contiguous activation blocks.
__global__ void block_dots_kernel(const uint8_t* __restrict__ W, int64_t N, int64_t nb,
                                  const uint8_t* __restrict__ A, int M, int32_t* __restrict__ isum) {
  const int64_t total = (int64_t)M * N * nb;
  for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < total;
       g += (int64_t)gridDim.x * blockDim.x) {
    const int64_t b = g % nb;
    const int64_t n = (g / nb) % N;
    const int64_t m = g / (nb * N);
    const int R = layout_tile_rows(N);
    const int64_t t = n / R;
    const int i = (int)(n % R);
    const int r = tile_rows(t, N, R);
    const int64_t c = b / CHUNK_BLOCKS;
    const int j = (int)(b % CHUNK_BLOCKS);
    const uint8_t* chunk = W + chunk_offset(t, c, r, R, nb);
    const uint4 w0 = *reinterpret_cast<const uint4*>(chunk + chunk_quant_off(j, 0, i, r));
    const uint4 w1 = *reinterpret_cast<const uint4*>(chunk + chunk_quant_off(j, 1, i, r));
    uint4 a0, a1;
    load_block_quants_u16(A + (m * nb + b) * BLOCK_BYTES, a0, a1);
    isum[g] = dot_block(w0, w1, a0, a1);
  }
}

int grid_for(int64_t work, int per_cta) {
  int64_t g = (work + per_cta - 1) / per_cta;
  if (g < 1) g = 1;
  if (g > 65535LL * 32) g = 65535LL * 32;
  return (int)g;
}

}  // namespace

cudaError_t launch_quantize(const float* x, int64_t M, int64_t K, uint8_t* out, bool pdl,
                            cudaStream_t s) {
  const int64_t nblocks = M * (K / QK);
  // same carveout as the GEMV kernels, so it can share SMs with them
  cudaError_t e = cudaFuncSetAttribute(quantize_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                       (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid_for(nblocks, QUANT_THREADS / 32));
  cfg.blockDim = dim3(QUANT_THREADS);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, quantize_kernel, x, nblocks, out);
}

cudaError_t launch_repack(const uint8_t* src, int64_t N, int64_t K, uint8_t* dst, cudaStream_t s) {
  const int64_t nb = K / QK;
  const int R = layout_tile_rows(N);
  const int64_t total = ((N + R - 1) / R) * nb * R;
  repack_kernel<<<grid_for(total, 256), 256, 0, s>>>(const_cast<uint8_t*>(src), N, nb, R, dst, false, nullptr, 0);
  return cudaGetLastError();
}

cudaError_t launch_pack_act(const uint8_t* src, int64_t M, int64_t K, uint8_t* dst, bool pdl, cudaStream_t s,
                            unsigned* zero, int nzero) {
  const int64_t nb = K / QK;
  const int R = MAX_TILE_ROWS;
  const int64_t total = ((M + R - 1) / R) * nb * R;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid_for(total, 256));
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, repack_kernel, const_cast<uint8_t*>(src), M, nb, R, dst, false, zero, nzero);
}

cudaError_t launch_unpack(const uint8_t* packed, int64_t N, int64_t K, uint8_t* dst,
                          cudaStream_t s) {
  const int64_t nb = K / QK;
  const int R = layout_tile_rows(N);
  const int64_t total = ((N + R - 1) / R) * nb * R;
  repack_kernel<<<grid_for(total, 256), 256, 0, s>>>(dst, N, nb, R, const_cast<uint8_t*>(packed), true, nullptr, 0);
  return cudaGetLastError();
}

cudaError_t launch_block_dots(const uint8_t* W, int64_t N, int64_t K, const uint8_t* A, int M,
                              int32_t* isum, cudaStream_t s) {
  const int64_t nb = K / QK;
  block_dots_kernel<<<grid_for((int64_t)M * N * nb, 256), 256, 0, s>>>(W, N, nb, A, M, isum);
  return cudaGetLastError();
}

}  // namespace q8
