// q8_kv.cu -- the int8 KV cache codec: K/V rows written into cache slots as
// int8 quants with one fp32 scale per 32 values, and read back as fp32
// ("Ferro" README, "Exactness, scheduling and operations (LM serving)", item
// "KV cache": llama.cpp's q8_0 scheme for the cache).  The codebook is the
// activation quantizer's (d = amax / 127, q = roundf(x * (1/d)), 1/d from the
// fp32 d); the scale is kept in fp32.
//
// Both kernels are elementwise and bound by HBM: 8 lanes per 32-value block,
// one 16-byte fp32 load or store and one 4-byte quant access per lane, so a
// warp touches 512 contiguous fp32 bytes and 128 contiguous quant bytes of a
// row; grid-stride loops over a grid of a few CTAs per SM.
#include <cuda_runtime.h>

#include "q8_device.cuh"
#include "q8_internal.h"

namespace q8 {
namespace {

constexpr int KV_THREADS = 256;
constexpr int KV_BATCH = 4;  // blocks per lane group with their loads in flight together

// Write: the rows' loads do not depend on their slots, so a batch issues the
// slot loads and the row loads together; a row whose slot lies outside the
// cache is skipped and reported.
__global__ void __launch_bounds__(KV_THREADS) kv_quantize_kernel(const float* __restrict__ x, int64_t rows,
                                                                int nb, const int32_t* __restrict__ slots,
                                                                int64_t capacity, int8_t* __restrict__ cq,
                                                                float* __restrict__ cd, unsigned* err) {
  pdl_launch_dependents();
  pdl_wait();
  const int sub = threadIdx.x & 7;
  const int64_t D = (int64_t)nb * QK;
  const int64_t total = rows * nb;
  const int64_t groups = (int64_t)gridDim.x * (KV_THREADS / 8);
  const int64_t g0 = (int64_t)blockIdx.x * (KV_THREADS / 8) + (threadIdx.x >> 3);
  // this lane group's blocks are g0, g0 + groups, ...: their (row, block)
  // advance by (groups / nb, groups % nb) with a carry (no division per block)
  const int64_t qg = groups / nb, rg = groups - (groups / nb) * nb;
  int64_t r_cur = g0 / nb, b_cur = g0 - (g0 / nb) * nb;
  // trip counts are uniform across the warp: the shuffles see full warps
  for (int64_t base = 0; base < total; base += groups * KV_BATCH) {
    float4 v[KV_BATCH];
    int64_t blk[KV_BATCH], r[KV_BATCH], bb[KV_BATCH], s[KV_BATCH];
    bool in[KV_BATCH];
#pragma unroll
    for (int q = 0; q < KV_BATCH; ++q) {
      blk[q] = base + q * groups + g0;
      in[q] = blk[q] < total;
      r[q] = r_cur;
      bb[q] = b_cur;
      r_cur += qg;
      b_cur += rg;
      if (b_cur >= nb) {
        b_cur -= nb;
        ++r_cur;
      }
      s[q] = in[q] ? (slots != nullptr ? (int64_t)__ldcg(slots + r[q]) : r[q]) : -1;
      v[q] = in[q] ? __ldcs(reinterpret_cast<const float4*>(x + blk[q] * QK) + sub)
                   : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
    uint32_t w[KV_BATCH];
    float d[KV_BATCH];
    quantize_group8<KV_BATCH, false>(v, w, d);
#pragma unroll
    for (int q = 0; q < KV_BATCH; ++q) {
      if (!in[q]) continue;
      const int64_t b = bb[q];
      if (s[q] < 0 || s[q] >= capacity) {
        if (sub == 0 && b == 0) atomicOr(err, ERR_KV_SLOT);
        continue;
      }
      reinterpret_cast<uint32_t*>(cq + s[q] * D + b * QK)[sub] = w[q];
      if (sub == 0) cd[s[q] * nb + b] = d[q];
    }
  }
}

// Read back: a batch loads its slots first, then every block's quants and
// scale, then stores; a row whose slot lies outside the cache reads as zeros
// and is reported.
__global__ void __launch_bounds__(KV_THREADS) kv_dequantize_kernel(const int8_t* __restrict__ cq,
                                                                  const float* __restrict__ cd,
                                                                  int64_t capacity, int nb,
                                                                  const int32_t* __restrict__ slots,
                                                                  int64_t rows, float* __restrict__ out,
                                                                  unsigned* err) {
  pdl_launch_dependents();
  pdl_wait();
  const int sub = threadIdx.x & 7;
  const int64_t D = (int64_t)nb * QK;
  const int64_t total = rows * nb;
  const int64_t groups = (int64_t)gridDim.x * (KV_THREADS / 8);
  const int64_t g0 = (int64_t)blockIdx.x * (KV_THREADS / 8) + (threadIdx.x >> 3);
  const int64_t qg = groups / nb, rg = groups - (groups / nb) * nb;
  int64_t r_cur = g0 / nb, b_cur = g0 - (g0 / nb) * nb;
  for (int64_t base = 0; base < total; base += groups * KV_BATCH) {
    int64_t blk[KV_BATCH], b[KV_BATCH], s[KV_BATCH];
    bool in[KV_BATCH], ok[KV_BATCH];
#pragma unroll
    for (int q = 0; q < KV_BATCH; ++q) {
      blk[q] = base + q * groups + g0;
      in[q] = blk[q] < total;
      const int64_t r = r_cur;
      b[q] = b_cur;
      r_cur += qg;
      b_cur += rg;
      if (b_cur >= nb) {
        b_cur -= nb;
        ++r_cur;
      }
      s[q] = in[q] ? (slots != nullptr ? (int64_t)__ldcg(slots + r) : r) : -1;
    }
    uint32_t w[KV_BATCH];
    float d[KV_BATCH];
#pragma unroll
    for (int q = 0; q < KV_BATCH; ++q) {
      ok[q] = in[q] && s[q] >= 0 && s[q] < capacity;
      w[q] = ok[q] ? __ldcs(reinterpret_cast<const unsigned int*>(cq + s[q] * D + b[q] * QK) + sub) : 0u;
      d[q] = ok[q] ? __ldcs(cd + s[q] * nb + b[q]) : 0.0f;
    }
#pragma unroll
    for (int q = 0; q < KV_BATCH; ++q) {
      if (!in[q]) continue;
      if (!ok[q] && sub == 0 && b[q] == 0) atomicOr(err, ERR_KV_SLOT);
      float4 o;
      o.x = __fmul_rn((float)(int)(int8_t)(w[q] & 0xffu), d[q]);
      o.y = __fmul_rn((float)(int)(int8_t)((w[q] >> 8) & 0xffu), d[q]);
      o.z = __fmul_rn((float)(int)(int8_t)((w[q] >> 16) & 0xffu), d[q]);
      o.w = __fmul_rn((float)(int)(int8_t)(w[q] >> 24), d[q]);
      __stcs(reinterpret_cast<float4*>(out + blk[q] * QK) + sub, o);
    }
  }
}

int kv_grid(int64_t total_blocks, int sm_count) {
  const int64_t per_cta = KV_THREADS / 8;
  int64_t g = (total_blocks + per_cta - 1) / per_cta;
  const int64_t cap = (int64_t)sm_count * 8;  // 8 CTAs (2048 threads) per SM
  return (int)(g < cap ? (g < 1 ? 1 : g) : cap);
}

}  // namespace

cudaError_t launch_kv_quantize(const float* x, int64_t rows, int64_t D, const int32_t* slots, int64_t capacity,
                               int8_t* cq, float* cd, int sm_count, bool pdl, cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  unsigned* err = nullptr;
  if ((e = device_error_word(dev, &err)) != cudaSuccess) return e;
  const int nb = (int)(D / QK);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kv_grid(rows * nb, sm_count));
  cfg.blockDim = dim3(KV_THREADS);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kv_quantize_kernel, x, rows, nb, slots, capacity, cq, cd, err);
}

cudaError_t launch_kv_dequantize(const int8_t* cq, const float* cd, int64_t capacity, int64_t D,
                                 const int32_t* slots, int64_t rows, float* out, int sm_count, bool pdl,
                                 cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  unsigned* err = nullptr;
  if ((e = device_error_word(dev, &err)) != cudaSuccess) return e;
  const int nb = (int)(D / QK);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kv_grid(rows * nb, sm_count));
  cfg.blockDim = dim3(KV_THREADS);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kv_dequantize_kernel, cq, cd, capacity, nb, slots, rows, out, err);
}

}  // namespace q8
