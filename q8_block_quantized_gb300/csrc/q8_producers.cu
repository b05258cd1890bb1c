// q8_producers.cu -- fused producers of the next GEMM's int8 input ("Ferro"
// README, "How the iGPU path is fast", item 3: the residual add, the norm
// and the int8 quantization in one pass; SwiGLU emitting the next GEMM's
// int8 input directly).
//
// Both kernels end in the activation quantization of q8_quantize_act (the
// same bits) and write row-contiguous Q8_0 blocks [M][K/32].  Their
// floating-point steps are single-precision operations with one IEEE
// rounding each (explicit _rn intrinsics, so no contraction into fma):
//   RMSNorm: h = x + delta; s = sum_k h_k^2 as the pairwise tree over k,
//            padded with zeros to a power of two; ms = s / K;
//            r = 1 / sqrt(ms + eps); y_k = (h_k * r) * gamma_k.
//   SwiGLU:  h = silu(g) * u, silu(g) = g / (1 + e^-g), e^x by the fixed
//            procedure exp_cw (q8_device.cuh).
#include <cuda_runtime.h>

#include "q8_device.cuh"
#include "q8_internal.h"

namespace q8 {
namespace {

constexpr int NORM_THREADS = 256;    // 8 warps per row
constexpr int SWIGLU_THREADS = 256;  // 32 blocks per pass, 8 lanes each
constexpr int NORM_LEVELS = 20;      // binary counter over chunks: up to 2^19 chunks of 8

__device__ __forceinline__ float4 add4(float4 a, float4 b) {
  return make_float4(__fadd_rn(a.x, b.x), __fadd_rn(a.y, b.y), __fadd_rn(a.z, b.z), __fadd_rn(a.w, b.w));
}

// ---- residual add + RMSNorm + quantization: one CTA per row ----
// The sum of squares is the pairwise tree over k with P = 2^ceil(log2 K)
// leaves (zeros past K).  Thread t sums the aligned leaf segment
// [tL, (t+1)L), L = P / 256 (one leaf for threads t < P when P < 256), in
// chunks of 8 leaves merged by a binary counter (what is left merges from the
// lowest level up, which is what the zero leaves give); then a butterfly
// inside each warp and a pairwise tree over the 8 warps.  Each step adds two
// adjacent subtrees of equal size, so the result is the tree sum.
__global__ void __launch_bounds__(NORM_THREADS)
    rmsnorm_quant_kernel(const float* x, const float* delta, const float* __restrict__ gamma, float eps,
                         int64_t K, float* h_out, uint8_t* __restrict__ out) {
  // h_out may be x or delta (an in-place residual update): no restrict on them
  pdl_launch_dependents();
  pdl_wait();
  __shared__ float wsum[NORM_THREADS / 32];
  __shared__ float rs;
  const int64_t m = blockIdx.x;
  const float* xr = x + m * K;
  const float* dr = delta != nullptr ? delta + m * K : nullptr;
  float* hr = h_out != nullptr ? h_out + m * K : nullptr;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  int64_t P = 1;
  while (P < K) P <<= 1;
  const int64_t L = P >= NORM_THREADS ? P / NORM_THREADS : 1;
  const int64_t k0 = (int64_t)threadIdx.x * L;
  float seg = 0.0f;
  if (L < 8) {
    // 1, 2 or 4 leaves (K <= 512): scalar loads
    float sq[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t k = k0 + j;
      if (j < L && k < K) {
        const float h = dr != nullptr ? __fadd_rn(__ldcg(xr + k), __ldcg(dr + k)) : __ldcg(xr + k);
        if (hr != nullptr) hr[k] = h;
        sq[j] = __fmul_rn(h, h);
      }
    }
    seg = L == 1 ? sq[0] : L == 2 ? __fadd_rn(sq[0], sq[1])
                                  : __fadd_rn(__fadd_rn(sq[0], sq[1]), __fadd_rn(sq[2], sq[3]));
  } else {
    float slot[NORM_LEVELS];
    int64_t c = 0;
    // chunks of 8 leaves; K is a multiple of 32, so a chunk is all data or all padding
    for (; c < L / 8 && k0 + 8 * c < K; ++c) {
      const int64_t k = k0 + 8 * c;
      float4 a = __ldcg(reinterpret_cast<const float4*>(xr + k));
      float4 b = __ldcg(reinterpret_cast<const float4*>(xr + k + 4));
      if (dr != nullptr) {
        a = add4(a, __ldcg(reinterpret_cast<const float4*>(dr + k)));
        b = add4(b, __ldcg(reinterpret_cast<const float4*>(dr + k + 4)));
      }
      if (hr != nullptr) {
        *reinterpret_cast<float4*>(hr + k) = a;
        *reinterpret_cast<float4*>(hr + k + 4) = b;
      }
      float v = __fadd_rn(__fadd_rn(__fadd_rn(__fmul_rn(a.x, a.x), __fmul_rn(a.y, a.y)),
                                    __fadd_rn(__fmul_rn(a.z, a.z), __fmul_rn(a.w, a.w))),
                          __fadd_rn(__fadd_rn(__fmul_rn(b.x, b.x), __fmul_rn(b.y, b.y)),
                                    __fadd_rn(__fmul_rn(b.z, b.z), __fmul_rn(b.w, b.w))));
      bool placed = false;
#pragma unroll
      for (int l = 0; l < NORM_LEVELS; ++l) {
        if (!placed) {
          if ((c >> l) & 1) {
            v = __fadd_rn(slot[l], v);
          } else {
            slot[l] = v;
            placed = true;
          }
        }
      }
    }
    bool have = false;
#pragma unroll
    for (int l = 0; l < NORM_LEVELS; ++l) {
      if ((c >> l) & 1) {
        seg = have ? __fadd_rn(slot[l], seg) : slot[l];
        have = true;
      }
    }
  }
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) seg = __fadd_rn(seg, __shfl_xor_sync(0xffffffffu, seg, o));
  if (lane == 0) wsum[warp] = seg;
  __syncthreads();
  if (threadIdx.x == 0) {
    const float s = __fadd_rn(__fadd_rn(__fadd_rn(wsum[0], wsum[1]), __fadd_rn(wsum[2], wsum[3])),
                              __fadd_rn(__fadd_rn(wsum[4], wsum[5]), __fadd_rn(wsum[6], wsum[7])));
    const float ms = __fdiv_rn(s, (float)K);
    rs = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
  }
  __syncthreads();  // also makes this CTA's h stores visible to its pass 2
  const float r = rs;

  // pass 2: y = (h * r) * gamma, quantized; 8 lanes per block
  const int sub = threadIdx.x & 7, grp = threadIdx.x >> 3;
  const int64_t nb = K / QK;
  for (int64_t b0 = 0; b0 < nb; b0 += NORM_THREADS / 8) {  // same trip count in every thread
    const int64_t b = b0 + grp;
    float4 v[1] = {make_float4(0.0f, 0.0f, 0.0f, 0.0f)};
    if (b < nb) {
      const int64_t k = b * QK + 4 * sub;
      float4 h;
      if (hr != nullptr) {
        h = __ldcg(reinterpret_cast<const float4*>(hr + k));
      } else {
        h = __ldcg(reinterpret_cast<const float4*>(xr + k));
        if (dr != nullptr) h = add4(h, __ldcg(reinterpret_cast<const float4*>(dr + k)));
      }
      const float4 g = __ldcg(reinterpret_cast<const float4*>(gamma + k));
      v[0] = make_float4(__fmul_rn(__fmul_rn(h.x, r), g.x), __fmul_rn(__fmul_rn(h.y, r), g.y),
                         __fmul_rn(__fmul_rn(h.z, r), g.z), __fmul_rn(__fmul_rn(h.w, r), g.w));
    }
    uint32_t w[1];
    float d[1];
    quantize_group8<1>(v, w, d);
    if (b < nb) store_block_lane(out + (m * nb + b) * BLOCK_BYTES, sub, w[0], d[0]);
  }
}

// Rows of K <= 8192 (P <= 8192 leaves): the same tree with coalesced loads
// and h kept in registers.  Thread t holds the float4 groups f = t + 256 j,
// j < J = max(1, P / 1024): a group's 4 leaves are a subtree, a warp's 32
// consecutive groups (butterfly) one of 128 leaves, the CTA's 256 groups of
// index j (tree over the 8 warps) one of 1024 leaves, and the J of those
// meet in a pairwise tree.  In pass 2 the 8 lanes that hold a block's
// 8 groups are the 8 consecutive lanes of a quantization group.
template <int J>
__global__ void __launch_bounds__(NORM_THREADS)
    rmsnorm_quant_reg_kernel(const float* x, const float* delta, const float* __restrict__ gamma, float eps,
                             int64_t K, float* h_out, uint8_t* __restrict__ out) {
  // h_out may be x or delta (an in-place residual update): no restrict on them
  pdl_launch_dependents();
  pdl_wait();
  __shared__ float wsum[J][NORM_THREADS / 32];
  __shared__ float rs;
  const int64_t m = blockIdx.x;
  const float* xr = x + m * K;
  const float* dr = delta != nullptr ? delta + m * K : nullptr;
  float* hr = h_out != nullptr ? h_out + m * K : nullptr;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float4 v[J];
  float part[J];
#pragma unroll
  for (int j = 0; j < J; ++j) {
    const int64_t k = 4 * ((int64_t)threadIdx.x + NORM_THREADS * j);
    v[j] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (k < K) {
      v[j] = __ldcg(reinterpret_cast<const float4*>(xr + k));
      if (dr != nullptr) v[j] = add4(v[j], __ldcg(reinterpret_cast<const float4*>(dr + k)));
    }
  }
#pragma unroll
  for (int j = 0; j < J; ++j) {
    const int64_t k = 4 * ((int64_t)threadIdx.x + NORM_THREADS * j);
    if (hr != nullptr && k < K) *reinterpret_cast<float4*>(hr + k) = v[j];
    part[j] = __fadd_rn(__fadd_rn(__fmul_rn(v[j].x, v[j].x), __fmul_rn(v[j].y, v[j].y)),
                        __fadd_rn(__fmul_rn(v[j].z, v[j].z), __fmul_rn(v[j].w, v[j].w)));
  }
#pragma unroll
  for (int o = 1; o < 32; o <<= 1)
#pragma unroll
    for (int j = 0; j < J; ++j) part[j] = __fadd_rn(part[j], __shfl_xor_sync(0xffffffffu, part[j], o));
  if (lane == 0)
#pragma unroll
    for (int j = 0; j < J; ++j) wsum[j][warp] = part[j];
  __syncthreads();
  if (threadIdx.x == 0) {
    float t[J];
#pragma unroll
    for (int j = 0; j < J; ++j)
      t[j] = __fadd_rn(__fadd_rn(__fadd_rn(wsum[j][0], wsum[j][1]), __fadd_rn(wsum[j][2], wsum[j][3])),
                       __fadd_rn(__fadd_rn(wsum[j][4], wsum[j][5]), __fadd_rn(wsum[j][6], wsum[j][7])));
#pragma unroll
    for (int w = J; w > 1; w >>= 1)
#pragma unroll
      for (int j = 0; j < w / 2; ++j) t[j] = __fadd_rn(t[2 * j], t[2 * j + 1]);
    const float ms = __fdiv_rn(t[0], (float)K);
    rs = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
  }
  __syncthreads();
  const float r = rs;
  const int sub = threadIdx.x & 7;
  const int64_t nb = K / QK;
#pragma unroll
  for (int j = 0; j < J; ++j) {
    const int64_t f = (int64_t)threadIdx.x + NORM_THREADS * j;  // block f / 8, lane f % 8 = sub
    float4 y[1] = {make_float4(0.0f, 0.0f, 0.0f, 0.0f)};
    if (4 * f < K) {
      const float4 g = __ldcg(reinterpret_cast<const float4*>(gamma + 4 * f));
      y[0] = make_float4(__fmul_rn(__fmul_rn(v[j].x, r), g.x), __fmul_rn(__fmul_rn(v[j].y, r), g.y),
                         __fmul_rn(__fmul_rn(v[j].z, r), g.z), __fmul_rn(__fmul_rn(v[j].w, r), g.w));
    }
    uint32_t w[1];
    float d[1];
    quantize_group8<1>(y, w, d);
    if (4 * f < K) store_block_lane(out + (m * nb + f / 8) * BLOCK_BYTES, sub, w[0], d[0]);
  }
}

// ---- SwiGLU + quantization ----
// SwiGLU: swiglu_one and its e^x (exp_cw) are in q8_device.cuh.

// gu is [M][2F] (gate = columns [0, F), up = [F, 2F)); block b of the output
// (row b / nbr, block b % nbr) reads 32 gate and 32 up values.  A group of 8
// lanes takes SWIGLU_B blocks per pass (two measured slower: the kernel is
// bound by the arithmetic of the exact e^x and division, not by latency).
// The block index arithmetic runs in Idx (32-bit whenever the block count
// fits: a 64-bit division per block costs as much as the block's exponentials).
constexpr int SWIGLU_B = 1;
template <typename Idx>
__global__ void __launch_bounds__(SWIGLU_THREADS)
    swiglu_quant_kernel(const float* __restrict__ gu, int64_t F, Idx nbr, Idx total, uint8_t* __restrict__ out) {
  pdl_launch_dependents();
  pdl_wait();
  const int sub = threadIdx.x & 7;
  const Idx grp = (Idx)(((int64_t)blockIdx.x * SWIGLU_THREADS + threadIdx.x) >> 3);
  const Idx ngrp = (Idx)(((int64_t)gridDim.x * SWIGLU_THREADS) >> 3);
  for (Idx b0 = 0; b0 < total; b0 += ngrp * SWIGLU_B) {  // same trip count in every thread
    float4 g[SWIGLU_B], u[SWIGLU_B], v[SWIGLU_B];
#pragma unroll
    for (int q = 0; q < SWIGLU_B; ++q) {
      const Idx b = b0 + grp + q * ngrp;
      g[q] = u[q] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      if (b < total) {
        const Idx m = b / nbr, j = b - m * nbr;
        const float* row = gu + (int64_t)m * 2 * F + (int64_t)j * QK + 4 * sub;
        g[q] = __ldcg(reinterpret_cast<const float4*>(row));
        u[q] = __ldcg(reinterpret_cast<const float4*>(row + F));
      }
    }
#pragma unroll
    for (int q = 0; q < SWIGLU_B; ++q)
      v[q] = make_float4(swiglu_one(g[q].x, u[q].x), swiglu_one(g[q].y, u[q].y), swiglu_one(g[q].z, u[q].z),
                         swiglu_one(g[q].w, u[q].w));
    uint32_t w[SWIGLU_B];
    float d[SWIGLU_B];
    quantize_group8<SWIGLU_B>(v, w, d);
#pragma unroll
    for (int q = 0; q < SWIGLU_B; ++q) {
      const Idx b = b0 + grp + q * ngrp;
      if (b < total) store_block_lane(out + (int64_t)b * BLOCK_BYTES, sub, w[q], d[q]);
    }
  }
}

template <typename Kern, typename... Args>
cudaError_t launch_pdl(Kern kern, dim3 grid, int threads, bool pdl, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

}  // namespace

cudaError_t launch_rmsnorm_quantize(const float* x, const float* delta, const float* gamma, float eps,
                                    int64_t M, int64_t K, float* h_out, uint8_t* out, bool pdl,
                                    cudaStream_t s) {
  int64_t P = 1;
  while (P < K) P <<= 1;
  const dim3 grid((unsigned)M);
  switch (P <= 1024 ? 1 : P / 1024) {
    case 1: return launch_pdl(rmsnorm_quant_reg_kernel<1>, grid, NORM_THREADS, pdl, s, x, delta, gamma, eps, K, h_out, out);
    case 2: return launch_pdl(rmsnorm_quant_reg_kernel<2>, grid, NORM_THREADS, pdl, s, x, delta, gamma, eps, K, h_out, out);
    case 4: return launch_pdl(rmsnorm_quant_reg_kernel<4>, grid, NORM_THREADS, pdl, s, x, delta, gamma, eps, K, h_out, out);
    case 8: return launch_pdl(rmsnorm_quant_reg_kernel<8>, grid, NORM_THREADS, pdl, s, x, delta, gamma, eps, K, h_out, out);
    default:  // K > 8192: thread segments, h read again in pass 2
      return launch_pdl(rmsnorm_quant_kernel, grid, NORM_THREADS, pdl, s, x, delta, gamma, eps, K, h_out, out);
  }
}

cudaError_t launch_swiglu_quantize(const float* gu, int64_t M, int64_t F, uint8_t* out, int sm_count,
                                   bool pdl, cudaStream_t s) {
  const int64_t nbr = F / QK;
  const int64_t total = M * nbr;
  const int64_t per_cta = SWIGLU_THREADS / 8 * SWIGLU_B;
  int64_t grid = (total + per_cta - 1) / per_cta;
  const int64_t cap = (int64_t)sm_count * 16;
  if (grid > cap) grid = cap;
  // 32-bit indices while every index stays below 2^32 (b0 + ngrp included)
  if (total + grid * per_cta < ((int64_t)1 << 32))
    return launch_pdl(swiglu_quant_kernel<uint32_t>, dim3((unsigned)grid), SWIGLU_THREADS, pdl, s, gu, F,
                      (uint32_t)nbr, (uint32_t)total, out);
  return launch_pdl(swiglu_quant_kernel<int64_t>, dim3((unsigned)grid), SWIGLU_THREADS, pdl, s, gu, F, nbr,
                    total, out);
}

}  // namespace q8
