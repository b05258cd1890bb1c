// q8_internal.h -- host-side launch helpers shared between the libq8
// translation units (not part of the C ABI).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace q8 {

// Launch plan of one GEMV call: the work is cut into units of one R-row
// tile x RU rounds of P = 128 / R chunks (8 blocks each), S units per tile
// along K.
struct GemvPlan {
  int64_t N = 0, K = 0, NB = 0;
  int M = 0;
  int MT = 0;        // activation rows per kernel instantiation (1,2,4,8,16)
  int R = 0;         // packed tile height
  int T = 0;         // row tiles
  int nch = 0;       // chunks along K
  int RU = 0;        // rounds per unit
  int S = 0;         // units per tile (splits along K)
  int units = 0;
  int grid = 0;      // persistent CTAs
  int cluster = 1;   // CTAs per thread-block cluster (shared activation staging)
  bool u5 = false;   // block dots on the tcgen05 tensor cores (128-row tiles, 16 rows per pass)
  size_t smem = 0;   // dynamic shared memory per CTA
  size_t ws_bytes = 0;
  // 4-32 rows per pass: the virtual-tile kernel (q8_gemv_vt.cuh): units of
  // TV virtual tiles of 128 rows x RU chunks, UB staged blocks per unit,
  // partials [S][rows][Np] when split along K
  bool vt = false;
  int TV = 0, UB = 0, Np = 0;
  bool img = false;  // the activations are staged once per call into the workspace (16+ rows per pass)
};

struct DeviceInfo {
  int device = -1;
  int sm_count = 0;
  int cc_major = 0, cc_minor = 0;
};

cudaError_t current_device_info(DeviceInfo* out);
// allow_vt = false keeps every row count on the one-tile-per-unit kernel
// (the SwiGLU epilogue exists only there); allow_image = false plans the
// virtual-tile kernel without the staged activation images (less workspace).
bool plan_gemv(const DeviceInfo& dev, int64_t N, int64_t K, int M, bool fused, bool tcgen05, GemvPlan* p,
               bool allow_vt = true, bool allow_image = true);
bool plan_vt(const DeviceInfo& dev, int64_t N, int64_t K, int M, bool fused, bool image, GemvPlan* p);
cudaError_t launch_vt(const GemvPlan& p, const uint8_t* W, const uint8_t* A, const float* x, uint8_t* A_out,
                      float* y, void* workspace, bool pdl, cudaStream_t s);

// Kernel launchers (q8_aux.cu / q8_gemv.cu).  Each returns the CUDA error of
// the launch.  `pdl` launches with programmatic stream serialization.
cudaError_t launch_quantize(const float* x, int64_t M, int64_t K, uint8_t* out, bool pdl,
                            cudaStream_t s);
cudaError_t launch_repack(const uint8_t* src, int64_t N, int64_t K, uint8_t* dst, cudaStream_t s);
cudaError_t launch_unpack(const uint8_t* packed, int64_t N, int64_t K, uint8_t* dst,
                          cudaStream_t s);
cudaError_t launch_block_dots(const uint8_t* W, int64_t N, int64_t K, const uint8_t* A, int M,
                              int32_t* isum, cudaStream_t s);
// h_blocks non-null: the SwiGLU epilogue writes blocks of silu(gate) * up
// there instead of y (the plan must not split K; tiles of 64 or 128 rows).
cudaError_t launch_gemv(const GemvPlan& p, const uint8_t* W, const uint8_t* A, const float* x,
                        uint8_t* A_out, float* y, void* workspace, bool pdl, cudaStream_t s,
                        uint8_t* h_blocks = nullptr);
cudaError_t read_and_clear_gemv_error(unsigned* code);
// Limit of the GEMV kernels' ring waits for launches from now on (a test
// hook: 0 restores the default of 2 s).
void set_gemv_wait_limit_ns(uint64_t ns);
uint64_t gemv_wait_limit_ns();
// The device word the kernels set bits in when a bounded wait gives up.
cudaError_t device_error_word(int dev, unsigned** out);

// Prefill tile GEMM (q8_prefill.cu): activation blocks [M][K/32] are packed
// into 128-row tiles (the weights' packed layout with R = 128), then every
// 128 x 128 output tile is one CTA's work.
// (zero, nzero: words cleared before the packing, for the prefill GEMM's split flags)
cudaError_t launch_pack_act(const uint8_t* src, int64_t M, int64_t K, uint8_t* dst, bool pdl, cudaStream_t s,
                            unsigned* zero = nullptr, int nzero = 0);
// flags: PREFILL_FLAG_BYTES of split flags, cleared by the pack launch before it
constexpr size_t PREFILL_FLAG_BYTES = 4096;
cudaError_t launch_prefill(const DeviceInfo& dev, const uint8_t* W, int64_t N, int64_t K, const uint8_t* A_packed,
                           int64_t M, float* y, unsigned* flags, bool pdl, cudaStream_t s);
// whether launch_prefill splits this shape along K (its pack launch clears the flags first)
bool prefill_splits(const DeviceInfo& dev, int64_t N, int64_t K, int64_t M);

// Int8 KV cache codec (q8_kv.cu).  A row whose slot lies outside [0,
// capacity) is skipped (the dequantized row is written as zeros) and sets
// ERR_KV_SLOT in the device error word.
constexpr unsigned ERR_KV_SLOT = 8u;
cudaError_t launch_kv_quantize(const float* x, int64_t rows, int64_t D, const int32_t* slots, int64_t capacity,
                               int8_t* cq, float* cd, int sm_count, bool pdl, cudaStream_t s);
cudaError_t launch_kv_dequantize(const int8_t* cq, const float* cd, int64_t capacity, int64_t D,
                                 const int32_t* slots, int64_t rows, float* out, int sm_count, bool pdl,
                                 cudaStream_t s);

// Fused producers (q8_producers.cu).
cudaError_t launch_rmsnorm_quantize(const float* x, const float* delta, const float* gamma, float eps,
                                    int64_t M, int64_t K, float* h_out, uint8_t* out, bool pdl,
                                    cudaStream_t s);
cudaError_t launch_swiglu_quantize(const float* gu, int64_t M, int64_t F, uint8_t* out, int sm_count,
                                   bool pdl, cudaStream_t s);

}  // namespace q8
