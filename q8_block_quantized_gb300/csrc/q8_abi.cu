// q8_abi.cu -- the extern "C" entry points of libq8 (declared in q8.h):
// host-side argument checks, device checks, launch planning, launches.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "q8.h"
#include "q8_device.cuh"
#include "q8_internal.h"

namespace q8 {

namespace {
constexpr int MAX_DEVICES = 64;
std::mutex g_dev_mu;
DeviceInfo g_dev_cache[MAX_DEVICES];
bool g_dev_known[MAX_DEVICES] = {};
}  // namespace

cudaError_t current_device_info(DeviceInfo* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= MAX_DEVICES) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (!g_dev_known[dev]) {
    DeviceInfo d;
    d.device = dev;
    if ((e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess) return e;
    g_dev_cache[dev] = d;
    g_dev_known[dev] = true;
  }
  *out = g_dev_cache[dev];
  return cudaSuccess;
}

}  // namespace q8

using namespace q8;

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool k_ok(int64_t K) { return K > 0 && (K % QK) == 0 && K / QK <= ((int64_t)1 << 30); }

// Shared device check: sm_103 only.
int device_ok(DeviceInfo* d) {
  if (current_device_info(d) != cudaSuccess) return Q8_ECUDA;
  if (d->cc_major != 10 || d->cc_minor != 3) return Q8_EDEVICE;
  return Q8_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? Q8_OK : Q8_ECUDA; }

int check_gemm_common(const void* W, int64_t N, int64_t K, int M, const float* y, unsigned flags) {
  if (W == nullptr || y == nullptr) return Q8_EINVAL;
  if ((flags & ~(Q8_FLAG_PDL | Q8_FLAG_TCGEN05)) != 0) return Q8_EINVAL;
  if (N <= 0 || N > INT32_MAX || !k_ok(K) || M < 1 || M > Q8_MAX_M) return Q8_ESHAPE;
  if (!aligned(W, 16) || !aligned(y, 4)) return Q8_EALIGN;
  return Q8_OK;
}

int check_workspace(const GemvPlan& p, void* ws, size_t ws_bytes) {
  if (p.ws_bytes == 0) return Q8_OK;
  if (ws == nullptr || ws_bytes < p.ws_bytes) return Q8_EWORKSPACE;
  if (!aligned(ws, 16)) return Q8_EALIGN;
  return Q8_OK;
}

// The SwiGLU epilogue's extra conditions: 64- or 128-row tiles holding whole
// gate/up groups, and no split along K (checked on the plan).
int swiglu_gemm(const void* W, int64_t F, int64_t K, const void* A_blocks, const float* x, int M,
                void* out_blocks, void* workspace, size_t workspace_bytes, unsigned flags, void* stream) {
  if (W == nullptr || out_blocks == nullptr || (A_blocks == nullptr && x == nullptr)) return Q8_EINVAL;
  if ((flags & ~Q8_FLAG_PDL) != 0) return Q8_EINVAL;
  if (F <= 0 || F > INT32_MAX / 2 || !k_ok(K) || M < 1 || M > Q8_MAX_M) return Q8_ESHAPE;
  const int R = layout_tile_rows(2 * F);
  if ((R != 64 && R != 128) || F % (R / 2) != 0) return Q8_ESHAPE;
  if (!aligned(W, 16) || !aligned(out_blocks, 2)) return Q8_EALIGN;
  if ((A_blocks != nullptr && !aligned(A_blocks, 2)) || (x != nullptr && !aligned(x, 16))) return Q8_EALIGN;
  DeviceInfo d;
  int st = device_ok(&d);
  if (st != Q8_OK) return st;
  GemvPlan p;
  if (!plan_gemv(d, 2 * F, K, M, x != nullptr, false, &p, false) || p.S != 1) return Q8_ESHAPE;
  (void)workspace;
  (void)workspace_bytes;  // no split along K: no workspace is used
  return cuda_status(launch_gemv(p, static_cast<const uint8_t*>(W), static_cast<const uint8_t*>(A_blocks), x,
                                 nullptr, nullptr, nullptr, (flags & Q8_FLAG_PDL) != 0,
                                 static_cast<cudaStream_t>(stream), static_cast<uint8_t*>(out_blocks)));
}

// Packed activations of the prefill GEMM: the blocks' bytes, to 16 bytes.
size_t prefill_packed_bytes(int64_t K, int64_t M) {
  return ((size_t)M * (size_t)(K / QK) * BLOCK_BYTES + 15) & ~(size_t)15;
}

int prefill_gemm(const void* W, int64_t N, int64_t K, const void* A_blocks, const float* x, int M, float* y,
                 void* A_out, void* workspace, size_t workspace_bytes, unsigned flags, void* stream) {
  if (W == nullptr || y == nullptr || (A_blocks == nullptr && x == nullptr)) return Q8_EINVAL;
  if ((flags & ~Q8_FLAG_PDL) != 0) return Q8_EINVAL;
  if (N <= 0 || N > INT32_MAX || !k_ok(K) || K > Q8_MAX_PREFILL_K || M < 1) return Q8_ESHAPE;
  const int64_t T = Q8_PREFILL_TILE_ROWS;
  if (((N + T - 1) / T) * (((int64_t)M + T - 1) / T) > INT32_MAX) return Q8_ESHAPE;  // output tiles
  if (!aligned(W, 16) || !aligned(y, 4)) return Q8_EALIGN;
  if ((A_blocks != nullptr && !aligned(A_blocks, 2)) || (x != nullptr && !aligned(x, 4)) ||
      (A_out != nullptr && !aligned(A_out, 2)))
    return Q8_EALIGN;
  const size_t pk = prefill_packed_bytes(K, M);
  // workspace: the split flags, the packed activations, the blocks of x
  const size_t need = PREFILL_FLAG_BYTES + ((x != nullptr && A_out == nullptr) ? 2 * pk : pk);
  if (workspace == nullptr || workspace_bytes < need) return Q8_EWORKSPACE;
  if (!aligned(workspace, 16)) return Q8_EALIGN;
  DeviceInfo d;
  int st = device_ok(&d);
  if (st != Q8_OK) return st;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  bool pdl = (flags & Q8_FLAG_PDL) != 0;
  unsigned* split_flags = static_cast<unsigned*>(workspace);
  uint8_t* packed = static_cast<uint8_t*>(workspace) + PREFILL_FLAG_BYTES;
  const uint8_t* blocks = static_cast<const uint8_t*>(A_blocks);
  cudaError_t e;
  if (x != nullptr) {
    uint8_t* out = A_out != nullptr ? static_cast<uint8_t*>(A_out) : packed + pk;
    if ((e = launch_quantize(x, M, K, out, pdl, s)) != cudaSuccess) return Q8_ECUDA;
    blocks = out;
    pdl = true;  // the next launches depend on this library's own launch
  }
  const int nflags = prefill_splits(d, N, K, M) ? (int)(PREFILL_FLAG_BYTES / 4) : 0;
  if ((e = launch_pack_act(blocks, M, K, packed, pdl, s, split_flags, nflags)) != cudaSuccess) return Q8_ECUDA;
  return cuda_status(launch_prefill(d, static_cast<const uint8_t*>(W), N, K, packed, M, y, split_flags, true, s));
}

}  // namespace

extern "C" {

const char* q8_strerror(int status) {
  switch (status) {
    case Q8_OK: return "Q8_OK";
    case Q8_EINVAL: return "Q8_EINVAL: null pointer or bad flag";
    case Q8_ESHAPE: return "Q8_ESHAPE: shape out of range (K must be a positive multiple of 32)";
    case Q8_EALIGN: return "Q8_EALIGN: pointer not aligned as documented";
    case Q8_EDEVICE: return "Q8_EDEVICE: current device is not sm_103";
    case Q8_ECUDA: return "Q8_ECUDA: a CUDA runtime call failed";
    case Q8_EWORKSPACE: return "Q8_EWORKSPACE: workspace missing or too small";
    case Q8_ETIMEOUT: return "Q8_ETIMEOUT: a device-side wait gave up";
    case Q8_ESCRATCH: return "Q8_ESCRATCH: shape needs more than the built-in no-allocation scratch";
    default: return "unknown q8 status";
  }
}

int q8_abi_version(void) { return 1; }

size_t q8_blocks_bytes(int64_t rows, int64_t K) {
  if (rows <= 0 || !k_ok(K)) return 0;
  return (size_t)rows * (size_t)(K / QK) * BLOCK_BYTES;
}

size_t q8_packed_bytes(int64_t N, int64_t K) { return q8_blocks_bytes(N, K); }

int q8_packed_tile_rows(int64_t N) { return N > 0 ? layout_tile_rows(N) : 0; }

size_t q8_prefill_workspace_bytes(int64_t K, int M) {
  if (!k_ok(K) || K > Q8_MAX_PREFILL_K || M < 1) return 0;
  return PREFILL_FLAG_BYTES + 2 * prefill_packed_bytes(K, M);
}

int q8_gemm_prefill(const void* W, int64_t N, int64_t K, const void* A_blocks, int M, float* y, void* workspace,
                    size_t workspace_bytes, unsigned flags, void* stream) {
  if (A_blocks == nullptr) return Q8_EINVAL;
  return prefill_gemm(W, N, K, A_blocks, nullptr, M, y, nullptr, workspace, workspace_bytes, flags, stream);
}

int q8_fused_quant_gemm_prefill(const void* W, int64_t N, int64_t K, const float* x, int M, float* y,
                                void* A_blocks_out, void* workspace, size_t workspace_bytes, unsigned flags,
                                void* stream) {
  if (x == nullptr) return Q8_EINVAL;
  return prefill_gemm(W, N, K, nullptr, x, M, y, A_blocks_out, workspace, workspace_bytes, flags, stream);
}

size_t q8_workspace_bytes(int64_t N, int64_t K, int M) {
  if (N <= 0 || N > INT32_MAX || !k_ok(K) || M < 1 || M > Q8_MAX_M) return 0;
  DeviceInfo d;
  if (device_ok(&d) != Q8_OK) return 0;
  // the largest need over the kernel variants a call may pick
  size_t most = 0;
  for (int v = 0; v < 4; ++v) {
    GemvPlan p;
    if (!plan_gemv(d, N, K, M, (v & 1) != 0, (v & 2) != 0, &p)) return 0;
    if (p.ws_bytes > most) most = p.ws_bytes;
  }
  return most;
}

int q8_quantize_act(const float* x, int64_t M, int64_t K, void* out_blocks, unsigned flags,
                    void* stream) {
  if (x == nullptr || out_blocks == nullptr || (flags & ~Q8_FLAG_PDL) != 0) return Q8_EINVAL;
  if (M <= 0 || M > INT32_MAX || !k_ok(K)) return Q8_ESHAPE;
  if (!aligned(x, 4) || !aligned(out_blocks, 2)) return Q8_EALIGN;
  DeviceInfo d;
  int st = device_ok(&d);
  if (st != Q8_OK) return st;
  return cuda_status(launch_quantize(x, M, K, static_cast<uint8_t*>(out_blocks),
                                     (flags & Q8_FLAG_PDL) != 0, static_cast<cudaStream_t>(stream)));
}

int q8_repack_weights(const void* src_blocks, int64_t N, int64_t K, void* dst, void* stream) {
  if (src_blocks == nullptr || dst == nullptr) return Q8_EINVAL;
  if (N <= 0 || N > INT32_MAX || !k_ok(K)) return Q8_ESHAPE;
  if (!aligned(src_blocks, 2) || !aligned(dst, 16)) return Q8_EALIGN;
  DeviceInfo d;
  int st = device_ok(&d);
  if (st != Q8_OK) return st;
  return cuda_status(launch_repack(static_cast<const uint8_t*>(src_blocks), N, K,
                                   static_cast<uint8_t*>(dst), static_cast<cudaStream_t>(stream)));
}

int q8_unpack_weights(const void* packed, int64_t N, int64_t K, void* dst_blocks, void* stream) {
  if (packed == nullptr || dst_blocks == nullptr) return Q8_EINVAL;
  if (N <= 0 || N > INT32_MAX || !k_ok(K)) return Q8_ESHAPE;
  if (!aligned(packed, 16) || !aligned(dst_blocks, 2)) return Q8_EALIGN;
  DeviceInfo d;
  int st = device_ok(&d);
  if (st != Q8_OK) return st;
  return cuda_status(launch_unpack(static_cast<const uint8_t*>(packed), N, K,
                                   static_cast<uint8_t*>(dst_blocks), static_cast<cudaStream_t>(stream)));
}

int q8_gemm(const void* W, int64_t N, int64_t K, const void* A_blocks, int M, float* y,
            void* workspace, size_t workspace_bytes, unsigned flags, void* stream) {
  if (A_blocks == nullptr) return Q8_EINVAL;
  int st = check_gemm_common(W, N, K, M, y, flags);
  if (st != Q8_OK) return st;
  if (!aligned(A_blocks, 2)) return Q8_EALIGN;
  DeviceInfo d;
  if ((st = device_ok(&d)) != Q8_OK) return st;
  GemvPlan p;
  if (!plan_gemv(d, N, K, M, false, (flags & Q8_FLAG_TCGEN05) != 0, &p)) return Q8_ESHAPE;
  if ((st = check_workspace(p, workspace, workspace_bytes)) != Q8_OK) return st;
  return cuda_status(launch_gemv(p, static_cast<const uint8_t*>(W), static_cast<const uint8_t*>(A_blocks),
                                 nullptr, nullptr, y, workspace, (flags & Q8_FLAG_PDL) != 0,
                                 static_cast<cudaStream_t>(stream)));
}

int q8_fused_quant_gemm(const void* W, int64_t N, int64_t K, const float* x, int M, float* y,
                        void* A_blocks_out, void* workspace, size_t workspace_bytes, unsigned flags,
                        void* stream) {
  if (x == nullptr) return Q8_EINVAL;
  int st = check_gemm_common(W, N, K, M, y, flags);
  if (st != Q8_OK) return st;
  if (!aligned(x, 16) || (A_blocks_out != nullptr && !aligned(A_blocks_out, 2))) return Q8_EALIGN;
  DeviceInfo d;
  if ((st = device_ok(&d)) != Q8_OK) return st;
  GemvPlan p;
  if (!plan_gemv(d, N, K, M, true, (flags & Q8_FLAG_TCGEN05) != 0, &p)) return Q8_ESHAPE;
  if ((st = check_workspace(p, workspace, workspace_bytes)) != Q8_OK) return st;
  return cuda_status(launch_gemv(p, static_cast<const uint8_t*>(W), nullptr, x,
                                 static_cast<uint8_t*>(A_blocks_out), y, workspace,
                                 (flags & Q8_FLAG_PDL) != 0, static_cast<cudaStream_t>(stream)));
}

int q8_residual_rmsnorm_quantize(const float* x, const float* delta, const float* gamma, float eps,
                                 int64_t M, int64_t K, float* h_out, void* out_blocks, unsigned flags,
                                 void* stream) {
  if (x == nullptr || gamma == nullptr || out_blocks == nullptr || (flags & ~Q8_FLAG_PDL) != 0)
    return Q8_EINVAL;
  if (!(eps > 0.0f) || !(eps <= 3.0e38f)) return Q8_EINVAL;  // positive and finite (NaN fails)
  if (M <= 0 || M > INT32_MAX || !k_ok(K) || K > Q8_MAX_NORM_K) return Q8_ESHAPE;
  if (!aligned(x, 16) || !aligned(gamma, 16) || (delta != nullptr && !aligned(delta, 16)) ||
      (h_out != nullptr && !aligned(h_out, 16)) || !aligned(out_blocks, 2))
    return Q8_EALIGN;
  DeviceInfo d;
  int st = device_ok(&d);
  if (st != Q8_OK) return st;
  return cuda_status(launch_rmsnorm_quantize(x, delta, gamma, eps, M, K, h_out,
                                             static_cast<uint8_t*>(out_blocks), (flags & Q8_FLAG_PDL) != 0,
                                             static_cast<cudaStream_t>(stream)));
}

int q8_swiglu_quantize(const float* gate_up, int64_t M, int64_t F, void* out_blocks, unsigned flags,
                       void* stream) {
  if (gate_up == nullptr || out_blocks == nullptr || (flags & ~Q8_FLAG_PDL) != 0) return Q8_EINVAL;
  if (M <= 0 || M > INT32_MAX || !k_ok(F) || F > ((int64_t)1 << 30)) return Q8_ESHAPE;
  if (!aligned(gate_up, 16) || !aligned(out_blocks, 2)) return Q8_EALIGN;
  DeviceInfo d;
  int st = device_ok(&d);
  if (st != Q8_OK) return st;
  return cuda_status(launch_swiglu_quantize(gate_up, M, F, static_cast<uint8_t*>(out_blocks), d.sm_count,
                                            (flags & Q8_FLAG_PDL) != 0, static_cast<cudaStream_t>(stream)));
}

int q8_gemm_swiglu(const void* W, int64_t F, int64_t K, const void* A_blocks, int M, void* out_blocks,
                   unsigned flags, void* stream) {
  if (A_blocks == nullptr) return Q8_EINVAL;
  return swiglu_gemm(W, F, K, A_blocks, nullptr, M, out_blocks, nullptr, 0, flags, stream);
}

int q8_fused_quant_gemm_swiglu(const void* W, int64_t F, int64_t K, const float* x, int M, void* out_blocks,
                               unsigned flags, void* stream) {
  if (x == nullptr) return Q8_EINVAL;
  return swiglu_gemm(W, F, K, nullptr, x, M, out_blocks, nullptr, 0, flags, stream);
}


size_t q8_kv_cache_bytes(int64_t capacity, int64_t D) {
  if (capacity <= 0 || capacity > INT32_MAX || !k_ok(D) || D > Q8_MAX_KV_D) return 0;
  return (size_t)capacity * (size_t)(D / QK) * (QK + 4);
}

int q8_kv_quantize(const float* x, int64_t rows, int64_t D, const int32_t* slots, int64_t capacity,
                   int8_t* cache_q, float* cache_d, unsigned flags, void* stream) {
  if (x == nullptr || cache_q == nullptr || cache_d == nullptr || (flags & ~Q8_FLAG_PDL) != 0) return Q8_EINVAL;
  if (rows <= 0 || rows > INT32_MAX || capacity <= 0 || capacity > INT32_MAX || !k_ok(D) || D > Q8_MAX_KV_D)
    return Q8_ESHAPE;
  if (!aligned(x, 16) || !aligned(cache_q, 4) || !aligned(cache_d, 4) || (slots != nullptr && !aligned(slots, 4)))
    return Q8_EALIGN;
  DeviceInfo d;
  int st = device_ok(&d);
  if (st != Q8_OK) return st;
  return cuda_status(launch_kv_quantize(x, rows, D, slots, capacity, cache_q, cache_d, d.sm_count,
                                        (flags & Q8_FLAG_PDL) != 0, static_cast<cudaStream_t>(stream)));
}

int q8_kv_dequantize(const int8_t* cache_q, const float* cache_d, int64_t capacity, int64_t D, const int32_t* slots,
                     int64_t rows, float* out, unsigned flags, void* stream) {
  if (cache_q == nullptr || cache_d == nullptr || out == nullptr || (flags & ~Q8_FLAG_PDL) != 0) return Q8_EINVAL;
  if (rows <= 0 || rows > INT32_MAX || capacity <= 0 || capacity > INT32_MAX || !k_ok(D) || D > Q8_MAX_KV_D)
    return Q8_ESHAPE;
  if (!aligned(out, 16) || !aligned(cache_q, 4) || !aligned(cache_d, 4) || (slots != nullptr && !aligned(slots, 4)))
    return Q8_EALIGN;
  DeviceInfo d;
  int st = device_ok(&d);
  if (st != Q8_OK) return st;
  return cuda_status(launch_kv_dequantize(cache_q, cache_d, capacity, D, slots, rows, out, d.sm_count,
                                          (flags & Q8_FLAG_PDL) != 0, static_cast<cudaStream_t>(stream)));
}

int q8_block_dots(const void* W, int64_t N, int64_t K, const void* A_blocks, int M, int32_t* isum,
                  void* stream) {
  if (W == nullptr || A_blocks == nullptr || isum == nullptr) return Q8_EINVAL;
  if (N <= 0 || N > INT32_MAX || !k_ok(K) || M < 1 || M > Q8_MAX_DOTS_M) return Q8_ESHAPE;
  if (!aligned(W, 16) || !aligned(A_blocks, 2) || !aligned(isum, 4)) return Q8_EALIGN;
  DeviceInfo d;
  int st = device_ok(&d);
  if (st != Q8_OK) return st;
  return cuda_status(launch_block_dots(static_cast<const uint8_t*>(W), N, K,
                                       static_cast<const uint8_t*>(A_blocks), M, isum,
                                       static_cast<cudaStream_t>(stream)));
}

int q8_device_error(unsigned* code) {
  if (code == nullptr) return Q8_EINVAL;
  DeviceInfo d;
  int st = device_ok(&d);
  if (st != Q8_OK) return st;
  if (cudaDeviceSynchronize() != cudaSuccess) return Q8_ECUDA;
  unsigned v = 0;
  if (read_and_clear_gemv_error(&v) != cudaSuccess) return Q8_ECUDA;
  // a failed wait outranks a skipped KV row in the status byte; the bits say which
  const int status = (v & ~ERR_KV_SLOT) != 0 ? Q8_ETIMEOUT : Q8_ESHAPE;
  *code = v ? ((unsigned)(-status) << 8) | v : 0u;
  return Q8_OK;
}

int q8_set_wait_limit_ns(uint64_t ns) {
  set_gemv_wait_limit_ns(ns);
  return Q8_OK;
}

int q8_device_info(int* sm_count, int* cc_major, int* cc_minor) {
  DeviceInfo d;
  if (current_device_info(&d) != cudaSuccess) return Q8_ECUDA;
  if (sm_count) *sm_count = d.sm_count;
  if (cc_major) *cc_major = d.cc_major;
  if (cc_minor) *cc_minor = d.cc_minor;
  return Q8_OK;
}

}  // extern "C"
