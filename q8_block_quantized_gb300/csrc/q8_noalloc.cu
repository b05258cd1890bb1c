// q8_noalloc.cu -- q8_gemm_noalloc: the GEMV for callers that cannot
// allocate device memory.
//
// Who needs this: code that runs where device allocation is not allowed or
// not safe -- for example a plugin inside a host application whose own
// memory manager owns the whole device, or a latency-critical loop that must
// not pay cudaMalloc's unpredictable latency and implicit device
// synchronization.  q8_gemm asks its caller for a workspace whenever it
// splits the work along K; this entry point instead uses a fixed scratch
// area compiled into the library, so neither the caller nor the library
// allocates anything.
//
// The scratch is one file-scope device array.  Every GPU that loads the
// library holds it until the process exits.  All calls share it and it keeps
// the last call's contents, so calls that may run at the same time on the
// GPU (different streams, or different host threads) race on it.  Its first
// 16 KB are per-tile tickets that must be zero when a split call starts;
// every completed call leaves them zero, and this entry point also clears
// them (an asynchronous memset on the caller's stream, not an allocation)
// before each split launch.
#include <cuda_runtime.h>

#include <mutex>

#include "q8.h"
#include "q8_device.cuh"
#include "q8_gemv_impl.cuh"
#include "q8_internal.h"

namespace {

constexpr size_t NOALLOC_BYTES = Q8_NOALLOC_SCRATCH_BYTES;

// The scratch area.  In host code this name is only a stand-in for the
// symbol: the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char q8_noalloc_scratch[NOALLOC_BYTES];

constexpr int MAX_DEVICES = 64;
std::mutex g_mu;
void* g_scratch_ptr[MAX_DEVICES] = {};

// Device address of the scratch array on the current device, looked up once
// per device (with that device current) and cached.
cudaError_t scratch_address(int dev, void** out) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, q8_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" int q8_gemm_noalloc(const void* W, int64_t N, int64_t K, const void* A_blocks, int M,
                               float* y, unsigned flags, void* stream) {
  using namespace q8;
  if (W == nullptr || A_blocks == nullptr || y == nullptr) return Q8_EINVAL;
  if ((flags & ~Q8_FLAG_PDL) != 0) return Q8_EINVAL;
  if (N <= 0 || N > INT32_MAX || K <= 0 || (K % QK) != 0 || K / QK > ((int64_t)1 << 30) || M < 1 ||
      M > Q8_MAX_M)
    return Q8_ESHAPE;
  if (!aligned(W, 16) || !aligned(A_blocks, 2) || !aligned(y, 4)) return Q8_EALIGN;
  DeviceInfo d;
  if (current_device_info(&d) != cudaSuccess) return Q8_ECUDA;
  if (d.cc_major != 10 || d.cc_minor != 3) return Q8_EDEVICE;
  if (d.device < 0 || d.device >= MAX_DEVICES) return Q8_EDEVICE;
  GemvPlan p;
  if (!plan_gemv(d, N, K, M, false, false, &p)) return Q8_ESHAPE;
  // without the staged activation images if those do not fit (the bits are the same)
  if (p.ws_bytes > NOALLOC_BYTES && p.img && !plan_gemv(d, N, K, M, false, false, &p, true, false))
    return Q8_ESHAPE;
  if (p.ws_bytes > NOALLOC_BYTES) return Q8_ESCRATCH;  // this shape needs more scratch than built in
  void* ws = nullptr;
  if (p.ws_bytes > 0) {
    if (scratch_address(d.device, &ws) != cudaSuccess) return Q8_ECUDA;
    // tickets must start at zero (a call that was abandoned could leave them set)
    if (cudaMemsetAsync(ws, 0, TICKET_BYTES, static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return Q8_ECUDA;
  }
  const cudaError_t e = launch_gemv(p, static_cast<const uint8_t*>(W),
                                    static_cast<const uint8_t*>(A_blocks), nullptr, nullptr, y, ws,
                                    (flags & Q8_FLAG_PDL) != 0, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? Q8_OK : Q8_ECUDA;
}
