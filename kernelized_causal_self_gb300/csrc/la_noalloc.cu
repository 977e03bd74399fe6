// la_forward_noalloc: la_forward with its scratch in a fixed device array.
//
// For callers that cannot allocate device memory themselves (they are handed
// device pointers for inputs and outputs by an application or framework that
// owns the allocator, or they run where cudaMalloc is not permitted). The
// array below is the whole scratch; nothing is allocated or freed here.
#include <stddef.h>

#include <mutex>

#include "la_common.cuh"

namespace {

constexpr size_t kScratchBytes = LA_NOALLOC_SCRATCH_BYTES;

// One copy per device that loads the library, held until the process exits.
// In host code this name is only a host-side handle for the symbol, never a
// device address: the address is looked up per device below.
__device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the array on the current device; looked up once per
// device, with that device current.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" int la_forward_noalloc(const void* q, const void* k, const void* v, void* out, int B,
                                  int H, int N, int D, int M, int causal, int dtype,
                                  void* stream) {
  const size_t need = la_forward_workspace_bytes(B, H, N, D, M, causal, dtype);
  if (need > kScratchBytes) return LA_ERR_TOO_LARGE;
  // argument errors are reported by la_forward itself before anything runs;
  // resolve the scratch only for calls that will launch work
  if (N <= 0 || B < 1 || H < 1)
    return la_forward(q, k, v, out, B, H, N, D, M, causal, dtype, nullptr, 0, stream);
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return LA_ERR_CUDA;
  return la_forward(q, k, v, out, B, H, N, D, M, causal, dtype, scratch, kScratchBytes, stream);
}

extern "C" int la_forward_noalloc_status(void* stream) {
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return LA_ERR_CUDA;
  return la_workspace_status(scratch, kScratchBytes, stream);
}

extern "C" int la_debug_noalloc_set_status(int status, int wait_site, void* stream) {
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return LA_ERR_CUDA;
  static_assert(offsetof(la::WorkspaceHeader, status) == 0, "status word first");
  static_assert(offsetof(la::WorkspaceHeader, wait_site) == sizeof(int), "wait site second");
  const int word[2] = {status, wait_site};
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(scratch, word, sizeof(word), cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  return e == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}
