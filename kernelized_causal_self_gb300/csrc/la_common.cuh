// Shared device helpers for the linear-attention kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "la.h"

namespace la {

// phi(x) = elu(x) + 1 with alpha = 1 ("Transformers are RNNs", §3.2.1 of the
// paperlayer.ai summary; slide 3 of the zhengyuhong.cn deck).
__device__ __forceinline__ float phi(float x) { return x > 0.f ? x + 1.f : expf(x); }

// phi'(x) = 1 for x > 0, exp(x) = phi(x) for x <= 0; so phi'(x) = min(phi(x), 1).
__device__ __forceinline__ float phi_grad_from_phi(float p) { return fminf(p, 1.f); }

template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// Workspace header: the first 256 bytes of every workspace.
struct WorkspaceHeader {
  int status;     // LA_OK, LA_ERR_TIMEOUT (a bounded wait gave up) or LA_ERR_INVALID_ARG
                  // (la_extend met a slot outside its pool), written by kernels
  int wait_site;  // where a bounded wait gave up (debug)
  int tickets[2];  // items handed out so far (per-stream lengths: segment states, attention)
  unsigned int pad[60];
};
static_assert(sizeof(WorkspaceHeader) == 256, "header must stay 256 bytes");

constexpr size_t kHeaderBytes = 256;

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace la
