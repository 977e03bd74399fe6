// Recurrent decode step: one CTA per (stream, head).
//
// "Transformers are RNNs" deck, slide 4, and paperlayer.ai summary §3.3.2/§3.4:
// generation keeps the attention memory S (D x M) and normalizer memory Z (D)
// and, per new token, first adds it (S += phi(k) v^T, Z += phi(k)) and then
// reads out phi(q)^T S / phi(q)^T Z.
//
// The step is bound by the S read + write (2 * D * M * 4 bytes per stream-head
// against 4 * D * M flops), so the kernel is a streaming update: each thread
// owns one float4 column group of S and walks a strided set of rows with
// 128-bit loads and stores, folding the read-out phi(q)^T S into the same pass.
#include "la_common.cuh"
#include "la_internal.h"

namespace la {
namespace {

constexpr int kDecodeThreads = 128;

template <typename T>
__global__ void __launch_bounds__(kDecodeThreads)
decode_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
              float* __restrict__ S, float* __restrict__ Z, T* __restrict__ out, int D, int M) {
  __shared__ float fq[128], fk[128], vs[128];
  __shared__ float red[kDecodeThreads * 4];
  __shared__ float den_part[kDecodeThreads / 32];

  const size_t sh = blockIdx.x;
  const int tid = threadIdx.x;
  if (tid < D) {
    fq[tid] = phi(to_f32<T>(q[sh * D + tid]));
    fk[tid] = phi(to_f32<T>(k[sh * D + tid]));
  }
  if (tid < M) vs[tid] = to_f32<T>(v[sh * M + tid]);
  __syncthreads();

  // Z update and the denominator phi(q) . Z_new
  float dpart = 0.f;
  if (tid < D) {
    const float z = Z[sh * D + tid] + fk[tid];
    Z[sh * D + tid] = z;
    dpart = fq[tid] * z;
  }
  for (int o = 16; o > 0; o >>= 1) dpart += __shfl_xor_sync(0xffffffffu, dpart, o);
  if ((tid & 31) == 0) den_part[tid >> 5] = dpart;

  // S update and numerator, 128-bit accesses
  const int cg = M >> 2;                 // float4 column groups
  const int rgs = kDecodeThreads / cg;   // row groups
  const int my_cg = tid % cg, my_rg = tid / cg;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (my_rg < rgs) {
    float4* S4 = reinterpret_cast<float4*>(S + sh * (size_t)D * M);
    const float4 v4 = make_float4(vs[4 * my_cg], vs[4 * my_cg + 1], vs[4 * my_cg + 2],
                                  vs[4 * my_cg + 3]);
#pragma unroll 4
    for (int d = my_rg; d < D; d += rgs) {
      float4 s = S4[d * cg + my_cg];
      const float a = fk[d], b = fq[d];
      s.x += a * v4.x;
      s.y += a * v4.y;
      s.z += a * v4.z;
      s.w += a * v4.w;
      S4[d * cg + my_cg] = s;
      acc.x += b * s.x;
      acc.y += b * s.y;
      acc.z += b * s.z;
      acc.w += b * s.w;
    }
    red[my_rg * M + 4 * my_cg + 0] = acc.x;
    red[my_rg * M + 4 * my_cg + 1] = acc.y;
    red[my_rg * M + 4 * my_cg + 2] = acc.z;
    red[my_rg * M + 4 * my_cg + 3] = acc.w;
  }
  __syncthreads();
  if (tid < M) {
    float num = 0.f;
    for (int rg = 0; rg < rgs; ++rg) num += red[rg * M + tid];
    float den = 0.f;
#pragma unroll
    for (int w = 0; w < kDecodeThreads / 32; ++w) den += den_part[w];
    out[sh * M + tid] = from_f32<T>(num / den);
  }
}

}  // namespace

cudaError_t decode_step(const void* q, const void* k, const void* v, float* S, float* Z, void* out,
                        int n_sh, int D, int M, int dtype, cudaStream_t st) {
  if (dtype == LA_F32)
    decode_kernel<float><<<n_sh, kDecodeThreads, 0, st>>>(
        (const float*)q, (const float*)k, (const float*)v, S, Z, (float*)out, D, M);
  else
    decode_kernel<__nv_bfloat16><<<n_sh, kDecodeThreads, 0, st>>>(
        (const __nv_bfloat16*)q, (const __nv_bfloat16*)k, (const __nv_bfloat16*)v, S, Z,
        (__nv_bfloat16*)out, D, M);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace la
