// General-shape CUDA-core kernels for kernelized linear attention.
//
// These serve float32 inputs and any D, M (multiples of 8 up to 128) in either
// dtype. One CTA owns one (batch, head) sequence and walks it in chunks of
// kChunk tokens, carrying the state in shared memory in float32:
//
//   causal  ("Transformers are RNNs" deck, slide 4; paperlayer.ai summary §3.3)
//     S_i = S_{i-1} + phi(K_i) V_i^T, Z_i = Z_{i-1} + phi(K_i),
//     out_i = phi(Q_i)^T S_i / phi(Q_i)^T Z_i
//   non-causal (nubint.ai review, "Proposed method"): the same with full sums.
//
// Within a chunk the inclusive lower-triangular part is computed directly,
// A[i][j] = phi(Q_i).phi(K_j) for j <= i, which equals the recurrence exactly
// up to rounding order. The backward (paperlayer.ai summary §3.3.1, App. A)
// runs a forward-direction scan for dq and a reverse-direction scan for dk, dv.
#include "la_common.cuh"
#include "la_internal.h"

namespace la {
namespace {

constexpr int kChunk = 32;
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

template <typename T>
__device__ __forceinline__ void load_rows(const T* __restrict__ src, int rows_valid, int cols,
                                          float* dst, bool apply_phi) {
  for (int e = threadIdx.x; e < kChunk * cols; e += blockDim.x) {
    const int r = e / cols;
    float x = 0.f;
    if (r < rows_valid) {
      x = to_f32<T>(src[e]);
      if (apply_phi) x = phi(x);
    }
    dst[e] = x;
  }
}

// S[d][m] += sum_j fk[j][d] * vv[j][m];  Z[d] += sum_j fk[j][d]
__device__ __forceinline__ void accumulate_state(float* S, float* Z, const float* fk,
                                                 const float* vv, int D, int M) {
  for (int e = threadIdx.x; e < D * M; e += blockDim.x) {
    const int d = e / M, m = e % M;
    float acc = 0.f;
#pragma unroll 8
    for (int j = 0; j < kChunk; ++j) acc += fk[j * D + d] * vv[j * M + m];
    S[e] += acc;
  }
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float acc = 0.f;
    for (int j = 0; j < kChunk; ++j) acc += fk[j * D + d];
    Z[d] += acc;
  }
}

// scores[i][j] = a[i] . b[j] (length L) where keep(i, j), else 0
template <bool LOWER, bool UPPER>
__device__ __forceinline__ void pair_dots(const float* a, const float* b, int L, int nv,
                                          float* out) {
  for (int e = threadIdx.x; e < kChunk * kChunk; e += blockDim.x) {
    const int i = e / kChunk, j = e % kChunk;
    float acc = 0.f;
    const bool keep = i < nv && j < nv && (!LOWER || j <= i) && (!UPPER || j >= i);
    if (keep) {
      for (int d = 0; d < L; ++d) acc += a[i * L + d] * b[j * L + d];
    }
    out[e] = acc;
  }
}

// ----------------------------------------------------------------- forward

template <typename T, bool CAUSAL>
__global__ void __launch_bounds__(kThreads)
simt_forward_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                    T* __restrict__ out, float* __restrict__ S_out, float* __restrict__ Z_out,
                    int N, int D, int M) {
  extern __shared__ float sm[];
  float* S = sm;                   // D*M
  float* Z = S + D * M;            // D
  float* fq = Z + D;               // kChunk*D
  float* fk = fq + kChunk * D;     // kChunk*D
  float* vv = fk + kChunk * D;     // kChunk*M
  float* A = vv + kChunk * M;      // kChunk*kChunk
  float* den = A + kChunk * kChunk;  // kChunk

  const size_t bh = blockIdx.x;
  q += bh * (size_t)N * D;
  k += bh * (size_t)N * D;
  v += bh * (size_t)N * M;
  out += bh * (size_t)N * M;

  for (int e = threadIdx.x; e < D * M; e += blockDim.x) S[e] = 0.f;
  for (int e = threadIdx.x; e < D; e += blockDim.x) Z[e] = 0.f;
  __syncthreads();

  if (!CAUSAL) {  // full sums first
    for (int t0 = 0; t0 < N; t0 += kChunk) {
      const int nv = min(kChunk, N - t0);
      load_rows<T>(k + (size_t)t0 * D, nv, D, fk, true);
      load_rows<T>(v + (size_t)t0 * M, nv, M, vv, false);
      __syncthreads();
      accumulate_state(S, Z, fk, vv, D, M);
      __syncthreads();
    }
  }

  for (int t0 = 0; t0 < N; t0 += kChunk) {
    const int nv = min(kChunk, N - t0);
    load_rows<T>(q + (size_t)t0 * D, nv, D, fq, true);
    if (CAUSAL) {
      load_rows<T>(k + (size_t)t0 * D, nv, D, fk, true);
      load_rows<T>(v + (size_t)t0 * M, nv, M, vv, false);
    }
    __syncthreads();
    if (CAUSAL) pair_dots<true, false>(fq, fk, D, nv, A);
    __syncthreads();
    for (int i = threadIdx.x; i < kChunk; i += blockDim.x) {
      float acc = 0.f;
      for (int d = 0; d < D; ++d) acc += fq[i * D + d] * Z[d];
      if (CAUSAL)
        for (int j = 0; j <= i; ++j) acc += A[i * kChunk + j];
      den[i] = acc;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < nv * M; e += blockDim.x) {
      const int i = e / M, m = e % M;
      float acc = 0.f;
      for (int d = 0; d < D; ++d) acc += fq[i * D + d] * S[d * M + m];
      if (CAUSAL)
        for (int j = 0; j <= i; ++j) acc += A[i * kChunk + j] * vv[j * M + m];
      out[(size_t)t0 * M + e] = from_f32<T>(acc / den[i]);
    }
    __syncthreads();
    if (CAUSAL) {
      accumulate_state(S, Z, fk, vv, D, M);
      __syncthreads();
    }
  }

  if (S_out != nullptr) {
    for (int e = threadIdx.x; e < D * M; e += blockDim.x) S_out[bh * D * M + e] = S[e];
    for (int e = threadIdx.x; e < D; e += blockDim.x) Z_out[bh * D + e] = Z[e];
  }
}

// ---------------------------------------------------- backward: dq (forward scan)

// Writes dq and, per token, den_i and gd_i = -(dout_i . out_i) / den_i.
template <typename T, bool CAUSAL>
__global__ void __launch_bounds__(kThreads)
simt_bwd_dq_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                   const T* __restrict__ dout, float* __restrict__ dq,
                   float* __restrict__ ws_den, float* __restrict__ ws_gd, int N, int D, int M) {
  extern __shared__ float sm[];
  float* S = sm;                    // D*M
  float* Z = S + D * M;             // D
  float* fq = Z + D;                // kChunk*D
  float* fk = fq + kChunk * D;      // kChunk*D
  float* vv = fk + kChunk * D;      // kChunk*M
  float* g = vv + kChunk * M;       // kChunk*M   (dout, then gN)
  float* A = g + kChunk * M;        // kChunk*kChunk
  float* Tm = A + kChunk * kChunk;  // kChunk*kChunk
  float* den = Tm + kChunk * kChunk;  // kChunk
  float* gd = den + kChunk;         // kChunk

  const size_t bh = blockIdx.x;
  q += bh * (size_t)N * D;
  k += bh * (size_t)N * D;
  v += bh * (size_t)N * M;
  dout += bh * (size_t)N * M;
  dq += bh * (size_t)N * D;
  ws_den += bh * (size_t)N;
  ws_gd += bh * (size_t)N;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  for (int e = threadIdx.x; e < D * M; e += blockDim.x) S[e] = 0.f;
  for (int e = threadIdx.x; e < D; e += blockDim.x) Z[e] = 0.f;
  __syncthreads();
  if (!CAUSAL) {
    for (int t0 = 0; t0 < N; t0 += kChunk) {
      const int nv = min(kChunk, N - t0);
      load_rows<T>(k + (size_t)t0 * D, nv, D, fk, true);
      load_rows<T>(v + (size_t)t0 * M, nv, M, vv, false);
      __syncthreads();
      accumulate_state(S, Z, fk, vv, D, M);
      __syncthreads();
    }
  }

  for (int t0 = 0; t0 < N; t0 += kChunk) {
    const int nv = min(kChunk, N - t0);
    load_rows<T>(q + (size_t)t0 * D, nv, D, fq, true);
    load_rows<T>(dout + (size_t)t0 * M, nv, M, g, false);
    if (CAUSAL) {
      load_rows<T>(k + (size_t)t0 * D, nv, D, fk, true);
      load_rows<T>(v + (size_t)t0 * M, nv, M, vv, false);
    }
    __syncthreads();
    if (CAUSAL) pair_dots<true, false>(fq, fk, D, nv, A);
    __syncthreads();
    // one warp per row: den_i, out_i (on the fly) and gd_i
    for (int i = warp; i < kChunk; i += kWarps) {
      float dsum = 0.f;
      for (int d = lane; d < D; d += 32) dsum += fq[i * D + d] * Z[d];
      if (CAUSAL)
        for (int j = lane; j <= i; j += 32) dsum += A[i * kChunk + j];
      for (int o = 16; o > 0; o >>= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, o);
      float go = 0.f;
      for (int m = lane; m < M; m += 32) {
        float num = 0.f;
        for (int d = 0; d < D; ++d) num += fq[i * D + d] * S[d * M + m];
        if (CAUSAL)
          for (int j = 0; j <= i; ++j) num += A[i * kChunk + j] * vv[j * M + m];
        go += g[i * M + m] * (num / dsum);
      }
      for (int o = 16; o > 0; o >>= 1) go += __shfl_xor_sync(0xffffffffu, go, o);
      if (lane == 0) {
        const bool valid = i < nv;
        den[i] = valid ? dsum : 1.f;
        gd[i] = valid ? -go / dsum : 0.f;
        if (valid) {
          ws_den[t0 + i] = dsum;
          ws_gd[t0 + i] = -go / dsum;
        }
      }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < kChunk * M; e += blockDim.x) g[e] /= den[e / M];  // gN
    __syncthreads();
    if (CAUSAL) {  // Tm[i][j] = v_j . gN_i + gd_i for j <= i
      for (int e = threadIdx.x; e < kChunk * kChunk; e += blockDim.x) {
        const int i = e / kChunk, j = e % kChunk;
        float acc = 0.f;
        if (i < nv && j <= i) {
          for (int m = 0; m < M; ++m) acc += vv[j * M + m] * g[i * M + m];
          acc += gd[i];
        }
        Tm[e] = acc;
      }
      __syncthreads();
    }
    for (int e = threadIdx.x; e < nv * D; e += blockDim.x) {
      const int i = e / D, d = e % D;
      float acc = gd[i] * Z[d];
      for (int m = 0; m < M; ++m) acc += S[d * M + m] * g[i * M + m];
      if (CAUSAL)
        for (int j = 0; j <= i; ++j) acc += Tm[i * kChunk + j] * fk[j * D + d];
      dq[(size_t)t0 * D + e] = acc * phi_grad_from_phi(fq[e]);
    }
    __syncthreads();
    if (CAUSAL) {
      accumulate_state(S, Z, fk, vv, D, M);
      __syncthreads();
    }
  }
}

// ------------------------------------------------ backward: dk, dv (reverse scan)

template <typename T>
__device__ __forceinline__ void load_gN(const T* __restrict__ dout, const float* __restrict__ den_g,
                                        const float* __restrict__ gd_g, int nv, int M, float* g,
                                        float* gd) {
  for (int e = threadIdx.x; e < kChunk * M; e += blockDim.x) {
    const int r = e / M;
    g[e] = r < nv ? to_f32<T>(dout[e]) / den_g[r] : 0.f;
  }
  for (int r = threadIdx.x; r < kChunk; r += blockDim.x) gd[r] = r < nv ? gd_g[r] : 0.f;
}

// R[d][m] += sum_i fq[i][d] gN[i][m];  r[d] += sum_i gd[i] fq[i][d]
__device__ __forceinline__ void accumulate_reverse_state(float* R, float* r, const float* fq,
                                                         const float* g, const float* gd, int D,
                                                         int M) {
  for (int e = threadIdx.x; e < D * M; e += blockDim.x) {
    const int d = e / M, m = e % M;
    float acc = 0.f;
#pragma unroll 8
    for (int i = 0; i < kChunk; ++i) acc += fq[i * D + d] * g[i * M + m];
    R[e] += acc;
  }
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float acc = 0.f;
    for (int i = 0; i < kChunk; ++i) acc += gd[i] * fq[i * D + d];
    r[d] += acc;
  }
}

template <typename T, bool CAUSAL>
__global__ void __launch_bounds__(kThreads)
simt_bwd_dkdv_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                     const T* __restrict__ dout, float* __restrict__ dk, float* __restrict__ dv,
                     const float* __restrict__ ws_den, const float* __restrict__ ws_gd, int N,
                     int D, int M) {
  extern __shared__ float sm[];
  float* R = sm;                    // D*M
  float* r = R + D * M;             // D
  float* fq = r + D;                // kChunk*D
  float* fk = fq + kChunk * D;      // kChunk*D
  float* vv = fk + kChunk * D;      // kChunk*M
  float* g = vv + kChunk * M;       // kChunk*M  (gN)
  float* Pm = g + kChunk * M;       // kChunk*kChunk  Pm[i][j] = fq_i . fk_j  (i >= j)
  float* Um = Pm + kChunk * kChunk; // kChunk*kChunk  Um[i][j] = v_j . gN_i + gd_i (i >= j)
  float* gd = Um + kChunk * kChunk; // kChunk

  const size_t bh = blockIdx.x;
  q += bh * (size_t)N * D;
  k += bh * (size_t)N * D;
  v += bh * (size_t)N * M;
  dout += bh * (size_t)N * M;
  dk += bh * (size_t)N * D;
  dv += bh * (size_t)N * M;
  ws_den += bh * (size_t)N;
  ws_gd += bh * (size_t)N;

  for (int e = threadIdx.x; e < D * M; e += blockDim.x) R[e] = 0.f;
  for (int e = threadIdx.x; e < D; e += blockDim.x) r[e] = 0.f;
  __syncthreads();
  const int n_chunks = (N + kChunk - 1) / kChunk;
  if (!CAUSAL) {
    for (int c = 0; c < n_chunks; ++c) {
      const int t0 = c * kChunk, nv = min(kChunk, N - t0);
      load_rows<T>(q + (size_t)t0 * D, nv, D, fq, true);
      load_gN<T>(dout + (size_t)t0 * M, ws_den + t0, ws_gd + t0, nv, M, g, gd);
      __syncthreads();
      accumulate_reverse_state(R, r, fq, g, gd, D, M);
      __syncthreads();
    }
  }

  for (int c = n_chunks - 1; c >= 0; --c) {
    const int t0 = c * kChunk, nv = min(kChunk, N - t0);
    load_rows<T>(k + (size_t)t0 * D, nv, D, fk, true);
    load_rows<T>(v + (size_t)t0 * M, nv, M, vv, false);
    if (CAUSAL) {
      load_rows<T>(q + (size_t)t0 * D, nv, D, fq, true);
      load_gN<T>(dout + (size_t)t0 * M, ws_den + t0, ws_gd + t0, nv, M, g, gd);
    }
    __syncthreads();
    if (CAUSAL) {
      pair_dots<true, false>(fq, fk, D, nv, Pm);
      for (int e = threadIdx.x; e < kChunk * kChunk; e += blockDim.x) {
        const int i = e / kChunk, j = e % kChunk;
        float acc = 0.f;
        if (i < nv && j <= i) {
          for (int m = 0; m < M; ++m) acc += vv[j * M + m] * g[i * M + m];
          acc += gd[i];
        }
        Um[e] = acc;
      }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < nv * D; e += blockDim.x) {
      const int j = e / D, d = e % D;
      float acc = r[d];
      for (int m = 0; m < M; ++m) acc += R[d * M + m] * vv[j * M + m];
      if (CAUSAL)
        for (int i = j; i < nv; ++i) acc += Um[i * kChunk + j] * fq[i * D + d];
      dk[(size_t)t0 * D + e] = acc * phi_grad_from_phi(fk[e]);
    }
    for (int e = threadIdx.x; e < nv * M; e += blockDim.x) {
      const int j = e / M, m = e % M;
      float acc = 0.f;
      for (int d = 0; d < D; ++d) acc += R[d * M + m] * fk[j * D + d];
      if (CAUSAL)
        for (int i = j; i < nv; ++i) acc += Pm[i * kChunk + j] * g[i * M + m];
      dv[(size_t)t0 * M + e] = acc;
    }
    __syncthreads();
    if (CAUSAL) {
      accumulate_reverse_state(R, r, fq, g, gd, D, M);
      __syncthreads();
    }
  }
}

size_t fwd_smem(int D, int M) {
  return sizeof(float) * ((size_t)D * M + D + 2 * kChunk * D + kChunk * M + kChunk * kChunk + kChunk);
}
size_t dq_smem(int D, int M) {
  return sizeof(float) *
         ((size_t)D * M + D + 2 * kChunk * D + 2 * kChunk * M + 2 * kChunk * kChunk + 2 * kChunk);
}
size_t dkdv_smem(int D, int M) {
  return sizeof(float) *
         ((size_t)D * M + D + 2 * kChunk * D + 2 * kChunk * M + 2 * kChunk * kChunk + kChunk);
}

template <typename K, typename... Args>
cudaError_t launch(K kernel, int grid, size_t smem, cudaStream_t st, Args... args) {
  cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  kernel<<<grid, kThreads, smem, st>>>(args...);
  count_launches(1);
  return cudaGetLastError();
}

template <typename T>
cudaError_t forward_t(const void* q, const void* k, const void* v, void* out, float* S_out,
                      float* Z_out, int BH, int N, int D, int M, bool causal, cudaStream_t st) {
  const size_t smem = fwd_smem(D, M);
  auto args = [&](auto kern) {
    return launch(kern, BH, smem, st, (const T*)q, (const T*)k, (const T*)v, (T*)out, S_out,
                  Z_out, N, D, M);
  };
  return causal ? args(simt_forward_kernel<T, true>) : args(simt_forward_kernel<T, false>);
}

template <typename T>
cudaError_t backward_t(const void* q, const void* k, const void* v, const void* dout, float* dq,
                       float* dk, float* dv, int BH, int N, int D, int M, bool causal, void* ws,
                       cudaStream_t st) {
  float* den = reinterpret_cast<float*>(static_cast<char*>(ws) + kHeaderBytes);
  float* gd = den + (size_t)BH * N;
  cudaError_t err;
  if (causal)
    err = launch(simt_bwd_dq_kernel<T, true>, BH, dq_smem(D, M), st, (const T*)q, (const T*)k,
                 (const T*)v, (const T*)dout, dq, den, gd, N, D, M);
  else
    err = launch(simt_bwd_dq_kernel<T, false>, BH, dq_smem(D, M), st, (const T*)q, (const T*)k,
                 (const T*)v, (const T*)dout, dq, den, gd, N, D, M);
  if (err != cudaSuccess) return err;
  if (causal)
    return launch(simt_bwd_dkdv_kernel<T, true>, BH, dkdv_smem(D, M), st, (const T*)q,
                  (const T*)k, (const T*)v, (const T*)dout, dk, dv, (const float*)den,
                  (const float*)gd, N, D, M);
  return launch(simt_bwd_dkdv_kernel<T, false>, BH, dkdv_smem(D, M), st, (const T*)q, (const T*)k,
                (const T*)v, (const T*)dout, dk, dv, (const float*)den, (const float*)gd, N, D,
                M);
}

}  // namespace

cudaError_t simt_forward(const void* q, const void* k, const void* v, void* out, float* S_out,
                         float* Z_out, int BH, int N, int D, int M, bool causal, int dtype,
                         cudaStream_t st) {
  if (dtype == LA_F32) return forward_t<float>(q, k, v, out, S_out, Z_out, BH, N, D, M, causal, st);
  return forward_t<__nv_bfloat16>(q, k, v, out, S_out, Z_out, BH, N, D, M, causal, st);
}

size_t simt_backward_workspace(int BH, int N) {
  return kHeaderBytes + align_up(2 * sizeof(float) * (size_t)BH * N, 256);
}

cudaError_t simt_backward(const void* q, const void* k, const void* v, const void* dout, float* dq,
                          float* dk, float* dv, int BH, int N, int D, int M, bool causal,
                          int dtype, void* ws, cudaStream_t st) {
  if (dtype == LA_F32)
    return backward_t<float>(q, k, v, dout, dq, dk, dv, BH, N, D, M, causal, ws, st);
  return backward_t<__nv_bfloat16>(q, k, v, dout, dq, dk, dv, BH, N, D, M, causal, ws, st);
}

}  // namespace la
