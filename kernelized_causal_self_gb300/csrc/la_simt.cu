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

// load_rows for rows `rs` elements apart (the packed token-major layout)
template <typename T>
__device__ __forceinline__ void load_rows_strided(const T* __restrict__ src, int rows_valid,
                                                  int cols, size_t rs, float* dst, bool apply_phi) {
  for (int e = threadIdx.x; e < kChunk * cols; e += blockDim.x) {
    const int r = e / cols, c = e % cols;
    float x = 0.f;
    if (r < rows_valid) {
      x = to_f32<T>(src[(size_t)r * rs + c]);
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
                    T* __restrict__ out, StateIO io, WorkspaceHeader* hdr, int N, int D, int M) {
  extern __shared__ float sm[];
  float* S = sm;                   // D*M
  float* Z = S + D * M;            // D
  float* fq = Z + D;               // kChunk*D
  float* fk = fq + kChunk * D;     // kChunk*D
  float* vv = fk + kChunk * D;     // kChunk*M
  float* A = vv + kChunk * M;      // kChunk*kChunk
  float* den = A + kChunk * kChunk;  // kChunk

  const size_t bh = blockIdx.x;
  // this sequence's first row and the distance between its token rows: [BH][N][D],
  // or the packed [T][H][D] with stream b = bh / H in rows cu[b] .. cu[b + 1] - 1
  size_t rq = D, rv = M;
  int len = N;
  if (io.cu != nullptr) {
    const int b = (int)(bh / io.H), s0 = io.cu[b], e0 = io.cu[b + 1];
    const bool ok = 0 <= s0 && s0 <= e0 && e0 <= io.T;
    if (!(ok && e0 - s0 <= N) && threadIdx.x == 0) atomicExch(&hdr->status, (int)LA_ERR_INVALID_ARG);
    len = ok ? min(e0 - s0, N) : 0;
    const size_t r0 = ok ? (size_t)s0 : 0, hh = bh % io.H;
    rq = (size_t)io.H * D;
    rv = (size_t)io.H * M;
    q += r0 * rq + hh * D;
    k += r0 * rq + hh * D;
    v += r0 * rv + hh * M;
    out += r0 * rv + hh * M;
  } else {
    q += bh * (size_t)N * D;
    k += bh * (size_t)N * D;
    v += bh * (size_t)N * M;
    out += bh * (size_t)N * M;
    // this stream's token count (the rest of the sequence is padding, never read)
    if (io.lens != nullptr) len = max(0, min(io.lens[bh / io.H], N));
  }

  // the sequence's state entry: initial state (extend) and final state (prefill, extend)
  size_t entry = bh;
  bool entry_ok = io.S != nullptr;
  if (entry_ok && io.slots != nullptr) {
    const int slot = io.slots[bh / io.H];
    entry_ok = slot >= 0 && slot < io.pool;
    entry = (size_t)slot * io.H + bh % io.H;
    if (!entry_ok && threadIdx.x == 0) atomicExch(&hdr->status, (int)LA_ERR_INVALID_ARG);
  }
  const bool init = entry_ok && io.read_init;
  N = len;
  for (int e = threadIdx.x; e < D * M; e += blockDim.x) S[e] = init ? io.S[entry * D * M + e] : 0.f;
  for (int e = threadIdx.x; e < D; e += blockDim.x) Z[e] = init ? io.Z[entry * D + e] : 0.f;
  __syncthreads();

  if (!CAUSAL) {  // full sums first
    for (int t0 = 0; t0 < N; t0 += kChunk) {
      const int nv = min(kChunk, N - t0);
      load_rows_strided<T>(k + (size_t)t0 * rq, nv, D, rq, fk, true);
      load_rows_strided<T>(v + (size_t)t0 * rv, nv, M, rv, vv, false);
      __syncthreads();
      accumulate_state(S, Z, fk, vv, D, M);
      __syncthreads();
    }
  }

  for (int t0 = 0; t0 < N; t0 += kChunk) {
    const int nv = min(kChunk, N - t0);
    load_rows_strided<T>(q + (size_t)t0 * rq, nv, D, rq, fq, true);
    if (CAUSAL) {
      load_rows_strided<T>(k + (size_t)t0 * rq, nv, D, rq, fk, true);
      load_rows_strided<T>(v + (size_t)t0 * rv, nv, M, rv, vv, false);
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
      out[(size_t)(t0 + i) * rv + m] = from_f32<T>(acc / den[i]);
    }
    __syncthreads();
    if (CAUSAL) {
      accumulate_state(S, Z, fk, vv, D, M);
      __syncthreads();
    }
  }

  if (entry_ok && io.write_final) {
    for (int e = threadIdx.x; e < D * M; e += blockDim.x) io.S[entry * D * M + e] = S[e];
    for (int e = threadIdx.x; e < D; e += blockDim.x) io.Z[entry * D + e] = Z[e];
  }
}

// ---------------------------------------------------- backward: dq (forward scan)
//
// The gradient of phi(Q_i) is S_i gN_i + gd_i Z_i, and the two terms cancel
// strongly (exactly at i = 0, where out_0 = v_0 whatever q_0 is). The backward
// kernels therefore carry state and form these combinations in the accumulator
// type Acc: double for float32 inputs (so the result keeps float32 accuracy
// relative to its own size), float for bfloat16 inputs.

template <typename Acc>
__device__ __forceinline__ void accumulate_state_acc(Acc* S, Acc* Z, const float* fk,
                                                     const float* vv, int D, int M) {
  for (int e = threadIdx.x; e < D * M; e += blockDim.x) {
    const int d = e / M, m = e % M;
    Acc acc = 0;
#pragma unroll 8
    for (int j = 0; j < kChunk; ++j) acc += (Acc)fk[j * D + d] * (Acc)vv[j * M + m];
    S[e] += acc;
  }
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    Acc acc = 0;
    for (int j = 0; j < kChunk; ++j) acc += (Acc)fk[j * D + d];
    Z[d] += acc;
  }
}

template <typename Acc>
__device__ __forceinline__ Acc warp_sum(Acc x) {
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Writes dq and, per token, den_i and gd_i = -(dout_i . out_i) / den_i.
// S0, Z0: the state before the sequence ([bh][D][M], [bh][D]; nullptr: zero).
template <typename T, typename Acc, bool CAUSAL>
__global__ void __launch_bounds__(kThreads)
simt_bwd_dq_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                   const T* __restrict__ dout, float* __restrict__ dq,
                   Acc* __restrict__ ws_den, Acc* __restrict__ ws_gd, int N, int D, int M,
                   const float* __restrict__ S0, const float* __restrict__ Z0) {
  extern __shared__ __align__(16) unsigned char smraw[];
  Acc* S = reinterpret_cast<Acc*>(smraw);  // D*M
  Acc* Z = S + D * M;                       // D
  Acc* A = Z + D;                           // kChunk*kChunk  phi(q_i).phi(k_j), j <= i
  Acc* Tm = A + kChunk * kChunk;            // kChunk*kChunk  v_j.gN_i + gd_i, j <= i
  Acc* den = Tm + kChunk * kChunk;          // kChunk
  Acc* gd = den + kChunk;                   // kChunk
  Acc* g = gd + kChunk;                     // kChunk*M   (dout, then gN)
  float* fq = reinterpret_cast<float*>(g + kChunk * M);  // kChunk*D
  float* fk = fq + kChunk * D;                           // kChunk*D
  float* vv = fk + kChunk * D;                           // kChunk*M

  const size_t bh = blockIdx.x;
  q += bh * (size_t)N * D;
  k += bh * (size_t)N * D;
  v += bh * (size_t)N * M;
  dout += bh * (size_t)N * M;
  dq += bh * (size_t)N * D;
  ws_den += bh * (size_t)N;
  ws_gd += bh * (size_t)N;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  for (int e = threadIdx.x; e < D * M; e += blockDim.x)
    S[e] = S0 != nullptr ? (Acc)S0[bh * D * M + e] : (Acc)0;
  for (int e = threadIdx.x; e < D; e += blockDim.x) Z[e] = Z0 != nullptr ? (Acc)Z0[bh * D + e] : (Acc)0;
  __syncthreads();
  if (!CAUSAL) {
    for (int t0 = 0; t0 < N; t0 += kChunk) {
      const int nv = min(kChunk, N - t0);
      load_rows<T>(k + (size_t)t0 * D, nv, D, fk, true);
      load_rows<T>(v + (size_t)t0 * M, nv, M, vv, false);
      __syncthreads();
      accumulate_state_acc<Acc>(S, Z, fk, vv, D, M);
      __syncthreads();
    }
  }

  for (int t0 = 0; t0 < N; t0 += kChunk) {
    const int nv = min(kChunk, N - t0);
    load_rows<T>(q + (size_t)t0 * D, nv, D, fq, true);
    for (int e = threadIdx.x; e < kChunk * M; e += blockDim.x)
      g[e] = (e / M) < nv ? (Acc)to_f32<T>(dout[(size_t)t0 * M + e]) : (Acc)0;
    if (CAUSAL) {
      load_rows<T>(k + (size_t)t0 * D, nv, D, fk, true);
      load_rows<T>(v + (size_t)t0 * M, nv, M, vv, false);
    }
    __syncthreads();
    if (CAUSAL) {
      for (int e = threadIdx.x; e < kChunk * kChunk; e += blockDim.x) {
        const int i = e / kChunk, j = e % kChunk;
        Acc acc = 0;
        if (i < nv && j <= i)
          for (int d = 0; d < D; ++d) acc += (Acc)fq[i * D + d] * (Acc)fk[j * D + d];
        A[e] = acc;
      }
    }
    __syncthreads();
    // one warp per row: den_i, out_i (on the fly) and gd_i
    for (int i = warp; i < kChunk; i += kWarps) {
      Acc dsum = 0;
      for (int d = lane; d < D; d += 32) dsum += (Acc)fq[i * D + d] * Z[d];
      if (CAUSAL)
        for (int j = lane; j <= i; j += 32) dsum += A[i * kChunk + j];
      dsum = warp_sum(dsum);
      Acc go = 0;
      for (int m = lane; m < M; m += 32) {
        Acc num = 0;
        for (int d = 0; d < D; ++d) num += (Acc)fq[i * D + d] * S[d * M + m];
        if (CAUSAL)
          for (int j = 0; j <= i; ++j) num += A[i * kChunk + j] * (Acc)vv[j * M + m];
        go += g[i * M + m] * (num / dsum);
      }
      go = warp_sum(go);
      if (lane == 0) {
        const bool valid = i < nv;
        den[i] = valid ? dsum : (Acc)1;
        gd[i] = valid ? -go / dsum : (Acc)0;
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
        Acc acc = 0;
        if (i < nv && j <= i) {
          for (int m = 0; m < M; ++m) acc += (Acc)vv[j * M + m] * g[i * M + m];
          acc += gd[i];
        }
        Tm[e] = acc;
      }
      __syncthreads();
    }
    for (int e = threadIdx.x; e < nv * D; e += blockDim.x) {
      const int i = e / D, d = e % D;
      Acc acc = gd[i] * Z[d];
      for (int m = 0; m < M; ++m) acc += S[d * M + m] * g[i * M + m];
      if (CAUSAL)
        for (int j = 0; j <= i; ++j) acc += Tm[i * kChunk + j] * (Acc)fk[j * D + d];
      dq[(size_t)t0 * D + e] = (float)(acc * (Acc)phi_grad_from_phi(fq[e]));
    }
    __syncthreads();
    if (CAUSAL) {
      accumulate_state_acc<Acc>(S, Z, fk, vv, D, M);
      __syncthreads();
    }
  }
}

// ------------------------------------------------ backward: dk, dv (reverse scan)

// R[d][m] += sum_i fq[i][d] gN[i][m];  r[d] += sum_i gd[i] fq[i][d]
template <typename Acc>
__device__ __forceinline__ void accumulate_reverse_state(Acc* R, Acc* r, const float* fq,
                                                         const Acc* g, const Acc* gd, int D,
                                                         int M) {
  for (int e = threadIdx.x; e < D * M; e += blockDim.x) {
    const int d = e / M, m = e % M;
    Acc acc = 0;
#pragma unroll 8
    for (int i = 0; i < kChunk; ++i) acc += (Acc)fq[i * D + d] * g[i * M + m];
    R[e] += acc;
  }
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    Acc acc = 0;
    for (int i = 0; i < kChunk; ++i) acc += gd[i] * (Acc)fq[i * D + d];
    r[d] += acc;
  }
}

template <typename T, typename Acc>
__device__ __forceinline__ void load_gN(const T* __restrict__ dout, const Acc* __restrict__ den_g,
                                        const Acc* __restrict__ gd_g, int nv, int M, Acc* g,
                                        Acc* gd) {
  for (int e = threadIdx.x; e < kChunk * M; e += blockDim.x) {
    const int r = e / M;
    g[e] = r < nv ? (Acc)to_f32<T>(dout[e]) / den_g[r] : (Acc)0;
  }
  for (int r = threadIdx.x; r < kChunk; r += blockDim.x) gd[r] = r < nv ? gd_g[r] : (Acc)0;
}

// R0, r0: the reverse sums after the sequence ([bh][D][M], [bh][D]; nullptr: zero).
template <typename T, typename Acc, bool CAUSAL>
__global__ void __launch_bounds__(kThreads)
simt_bwd_dkdv_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                     const T* __restrict__ dout, float* __restrict__ dk, float* __restrict__ dv,
                     const Acc* __restrict__ ws_den, const Acc* __restrict__ ws_gd, int N, int D,
                     int M, const float* __restrict__ R0, const float* __restrict__ r0) {
  extern __shared__ __align__(16) unsigned char smraw[];
  Acc* R = reinterpret_cast<Acc*>(smraw);  // D*M
  Acc* r = R + D * M;                       // D
  Acc* Pm = r + D;                          // kChunk*kChunk  phi(q_i).phi(k_j), i >= j
  Acc* Um = Pm + kChunk * kChunk;           // kChunk*kChunk  v_j.gN_i + gd_i,  i >= j
  Acc* gd = Um + kChunk * kChunk;           // kChunk
  Acc* g = gd + kChunk;                     // kChunk*M  (gN)
  float* fq = reinterpret_cast<float*>(g + kChunk * M);  // kChunk*D
  float* fk = fq + kChunk * D;                           // kChunk*D
  float* vv = fk + kChunk * D;                           // kChunk*M

  const size_t bh = blockIdx.x;
  q += bh * (size_t)N * D;
  k += bh * (size_t)N * D;
  v += bh * (size_t)N * M;
  dout += bh * (size_t)N * M;
  dk += bh * (size_t)N * D;
  dv += bh * (size_t)N * M;
  ws_den += bh * (size_t)N;
  ws_gd += bh * (size_t)N;

  for (int e = threadIdx.x; e < D * M; e += blockDim.x)
    R[e] = R0 != nullptr ? (Acc)R0[bh * D * M + e] : (Acc)0;
  for (int e = threadIdx.x; e < D; e += blockDim.x) r[e] = r0 != nullptr ? (Acc)r0[bh * D + e] : (Acc)0;
  __syncthreads();
  const int n_chunks = (N + kChunk - 1) / kChunk;
  if (!CAUSAL) {
    for (int c = 0; c < n_chunks; ++c) {
      const int t0 = c * kChunk, nv = min(kChunk, N - t0);
      load_rows<T>(q + (size_t)t0 * D, nv, D, fq, true);
      load_gN<T, Acc>(dout + (size_t)t0 * M, ws_den + t0, ws_gd + t0, nv, M, g, gd);
      __syncthreads();
      accumulate_reverse_state<Acc>(R, r, fq, g, gd, D, M);
      __syncthreads();
    }
  }

  for (int c = n_chunks - 1; c >= 0; --c) {
    const int t0 = c * kChunk, nv = min(kChunk, N - t0);
    load_rows<T>(k + (size_t)t0 * D, nv, D, fk, true);
    load_rows<T>(v + (size_t)t0 * M, nv, M, vv, false);
    if (CAUSAL) {
      load_rows<T>(q + (size_t)t0 * D, nv, D, fq, true);
      load_gN<T, Acc>(dout + (size_t)t0 * M, ws_den + t0, ws_gd + t0, nv, M, g, gd);
    }
    __syncthreads();
    if (CAUSAL) {
      for (int e = threadIdx.x; e < kChunk * kChunk; e += blockDim.x) {
        const int i = e / kChunk, j = e % kChunk;
        Acc p = 0, u = 0;
        if (i < nv && j <= i) {
          for (int d = 0; d < D; ++d) p += (Acc)fq[i * D + d] * (Acc)fk[j * D + d];
          for (int m = 0; m < M; ++m) u += (Acc)vv[j * M + m] * g[i * M + m];
          u += gd[i];
        }
        Pm[e] = p;
        Um[e] = u;
      }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < nv * D; e += blockDim.x) {
      const int j = e / D, d = e % D;
      Acc acc = r[d];
      for (int m = 0; m < M; ++m) acc += R[d * M + m] * (Acc)vv[j * M + m];
      if (CAUSAL)
        for (int i = j; i < nv; ++i) acc += Um[i * kChunk + j] * (Acc)fq[i * D + d];
      dk[(size_t)t0 * D + e] = (float)(acc * (Acc)phi_grad_from_phi(fk[e]));
    }
    for (int e = threadIdx.x; e < nv * M; e += blockDim.x) {
      const int j = e / M, m = e % M;
      Acc acc = 0;
      for (int d = 0; d < D; ++d) acc += R[d * M + m] * (Acc)fk[j * D + d];
      if (CAUSAL)
        for (int i = j; i < nv; ++i) acc += Pm[i * kChunk + j] * g[i * M + m];
      dv[(size_t)t0 * M + e] = (float)acc;
    }
    __syncthreads();
    if (CAUSAL) {
      accumulate_reverse_state<Acc>(R, r, fq, g, gd, D, M);
      __syncthreads();
    }
  }
}

// ------------------------------------------------ state sums, reverse sums

// S = sum_j phi(k_j) v_j^T, Z = sum_j phi(k_j) of each sequence into io's entries.
template <typename T>
__global__ void __launch_bounds__(kThreads)
simt_state_sums_kernel(const T* __restrict__ k, const T* __restrict__ v, StateIO io, int N, int D,
                       int M) {
  extern __shared__ float sm[];
  float* S = sm;                // D*M
  float* Z = S + D * M;         // D
  float* fk = Z + D;            // kChunk*D
  float* vv = fk + kChunk * D;  // kChunk*M
  const size_t bh = blockIdx.x;
  k += bh * (size_t)N * D;
  v += bh * (size_t)N * M;
  for (int e = threadIdx.x; e < D * M; e += blockDim.x) S[e] = 0.f;
  for (int e = threadIdx.x; e < D; e += blockDim.x) Z[e] = 0.f;
  __syncthreads();
  for (int t0 = 0; t0 < N; t0 += kChunk) {
    const int nv = min(kChunk, N - t0);
    load_rows<T>(k + (size_t)t0 * D, nv, D, fk, true);
    load_rows<T>(v + (size_t)t0 * M, nv, M, vv, false);
    __syncthreads();
    accumulate_state(S, Z, fk, vv, D, M);
    __syncthreads();
  }
  for (int e = threadIdx.x; e < D * M; e += blockDim.x) io.S[bh * D * M + e] = S[e];
  for (int e = threadIdx.x; e < D; e += blockDim.x) io.Z[bh * D + e] = Z[e];
}

// R = sum_i phi(q_i) gN_i^T, r = sum_i gd_i phi(q_i) of each sequence (its own
// reverse sums, from den_i and gd_i of the dq pass) into R_out [bh][D][M], r_out [bh][D].
template <typename T, typename Acc>
__global__ void __launch_bounds__(kThreads)
simt_reverse_sums_kernel(const T* __restrict__ q, const T* __restrict__ dout,
                         const Acc* __restrict__ ws_den, const Acc* __restrict__ ws_gd,
                         float* __restrict__ R_out, float* __restrict__ r_out, int N, int D, int M) {
  extern __shared__ __align__(16) unsigned char smraw[];
  Acc* R = reinterpret_cast<Acc*>(smraw);  // D*M
  Acc* r = R + D * M;                       // D
  Acc* gd = r + D;                          // kChunk
  Acc* g = gd + kChunk;                     // kChunk*M  (gN)
  float* fq = reinterpret_cast<float*>(g + kChunk * M);  // kChunk*D
  const size_t bh = blockIdx.x;
  q += bh * (size_t)N * D;
  dout += bh * (size_t)N * M;
  ws_den += bh * (size_t)N;
  ws_gd += bh * (size_t)N;
  for (int e = threadIdx.x; e < D * M; e += blockDim.x) R[e] = 0;
  for (int e = threadIdx.x; e < D; e += blockDim.x) r[e] = 0;
  __syncthreads();
  for (int t0 = 0; t0 < N; t0 += kChunk) {
    const int nv = min(kChunk, N - t0);
    load_rows<T>(q + (size_t)t0 * D, nv, D, fq, true);
    load_gN<T, Acc>(dout + (size_t)t0 * M, ws_den + t0, ws_gd + t0, nv, M, g, gd);
    __syncthreads();
    accumulate_reverse_state<Acc>(R, r, fq, g, gd, D, M);
    __syncthreads();
  }
  for (int e = threadIdx.x; e < D * M; e += blockDim.x) R_out[bh * D * M + e] = (float)R[e];
  for (int e = threadIdx.x; e < D; e += blockDim.x) r_out[bh * D + e] = (float)r[e];
}

size_t sums_smem(int D, int M) {
  return sizeof(float) * ((size_t)D * M + D + kChunk * D + kChunk * M);
}
template <typename Acc>
size_t rsums_smem(int D, int M) {
  return sizeof(Acc) * ((size_t)D * M + D + kChunk + kChunk * M) + sizeof(float) * kChunk * D;
}

size_t fwd_smem(int D, int M) {
  return sizeof(float) * ((size_t)D * M + D + 2 * kChunk * D + kChunk * M + kChunk * kChunk + kChunk);
}
template <typename Acc>
size_t dq_smem(int D, int M) {
  return sizeof(Acc) * ((size_t)D * M + D + 2 * kChunk * kChunk + 2 * kChunk + kChunk * M) +
         sizeof(float) * (2 * kChunk * D + kChunk * M);
}
template <typename Acc>
size_t dkdv_smem(int D, int M) {
  return sizeof(Acc) * ((size_t)D * M + D + 2 * kChunk * kChunk + kChunk + kChunk * M) +
         sizeof(float) * (2 * kChunk * D + kChunk * M);
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
cudaError_t forward_t(const void* q, const void* k, const void* v, void* out, const StateIO& io,
                      int BH, int N, int D, int M, bool causal, WorkspaceHeader* hdr,
                      cudaStream_t st) {
  const size_t smem = fwd_smem(D, M);
  auto args = [&](auto kern) {
    return launch(kern, BH, smem, st, (const T*)q, (const T*)k, (const T*)v, (T*)out, io, hdr, N,
                  D, M);
  };
  return causal ? args(simt_forward_kernel<T, true>) : args(simt_forward_kernel<T, false>);
}

template <typename T, typename Acc>
cudaError_t backward_q_t(const void* q, const void* k, const void* v, const void* dout, float* dq,
                         const StateIO* pre, const StateIO* own, int BH, int N, int D, int M,
                         bool causal, void* ws, cudaStream_t st) {
  Acc* den = reinterpret_cast<Acc*>(static_cast<char*>(ws) + kHeaderBytes);
  Acc* gd = den + (size_t)BH * N;
  const float* S0 = (causal && pre != nullptr) ? pre->S : nullptr;
  const float* Z0 = (causal && pre != nullptr) ? pre->Z : nullptr;
  cudaError_t err;
  if (causal)
    err = launch(simt_bwd_dq_kernel<T, Acc, true>, BH, dq_smem<Acc>(D, M), st, (const T*)q,
                 (const T*)k, (const T*)v, (const T*)dout, dq, den, gd, N, D, M, S0, Z0);
  else
    err = launch(simt_bwd_dq_kernel<T, Acc, false>, BH, dq_smem<Acc>(D, M), st, (const T*)q,
                 (const T*)k, (const T*)v, (const T*)dout, dq, den, gd, N, D, M, S0, Z0);
  if (err != cudaSuccess || own == nullptr) return err;
  return launch(simt_reverse_sums_kernel<T, Acc>, BH, rsums_smem<Acc>(D, M), st, (const T*)q,
                (const T*)dout, (const Acc*)den, (const Acc*)gd, own->S, own->Z, N, D, M);
}

template <typename T, typename Acc>
cudaError_t backward_kv_t(const void* q, const void* k, const void* v, const void* dout, float* dk,
                          float* dv, const StateIO* suf, int BH, int N, int D, int M, bool causal,
                          void* ws, cudaStream_t st) {
  Acc* den = reinterpret_cast<Acc*>(static_cast<char*>(ws) + kHeaderBytes);
  Acc* gd = den + (size_t)BH * N;
  const float* R0 = (causal && suf != nullptr) ? suf->S : nullptr;
  const float* r0 = (causal && suf != nullptr) ? suf->Z : nullptr;
  if (causal)
    return launch(simt_bwd_dkdv_kernel<T, Acc, true>, BH, dkdv_smem<Acc>(D, M), st, (const T*)q,
                  (const T*)k, (const T*)v, (const T*)dout, dk, dv, (const Acc*)den,
                  (const Acc*)gd, N, D, M, R0, r0);
  return launch(simt_bwd_dkdv_kernel<T, Acc, false>, BH, dkdv_smem<Acc>(D, M), st, (const T*)q,
                (const T*)k, (const T*)v, (const T*)dout, dk, dv, (const Acc*)den,
                (const Acc*)gd, N, D, M, R0, r0);
}

}  // namespace

cudaError_t simt_forward(const void* q, const void* k, const void* v, void* out,
                         const StateIO& io, int BH, int N, int D, int M, bool causal, int dtype,
                         WorkspaceHeader* hdr, cudaStream_t st) {
  if (dtype == LA_F32) return forward_t<float>(q, k, v, out, io, BH, N, D, M, causal, hdr, st);
  return forward_t<__nv_bfloat16>(q, k, v, out, io, BH, N, D, M, causal, hdr, st);
}

size_t simt_backward_workspace(int BH, int N) {
  return kHeaderBytes + align_up(2 * sizeof(double) * (size_t)BH * N, 256);
}

cudaError_t simt_backward_q(const void* q, const void* k, const void* v, const void* dout,
                            float* dq, const StateIO* pre, const StateIO* own, int BH, int N,
                            int D, int M, bool causal, int dtype, void* ws, cudaStream_t st) {
  if (dtype == LA_F32)
    return backward_q_t<float, double>(q, k, v, dout, dq, pre, own, BH, N, D, M, causal, ws, st);
  return backward_q_t<__nv_bfloat16, float>(q, k, v, dout, dq, pre, own, BH, N, D, M, causal, ws,
                                            st);
}

cudaError_t simt_backward_kv(const void* q, const void* k, const void* v, const void* dout,
                             float* dk, float* dv, const StateIO* suf, int BH, int N, int D,
                             int M, bool causal, int dtype, void* ws, cudaStream_t st) {
  if (dtype == LA_F32)
    return backward_kv_t<float, double>(q, k, v, dout, dk, dv, suf, BH, N, D, M, causal, ws, st);
  return backward_kv_t<__nv_bfloat16, float>(q, k, v, dout, dk, dv, suf, BH, N, D, M, causal,
                                             ws, st);
}

cudaError_t simt_backward(const void* q, const void* k, const void* v, const void* dout, float* dq,
                          float* dk, float* dv, int BH, int N, int D, int M, bool causal,
                          int dtype, void* ws, cudaStream_t st) {
  cudaError_t e = simt_backward_q(q, k, v, dout, dq, nullptr, nullptr, BH, N, D, M, causal, dtype,
                                  ws, st);
  if (e != cudaSuccess) return e;
  return simt_backward_kv(q, k, v, dout, dk, dv, nullptr, BH, N, D, M, causal, dtype, ws, st);
}

cudaError_t simt_state_sums(const void* k, const void* v, const StateIO& io, int BH, int N, int D,
                            int M, int dtype, cudaStream_t st) {
  if (dtype == LA_F32)
    return launch(simt_state_sums_kernel<float>, BH, sums_smem(D, M), st, (const float*)k,
                  (const float*)v, io, N, D, M);
  return launch(simt_state_sums_kernel<__nv_bfloat16>, BH, sums_smem(D, M), st,
                (const __nv_bfloat16*)k, (const __nv_bfloat16*)v, io, N, D, M);
}

}  // namespace la
