// Random Fourier features, bf16 inputs with D = M = F = 64.
//
// paperlayer.ai summary §5 names random Fourier features, approximating the RBF
// kernel, as the feature map to try next. With the F rows w_f of W and the phases
// b_f given (the caller draws them: w_f ~ N(0, sigma^-2 I), b_f ~ U[0, 2 pi) for
// the RBF kernel of width sigma),
//   phi(x) = sqrt(2 / F) [cos(w_1 . x + b_1), ..., cos(w_F . x + b_F)],
// so that phi(x) . phi(y) estimates exp(-|x - y|^2 / (2 sigma^2)); the attention
// is then the linear attention of la_forward with this phi in place of elu + 1.
//
// tc_rff_feature_kernel: one CTA per 128-row tile of q or k: X W^T on tcgen05
// (M = 128 rows, N = F = 64, K = D = 64; W is the K-major B operand), then in
// float32 on the CUDA cores cos(. + b) sqrt(2 / F), rounded to bf16 and stored
// with a TMA store into the feature buffer. The forward kernels then run in
// their identity-feature mode on the two feature buffers.
#include <cuda_bf16.h>

#include "la_tc_common.cuh"

namespace la {
namespace tcx {
namespace {

constexpr int kRffThreads = 128;  // thread = tile row
// X tile, W tile (64 x 64), barriers: eight CTAs per SM, their 64 TMEM columns each
// filling the SM's 512
constexpr int kRffSmem = 1024 + kTile + kDim * 128 + 256;

__global__ void __launch_bounds__(kRffThreads)
tc_rff_feature_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_fq,
                      const __grid_constant__ CUtensorMap tm_fk, const float* __restrict__ bias, int N,
                      int tiles, WorkspaceHeader* hdr) {
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  uint8_t* xt = sm;             // 128 x 64 bf16 (then the features, staged for the store)
  uint8_t* wt = xt + kTile;     // 64 x 64 bf16
  uint64_t* full = reinterpret_cast<uint64_t*>(wt + kDim * 128);
  uint64_t* mma_bar = full + 1;
  uint64_t* drain = mma_bar + 1;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(drain + 1);

  const int tid = threadIdx.x, warp = tid / 32;
  const bool is_k = blockIdx.x >= tiles;
  const int tile = is_k ? blockIdx.x - tiles : blockIdx.x;
  const int n_chunks = (N + kC - 1) / kC;
  const int bh = tile / n_chunks, t0 = (tile % n_chunks) * kC;
  const CUtensorMap* tm_x = is_k ? &tm_k : &tm_q;
  const CUtensorMap* tm_f = is_k ? &tm_fk : &tm_fq;
  if (tid == 0) {
    mbar_init(full, 1);
    mbar_init(mma_bar, 1);
    mbar_init(drain, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tslot, 64);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tbase = *tslot;
  const uint32_t tl = tbase + ((uint32_t)(warp * 32) << 16);
  pdl_wait();
  if (tid == 0) {
    mbar_arrive_expect_tx(full, kTile + kDim * 128);
    tma_load_3d(xt, tm_x, full, 0, t0, bh);
    tma_load_3d(wt, &tm_w, full, 0, 0, 0);
  }
  bool ok = wait_uniform(full, 0, hdr, 61);
  if (ok) {
    if (tid == 0) {  // X W^T: A = X (K-major), B = W (rows f = N, d contiguous = K-major)
      const uint32_t id = idesc_bf16(128, 64, false, false);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        mma_ss(tbase, sdesc(smem_u32(xt) + k * 32, 16, 1024), sdesc(smem_u32(wt) + k * 32, 16, 1024), id, k);
      mma_commit(mma_bar);
    }
    ok = wait_uniform(mma_bar, 0, hdr, 62);
  }
  if (ok) {
    fence_after_sync();
    uint32_t ra[32], rb[32];
    tmem_ld32x2(tl, ra, tl + 32, rb);
    const float scale = sqrtf(2.f / kDim);
    // phi = sqrt(2/F) cos(x . w_f + b_f) -> bf16, over the X tile (every MMA that read it is
    // done); the hardware cosine: its absolute error (~1e-6 for the arguments of unit-scale
    // inputs and weights) is far below the bf16 rounding of the result
#pragma unroll
    for (int c16 = 0; c16 < 8; ++c16) {
      const uint32_t* src = c16 < 4 ? ra : rb;
      const int b0 = (c16 & 3) * 8, f0 = c16 * 8;
      uint32_t w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        w[q] = pack_bf16(scale * __cosf(__uint_as_float(src[b0 + 2 * q]) + bias[f0 + 2 * q]),
                         scale * __cosf(__uint_as_float(src[b0 + 2 * q + 1]) + bias[f0 + 2 * q + 1]));
      *reinterpret_cast<uint4*>(xt + sw128(tid, c16 * 16)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    fence_proxy_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (tid == 0) {  // rows past the sequence end are clipped by the tensor map
      tma_store_3d(tm_f, xt, 0, t0, bh);
      bulk_commit();
      bulk_wait_all<0>();
    }
  }
  pdl_trigger();
  if (tid == 0 && !ok) {  // after an early exit: the copies issued are done
    if (!mbar_wait(full, 0)) record_timeout(hdr, 63);
  }
  drain_mmas(drain, hdr, 64);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (warp == 0) tmem_dealloc(tbase, 64);
}

}  // namespace
}  // namespace tcx

using namespace tcx;

bool rff_supported(int D, int M, int F, int dtype) {
  return dtype == LA_BF16 && D == 64 && M == 64 && F == 64;
}

// la_forward's workspace (its status header first), then the two feature buffers
// (bf16 [BH][N][F])
size_t rff_workspace(int BH, int N) {
  return tc_forward_workspace(BH, N) + 2 * align_up(sizeof(__nv_bfloat16) * (size_t)BH * N * kDim, 256);
}

cudaError_t rff_forward(const void* q, const void* k, const void* v, const void* W,
                        const float* bias, void* out, int BH, int N, bool causal, void* ws,
                        cudaStream_t st) {
  char* base = static_cast<char*>(ws);
  const size_t fb = align_up(sizeof(__nv_bfloat16) * (size_t)BH * N * kDim, 256);
  void* fws = base;
  void* fq = base + tc_forward_workspace(BH, N);
  void* fk = static_cast<char*>(fq) + fb;
  WorkspaceHeader* hdr = static_cast<WorkspaceHeader*>(fws);
  CUtensorMap tq, tk, tw, tfq, tfk;
  const uint64_t n = (uint64_t)N, bh = (uint64_t)BH;
  if (!make_tmap_bf16_3d(&tq, q, kDim, n, bh, kDim, kC, 1) ||
      !make_tmap_bf16_3d(&tk, k, kDim, n, bh, kDim, kC, 1) ||
      !make_tmap_bf16_3d(&tw, W, kDim, kDim, 1, kDim, kDim, 1) ||
      !make_tmap_bf16_3d(&tfq, fq, kDim, n, bh, kDim, kC, 1) ||
      !make_tmap_bf16_3d(&tfk, fk, kDim, n, bh, kDim, kC, 1))
    return cudaErrorInvalidValue;
  cudaError_t e = configure(tc_rff_feature_kernel, kRffSmem);
  if (e != cudaSuccess) return e;
  const int tiles = BH * ((N + kC - 1) / kC);
  e = launch_pdl(tc_rff_feature_kernel, dim3(2 * tiles), dim3(kRffThreads), kRffSmem, st, tq, tk, tw,
                 tfq, tfk, bias, N, tiles, hdr);
  count_launches(1);
  if (e != cudaSuccess) return e;
  return tc_forward(fq, fk, v, out, StateIO{}, BH, N, causal, fws, st, nullptr, true);
}

}  // namespace la
