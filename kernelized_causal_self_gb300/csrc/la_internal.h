// Launchers shared between the C-ABI layer and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

#include "la_common.cuh"

namespace la {

// Where a causal forward takes its initial state and leaves its final state:
// S [entries][D][M] and Z [entries][D] float32, sequence bh = b * H + h at entry
// slots[b] * H + h (slots == nullptr: entry bh). read_init: start from the
// entry's contents (and overwrite them in place), else start from zero.
// Entries of slots outside [0, pool) skip that sequence's state and set the
// workspace status word to LA_ERR_INVALID_ARG.
struct StateIO {
  float* S = nullptr;
  float* Z = nullptr;
  const int* slots = nullptr;
  int H = 1;
  int pool = 0;
  bool read_init = false;
  // per-stream token counts (device int[B], each clamped to [0, N]); nullptr: all N
  const int* lens = nullptr;
  // packed token-major layout [T][H][D] (tensor-core forward, CUDA-core forward):
  // stream b holds rows cu[b] .. cu[b + 1] - 1 (device int[B + 1]); nullptr: [BH][N][D]
  const int* cu = nullptr;
  int T = 0;
  // write the final state back to the entries (prefill, extend); false: the
  // entries are read-only initial states (sequence shards)
  bool write_final = true;
  // (scans of the backward's reverse sums) the per-segment sums are R [d][m]
  // rather than S^T [m][d]; the entries are [D][M] either way
  bool rows_are_d = false;
};

// Test hook of the failure-detection tests (la_debug_forward_fault,
// la_debug_backward_fault): CTA 0 of the call's main kernel (the forward's chunk
// attention, the backward's forward-direction kernel) withholds its TMA load
// number `load` and bounds its main-loop waits by `wait_ns`. load < 0: off.
struct FaultHook {
  int load = -1;
  unsigned long long wait_ns = 0;
  // run the one-launch (cluster) forward where the shape allows it, rather than the
  // segment-state, scan and attention kernels
  bool fused = false;
};

// Adds n to the process-wide kernel launch count reported by la_kernel_launches().
void count_launches(unsigned n);

// ---- general-shape CUDA-core path (any dtype, D and M multiples of 8 up to 128)
cudaError_t simt_forward(const void* q, const void* k, const void* v, void* out,
                         const StateIO& io, int BH, int N, int D, int M, bool causal, int dtype,
                         WorkspaceHeader* hdr, cudaStream_t st);
size_t simt_backward_workspace(int BH, int N);
cudaError_t simt_backward(const void* q, const void* k, const void* v, const void* dout, float* dq,
                          float* dk, float* dv, int BH, int N, int D, int M, bool causal,
                          int dtype, void* ws, cudaStream_t st);

// state sums of each sequence: S = sum_j phi(k_j) v_j^T, Z = sum_j phi(k_j) into io's
// entries (general shapes)
cudaError_t simt_state_sums(const void* k, const void* v, const StateIO& io, int BH, int N, int D,
                            int M, int dtype, cudaStream_t st);
// backward of sequence shards on the CUDA-core path: the dq pass from the prefix state in
// `pre` (S, Z entries, read-only; nullptr: zero) writing the shard's own reverse sums into
// `own` (R, r entries; nullptr: not written), and the dk/dv pass from the suffix sums in
// `suf` (nullptr: zero). The workspace carries den_i, gd_i from the first to the second.
cudaError_t simt_backward_q(const void* q, const void* k, const void* v, const void* dout,
                            float* dq, const StateIO* pre, const StateIO* own, int BH, int N,
                            int D, int M, bool causal, int dtype, void* ws, cudaStream_t st);
cudaError_t simt_backward_kv(const void* q, const void* k, const void* v, const void* dout,
                             float* dk, float* dv, const StateIO* suf, int BH, int N, int D,
                             int M, bool causal, int dtype, void* ws, cudaStream_t st);

// ---- tensor-core path (bf16, D = M = 64): tcgen05 + TMEM + TMA
bool tc_forward_supported(int D, int M, int dtype);
size_t tc_forward_workspace(int BH, int N);
// identity: q and k hold features already (the identity feature map), else elu + 1 applies.
cudaError_t tc_forward(const void* q, const void* k, const void* v, void* out, const StateIO& io,
                       int BH, int N, bool causal, void* ws, cudaStream_t st,
                       const FaultHook* fault = nullptr, bool identity = false);
cudaError_t tc_state_sums(const void* k, const void* v, const StateIO& io, int BH, int N, void* ws,
                          cudaStream_t st);
size_t tc_backward_workspace(int BH, int N);
// The backward in its two passes (see simt_backward_q / simt_backward_kv); tc_backward
// runs both from zero states.
cudaError_t tc_backward_q(const void* q, const void* k, const void* v, const void* dout,
                          float* dq, const StateIO* pre, const StateIO* own, int BH, int N,
                          bool causal, void* ws, cudaStream_t st, const FaultHook* fault = nullptr,
                          const float* fwd_prefix = nullptr);
// The per-segment states a tensor-core la_forward call left in its workspace (causal:
// exclusive prefixes; non-causal: totals), laid out as the backward reads them (both use
// make_geometry(BH, N)); nullptr if that forward computed none (one chunk per sequence).
const float* tc_forward_prefix(const void* fwd_ws, int BH, int N, bool causal);
cudaError_t tc_backward_kv(const void* q, const void* k, const void* v, const void* dout,
                           float* dk, float* dv, const StateIO* suf, int BH, int N, bool causal,
                           void* ws, cudaStream_t st);
cudaError_t tc_backward(const void* q, const void* k, const void* v, const void* dout, float* dq,
                        float* dk, float* dv, int BH, int N, bool causal, void* ws,
                        cudaStream_t st, const FaultHook* fault = nullptr);

// ---- degree-2 polynomial feature map (bf16, D = M = 64, causal): tcgen05 + TMEM + TMA
bool poly2_supported(int D, int M, int dtype, int causal);
size_t poly2_workspace(int BH, int N);
cudaError_t poly2_forward(const void* q, const void* k, const void* v, void* out, int BH, int N,
                          void* ws, cudaStream_t st);

// ---- random Fourier features (bf16, D = M = F = 64): features on tcgen05, then the
// identity-feature forward
bool rff_supported(int D, int M, int F, int dtype);
size_t rff_workspace(int BH, int N);
cudaError_t rff_forward(const void* q, const void* k, const void* v, const void* W,
                        const float* bias, void* out, int BH, int N, bool causal, void* ws,
                        cudaStream_t st);

// ---- decode step (memory-bound CUDA-core kernel)
cudaError_t decode_step(const void* q, const void* k, const void* v, float* S, float* Z, void* out,
                        int n_sh, int D, int M, int dtype, cudaStream_t st);

}  // namespace la
