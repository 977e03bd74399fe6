// C-ABI entry points: argument validation and kernel selection.
//
// Every entry point validates its arguments on the host, launches on the
// caller's stream and returns a status; nothing is allocated, synchronised or
// thrown across the boundary.
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <initializer_list>

#include "la_common.cuh"
#include "la_internal.h"

namespace la {
namespace {
std::atomic<unsigned long long> g_launches{0};
}
void count_launches(unsigned n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
}  // namespace la

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool valid_dims(int B, int H, int N, int D, int M) {
  if (B < 1 || H < 1 || N < 0) return false;
  if (D < 8 || D > 128 || (D % 8) != 0) return false;
  if (M < 8 || M > 128 || (M % 8) != 0) return false;
  // element offsets are formed in 64-bit; keep B*H inside a grid dimension
  if ((long long)B * H > 0x7fffffffLL) return false;
  return true;
}

bool valid_dtype(int dtype) { return dtype == LA_F32 || dtype == LA_BF16; }

// Workspace queries: shapes that the entry points reject (including B * H
// beyond an int) need only the header.
bool query_dims_ok(int B, int H, int N) {
  return B >= 1 && H >= 1 && N >= 0 && (long long)B * H <= 0x7fffffffLL;
}

bool ptrs_ok(std::initializer_list<const void*> ps) {
  for (const void* p : ps)
    if (p == nullptr || !aligned16(p)) return false;
  return true;
}

int from_cuda(cudaError_t e) { return e == cudaSuccess ? LA_OK : LA_ERR_CUDA; }

cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// The caller's workspace arrives with arbitrary contents: clear its header
// (status word, wait site) on the stream before any kernel reads it.
cudaError_t clear_header(void* ws, cudaStream_t st) {
  return cudaMemsetAsync(ws, 0, la::kHeaderBytes, st);
}

}  // namespace

extern "C" {

const char* la_status_string(int status) {
  switch (status) {
    case LA_OK: return "ok";
    case LA_ERR_INVALID_ARG:
      return "invalid argument (null or misaligned pointer, bad dimension, or unsupported D/M/dtype)";
    case LA_ERR_WORKSPACE: return "workspace missing or too small";
    case LA_ERR_CUDA: return "CUDA runtime error";
    case LA_ERR_TIMEOUT: return "a bounded wait inside a kernel expired; outputs are invalid";
    case LA_ERR_TOO_LARGE:
      return "problem needs more scratch than la_forward_noalloc's fixed array holds";
    default: return "unknown status";
  }
}

int la_version(void) { return 100; }

unsigned long long la_kernel_launches(void) {
  return la::g_launches.load(std::memory_order_relaxed);
}

size_t la_forward_workspace_bytes(int B, int H, int N, int D, int M, int causal, int dtype) {
  (void)causal;
  if (!query_dims_ok(B, H, N)) return la::kHeaderBytes;
  if (la::tc_forward_supported(D, M, dtype)) return la::tc_forward_workspace(B * H, N);
  return la::kHeaderBytes;
}

int la_forward(const void* q, const void* k, const void* v, void* out, int B, int H, int N, int D,
               int M, int causal, int dtype, void* workspace, size_t workspace_bytes,
               void* stream) {
  if (!valid_dims(B, H, N, D, M) || !valid_dtype(dtype)) return LA_ERR_INVALID_ARG;
  if (N == 0) return LA_OK;
  if (!ptrs_ok({q, k, v, out})) return LA_ERR_INVALID_ARG;
  const size_t need = la_forward_workspace_bytes(B, H, N, D, M, causal, dtype);
  if (workspace == nullptr || !aligned16(workspace) || workspace_bytes < need)
    return LA_ERR_WORKSPACE;
  cudaStream_t st = as_stream(stream);
  cudaError_t e = clear_header(workspace, st);
  if (e != cudaSuccess) return LA_ERR_CUDA;
  if (la::tc_forward_supported(D, M, dtype))
    return from_cuda(la::tc_forward(q, k, v, out, la::StateIO{}, B * H, N, causal != 0,
                                    workspace, st));
  return from_cuda(la::simt_forward(q, k, v, out, la::StateIO{}, B * H, N, D, M, causal != 0,
                                    dtype, static_cast<la::WorkspaceHeader*>(workspace), st));
}

int la_prefill(const void* q, const void* k, const void* v, void* out, float* S, float* Z, int B,
               int H, int N, int D, int M, int dtype, void* workspace, size_t workspace_bytes,
               void* stream) {
  if (!valid_dims(B, H, N, D, M) || !valid_dtype(dtype)) return LA_ERR_INVALID_ARG;
  if (!ptrs_ok({S, Z})) return LA_ERR_INVALID_ARG;
  if (N == 0) {
    cudaStream_t st = as_stream(stream);
    cudaError_t e = cudaMemsetAsync(S, 0, sizeof(float) * (size_t)B * H * D * M, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(Z, 0, sizeof(float) * (size_t)B * H * D, st);
    return from_cuda(e);
  }
  if (!ptrs_ok({q, k, v, out})) return LA_ERR_INVALID_ARG;
  const size_t need = la_forward_workspace_bytes(B, H, N, D, M, 1, dtype);
  if (workspace == nullptr || !aligned16(workspace) || workspace_bytes < need)
    return LA_ERR_WORKSPACE;
  cudaStream_t st = as_stream(stream);
  cudaError_t e = clear_header(workspace, st);
  if (e != cudaSuccess) return LA_ERR_CUDA;
  la::StateIO io;
  io.S = S;
  io.Z = Z;
  io.H = H;
  io.pool = B;
  if (la::tc_forward_supported(D, M, dtype))
    return from_cuda(la::tc_forward(q, k, v, out, io, B * H, N, true, workspace, st));
  return from_cuda(la::simt_forward(q, k, v, out, io, B * H, N, D, M, true, dtype,
                                    static_cast<la::WorkspaceHeader*>(workspace), st));
}

int la_extend(const void* q, const void* k, const void* v, void* out, float* S_pool,
              float* Z_pool, const int* slots, const int* lens, int pool_size, int B, int H,
              int N, int D, int M, int dtype, void* workspace, size_t workspace_bytes,
              void* stream) {
  if (!valid_dims(B, H, N, D, M) || !valid_dtype(dtype)) return LA_ERR_INVALID_ARG;
  if (!ptrs_ok({S_pool, Z_pool})) return LA_ERR_INVALID_ARG;
  if (slots == nullptr ? pool_size < B : pool_size < 1) return LA_ERR_INVALID_ARG;
  if (slots != nullptr && (reinterpret_cast<uintptr_t>(slots) & 3u) != 0) return LA_ERR_INVALID_ARG;
  if (lens != nullptr && (reinterpret_cast<uintptr_t>(lens) & 3u) != 0) return LA_ERR_INVALID_ARG;
  if (N == 0) return LA_OK;
  if (!ptrs_ok({q, k, v, out})) return LA_ERR_INVALID_ARG;
  const size_t need = la_forward_workspace_bytes(B, H, N, D, M, 1, dtype);
  if (workspace == nullptr || !aligned16(workspace) || workspace_bytes < need)
    return LA_ERR_WORKSPACE;
  cudaStream_t st = as_stream(stream);
  cudaError_t e = clear_header(workspace, st);
  if (e != cudaSuccess) return LA_ERR_CUDA;
  la::StateIO io;
  io.S = S_pool;
  io.Z = Z_pool;
  io.slots = slots;
  io.H = H;
  io.pool = pool_size;
  io.read_init = true;
  io.lens = lens;
  if (la::tc_forward_supported(D, M, dtype))
    return from_cuda(la::tc_forward(q, k, v, out, io, B * H, N, true, workspace, st));
  return from_cuda(la::simt_forward(q, k, v, out, io, B * H, N, D, M, true, dtype,
                                    static_cast<la::WorkspaceHeader*>(workspace), st));
}

int la_extend_packed(const void* q, const void* k, const void* v, void* out, float* S_pool,
                     float* Z_pool, const int* slots, const int* cu_seqlens, int pool_size, int B,
                     int H, int total_tokens, int max_len, int D, int M, int dtype,
                     void* workspace, size_t workspace_bytes, void* stream) {
  if (B <= 0 || H <= 0 || max_len < 0 || total_tokens < 0 || total_tokens > (1 << 30))
    return LA_ERR_INVALID_ARG;
  if (!valid_dims(B, H, max_len, D, M) || !valid_dtype(dtype)) return LA_ERR_INVALID_ARG;
  if (!ptrs_ok({S_pool, Z_pool}) || cu_seqlens == nullptr) return LA_ERR_INVALID_ARG;
  if (slots == nullptr ? pool_size < B : pool_size < 1) return LA_ERR_INVALID_ARG;
  if (slots != nullptr && (reinterpret_cast<uintptr_t>(slots) & 3u) != 0) return LA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(cu_seqlens) & 3u) != 0) return LA_ERR_INVALID_ARG;
  if (max_len == 0 || total_tokens == 0) return LA_OK;
  if (!ptrs_ok({q, k, v, out})) return LA_ERR_INVALID_ARG;
  const size_t need = la_forward_workspace_bytes(B, H, max_len, D, M, 1, dtype);
  if (workspace == nullptr || !aligned16(workspace) || workspace_bytes < need)
    return LA_ERR_WORKSPACE;
  cudaStream_t st = as_stream(stream);
  cudaError_t e = clear_header(workspace, st);
  if (e != cudaSuccess) return LA_ERR_CUDA;
  la::StateIO io;
  io.S = S_pool;
  io.Z = Z_pool;
  io.slots = slots;
  io.H = H;
  io.pool = pool_size;
  io.read_init = true;
  io.cu = cu_seqlens;
  io.T = total_tokens;
  if (la::tc_forward_supported(D, M, dtype))
    return from_cuda(la::tc_forward(q, k, v, out, io, B * H, max_len, true, workspace, st));
  return from_cuda(la::simt_forward(q, k, v, out, io, B * H, max_len, D, M, true, dtype,
                                    static_cast<la::WorkspaceHeader*>(workspace), st));
}

size_t la_backward_workspace_bytes(int B, int H, int N, int D, int M, int causal, int dtype) {
  (void)causal;
  if (!query_dims_ok(B, H, N)) return la::kHeaderBytes;
  if (la::tc_forward_supported(D, M, dtype)) return la::tc_backward_workspace(B * H, N);
  return la::simt_backward_workspace(B * H, N);
}

int la_backward(const void* q, const void* k, const void* v, const void* dout, float* dq,
                float* dk, float* dv, int B, int H, int N, int D, int M, int causal, int dtype,
                void* workspace, size_t workspace_bytes, void* stream) {
  if (!valid_dims(B, H, N, D, M) || !valid_dtype(dtype)) return LA_ERR_INVALID_ARG;
  if (N == 0) return LA_OK;
  if (!ptrs_ok({q, k, v, dout, dq, dk, dv})) return LA_ERR_INVALID_ARG;
  const size_t need = la_backward_workspace_bytes(B, H, N, D, M, causal, dtype);
  if (workspace == nullptr || !aligned16(workspace) || workspace_bytes < need)
    return LA_ERR_WORKSPACE;
  cudaStream_t st = as_stream(stream);
  cudaError_t e = clear_header(workspace, st);
  if (e != cudaSuccess) return LA_ERR_CUDA;
  if (la::tc_forward_supported(D, M, dtype))
    return from_cuda(la::tc_backward(q, k, v, dout, dq, dk, dv, B * H, N, causal != 0, workspace,
                                     st));
  return from_cuda(la::simt_backward(q, k, v, dout, dq, dk, dv, B * H, N, D, M, causal != 0,
                                     dtype, workspace, st));
}

// ---------------------------------------------- degree-2 polynomial feature map

size_t la_poly2_workspace_bytes(int B, int H, int N, int D, int M, int causal, int dtype) {
  if (!query_dims_ok(B, H, N) || !la::poly2_supported(D, M, dtype, causal)) return la::kHeaderBytes;
  return la::poly2_workspace(B * H, N);
}

int la_forward_poly2(const void* q, const void* k, const void* v, void* out, int B, int H, int N,
                     int D, int M, int causal, int dtype, void* workspace, size_t workspace_bytes,
                     void* stream) {
  if (!valid_dims(B, H, N, D, M) || !valid_dtype(dtype)) return LA_ERR_INVALID_ARG;
  if (!la::poly2_supported(D, M, dtype, causal)) return LA_ERR_INVALID_ARG;
  if (N == 0) return LA_OK;
  if (!ptrs_ok({q, k, v, out})) return LA_ERR_INVALID_ARG;
  const size_t need = la_poly2_workspace_bytes(B, H, N, D, M, causal, dtype);
  if (workspace == nullptr || !aligned16(workspace) || workspace_bytes < need)
    return LA_ERR_WORKSPACE;
  cudaStream_t st = as_stream(stream);
  if (clear_header(workspace, st) != cudaSuccess) return LA_ERR_CUDA;
  return from_cuda(la::poly2_forward(q, k, v, out, B * H, N, workspace, st));
}

// ------------------------------------------------------ random Fourier features

size_t la_rff_workspace_bytes(int B, int H, int N, int D, int M, int F, int causal, int dtype) {
  (void)causal;
  if (!query_dims_ok(B, H, N) || !la::rff_supported(D, M, F, dtype)) return la::kHeaderBytes;
  return la::rff_workspace(B * H, N);
}

int la_forward_rff(const void* q, const void* k, const void* v, const void* W, const float* bias,
                   void* out, int B, int H, int N, int D, int M, int F, int causal, int dtype,
                   void* workspace, size_t workspace_bytes, void* stream) {
  if (!valid_dims(B, H, N, D, M) || !valid_dtype(dtype)) return LA_ERR_INVALID_ARG;
  if (!la::rff_supported(D, M, F, dtype)) return LA_ERR_INVALID_ARG;
  if (N == 0) return LA_OK;
  if (!ptrs_ok({q, k, v, W, bias, out})) return LA_ERR_INVALID_ARG;
  const size_t need = la_rff_workspace_bytes(B, H, N, D, M, F, causal, dtype);
  if (workspace == nullptr || !aligned16(workspace) || workspace_bytes < need)
    return LA_ERR_WORKSPACE;
  cudaStream_t st = as_stream(stream);
  if (clear_header(workspace, st) != cudaSuccess) return LA_ERR_CUDA;
  return from_cuda(la::rff_forward(q, k, v, W, bias, out, B * H, N, causal != 0, workspace, st));
}

// ------------------------------------------------------- sequence shards

namespace {

// (S, Z)-shaped state entries [B][H][D][M], [B][H][D] of a shard call, entry bh.
la::StateIO shard_io(float* S, float* Z, int B, int H, bool read_init, bool write_final) {
  la::StateIO io;
  io.S = S;
  io.Z = Z;
  io.H = H;
  io.pool = B;
  io.read_init = read_init;
  io.write_final = write_final;
  return io;
}

}  // namespace

int la_state_sums(const void* k, const void* v, float* S, float* Z, int B, int H, int N, int D,
                  int M, int dtype, void* workspace, size_t workspace_bytes, void* stream) {
  if (!valid_dims(B, H, N, D, M) || !valid_dtype(dtype)) return LA_ERR_INVALID_ARG;
  if (!ptrs_ok({S, Z})) return LA_ERR_INVALID_ARG;
  cudaStream_t st = as_stream(stream);
  if (N == 0) {
    cudaError_t e = cudaMemsetAsync(S, 0, sizeof(float) * (size_t)B * H * D * M, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(Z, 0, sizeof(float) * (size_t)B * H * D, st);
    return from_cuda(e);
  }
  if (!ptrs_ok({k, v})) return LA_ERR_INVALID_ARG;
  const size_t need = la_forward_workspace_bytes(B, H, N, D, M, 1, dtype);
  if (workspace == nullptr || !aligned16(workspace) || workspace_bytes < need)
    return LA_ERR_WORKSPACE;
  if (clear_header(workspace, st) != cudaSuccess) return LA_ERR_CUDA;
  const la::StateIO io = shard_io(S, Z, B, H, false, true);
  if (la::tc_forward_supported(D, M, dtype))
    return from_cuda(la::tc_state_sums(k, v, io, B * H, N, workspace, st));
  return from_cuda(la::simt_state_sums(k, v, io, B * H, N, D, M, dtype, st));
}

int la_forward_shard(const void* q, const void* k, const void* v, void* out, const float* S0,
                     const float* Z0, int B, int H, int N, int D, int M, int dtype,
                     void* workspace, size_t workspace_bytes, void* stream) {
  if (!valid_dims(B, H, N, D, M) || !valid_dtype(dtype)) return LA_ERR_INVALID_ARG;
  if (!ptrs_ok({S0, Z0})) return LA_ERR_INVALID_ARG;
  if (N == 0) return LA_OK;
  if (!ptrs_ok({q, k, v, out})) return LA_ERR_INVALID_ARG;
  const size_t need = la_forward_workspace_bytes(B, H, N, D, M, 1, dtype);
  if (workspace == nullptr || !aligned16(workspace) || workspace_bytes < need)
    return LA_ERR_WORKSPACE;
  cudaStream_t st = as_stream(stream);
  if (clear_header(workspace, st) != cudaSuccess) return LA_ERR_CUDA;
  // the entries are read, never written (the kernels take them through const-free
  // pointers but write only when write_final is set)
  const la::StateIO io = shard_io(const_cast<float*>(S0), const_cast<float*>(Z0), B, H, true, false);
  if (la::tc_forward_supported(D, M, dtype))
    return from_cuda(la::tc_forward(q, k, v, out, io, B * H, N, true, workspace, st));
  return from_cuda(la::simt_forward(q, k, v, out, io, B * H, N, D, M, true, dtype,
                                    static_cast<la::WorkspaceHeader*>(workspace), st));
}

int la_backward_shard_q(const void* q, const void* k, const void* v, const void* dout, float* dq,
                        const float* S0, const float* Z0, float* R_own, float* r_own, int B, int H,
                        int N, int D, int M, int dtype, void* workspace, size_t workspace_bytes,
                        void* stream) {
  if (!valid_dims(B, H, N, D, M) || !valid_dtype(dtype)) return LA_ERR_INVALID_ARG;
  if (!ptrs_ok({S0, Z0, R_own, r_own})) return LA_ERR_INVALID_ARG;
  cudaStream_t st = as_stream(stream);
  if (N == 0) {  // no tokens: the shard adds nothing to the reverse sums
    cudaError_t e = cudaMemsetAsync(R_own, 0, sizeof(float) * (size_t)B * H * D * M, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(r_own, 0, sizeof(float) * (size_t)B * H * D, st);
    return from_cuda(e);
  }
  if (!ptrs_ok({q, k, v, dout, dq})) return LA_ERR_INVALID_ARG;
  const size_t need = la_backward_workspace_bytes(B, H, N, D, M, 1, dtype);
  if (workspace == nullptr || !aligned16(workspace) || workspace_bytes < need)
    return LA_ERR_WORKSPACE;
  if (clear_header(workspace, st) != cudaSuccess) return LA_ERR_CUDA;
  const la::StateIO pre = shard_io(const_cast<float*>(S0), const_cast<float*>(Z0), B, H, true, false);
  la::StateIO own = shard_io(R_own, r_own, B, H, false, true);
  own.rows_are_d = true;
  if (la::tc_forward_supported(D, M, dtype))
    return from_cuda(la::tc_backward_q(q, k, v, dout, dq, &pre, &own, B * H, N, true, workspace,
                                       st));
  return from_cuda(la::simt_backward_q(q, k, v, dout, dq, &pre, &own, B * H, N, D, M, true,
                                       dtype, workspace, st));
}

int la_backward_shard_kv(const void* q, const void* k, const void* v, const void* dout, float* dk,
                         float* dv, const float* R0, const float* r0, int B, int H, int N, int D,
                         int M, int dtype, void* workspace, size_t workspace_bytes, void* stream) {
  if (!valid_dims(B, H, N, D, M) || !valid_dtype(dtype)) return LA_ERR_INVALID_ARG;
  if (!ptrs_ok({R0, r0})) return LA_ERR_INVALID_ARG;
  if (N == 0) return LA_OK;
  if (!ptrs_ok({q, k, v, dout, dk, dv})) return LA_ERR_INVALID_ARG;
  const size_t need = la_backward_workspace_bytes(B, H, N, D, M, 1, dtype);
  if (workspace == nullptr || !aligned16(workspace) || workspace_bytes < need)
    return LA_ERR_WORKSPACE;
  cudaStream_t st = as_stream(stream);
  // the header is not cleared: the status of the dq pass stays visible
  la::StateIO suf = shard_io(const_cast<float*>(R0), const_cast<float*>(r0), B, H, true, false);
  suf.rows_are_d = true;
  if (la::tc_forward_supported(D, M, dtype))
    return from_cuda(la::tc_backward_kv(q, k, v, dout, dk, dv, &suf, B * H, N, true, workspace,
                                        st));
  return from_cuda(la::simt_backward_kv(q, k, v, dout, dk, dv, &suf, B * H, N, D, M, true, dtype,
                                        workspace, st));
}

int la_backward_from_forward(const void* q, const void* k, const void* v, const void* dout,
                             float* dq, float* dk, float* dv, int B, int H, int N, int D, int M,
                             int causal, int dtype, const void* fwd_workspace,
                             size_t fwd_workspace_bytes, void* workspace, size_t workspace_bytes,
                             void* stream) {
  if (!valid_dims(B, H, N, D, M) || !valid_dtype(dtype)) return LA_ERR_INVALID_ARG;
  if (N == 0) return LA_OK;
  if (!ptrs_ok({q, k, v, dout, dq, dk, dv})) return LA_ERR_INVALID_ARG;
  const size_t need = la_backward_workspace_bytes(B, H, N, D, M, causal, dtype);
  if (workspace == nullptr || !aligned16(workspace) || workspace_bytes < need)
    return LA_ERR_WORKSPACE;
  const size_t need_fwd = la_forward_workspace_bytes(B, H, N, D, M, causal, dtype);
  if (fwd_workspace == nullptr || !aligned16(fwd_workspace) || fwd_workspace_bytes < need_fwd)
    return LA_ERR_WORKSPACE;
  cudaStream_t st = as_stream(stream);
  if (clear_header(workspace, st) != cudaSuccess) return LA_ERR_CUDA;
  if (!la::tc_forward_supported(D, M, dtype))  // the CUDA-core path keeps no forward states
    return from_cuda(la::simt_backward(q, k, v, dout, dq, dk, dv, B * H, N, D, M, causal != 0,
                                       dtype, workspace, st));
  const float* pre = la::tc_forward_prefix(fwd_workspace, B * H, N, causal != 0);
  cudaError_t e = la::tc_backward_q(q, k, v, dout, dq, nullptr, nullptr, B * H, N, causal != 0,
                                    workspace, st, nullptr, pre);
  if (e != cudaSuccess) return LA_ERR_CUDA;
  return from_cuda(la::tc_backward_kv(q, k, v, dout, dk, dv, nullptr, B * H, N, causal != 0,
                                      workspace, st));
}

int la_decode_step(const void* q, const void* k, const void* v, float* S, float* Z, void* out,
                   int n_streams, int H, int D, int M, int dtype, void* stream) {
  if (!valid_dims(n_streams, H, 1, D, M) || !valid_dtype(dtype)) return LA_ERR_INVALID_ARG;
  if (!ptrs_ok({q, k, v, S, Z, out})) return LA_ERR_INVALID_ARG;
  return from_cuda(la::decode_step(q, k, v, S, Z, out, n_streams * H, D, M, dtype,
                                   as_stream(stream)));
}

namespace {

// Shared by the two failure test hooks: the tensor-core path only, a withheld
// load number >= 0 and a wait limit between 1 us and the normal 2 s.
bool fault_args_ok(int D, int M, int dtype, int withhold_load, unsigned long long wait_ns) {
  return la::tc_forward_supported(D, M, dtype) && withhold_load >= 0 && wait_ns >= 1000ull &&
         wait_ns <= 2000000000ull;
}

}  // namespace

int la_debug_forward_fault(const void* q, const void* k, const void* v, void* out, int B, int H,
                           int N, int D, int M, int causal, int dtype, void* workspace,
                           size_t workspace_bytes, int withhold_load,
                           unsigned long long wait_limit_ns, void* stream) {
  if (!valid_dims(B, H, N, D, M) || !valid_dtype(dtype) || N == 0) return LA_ERR_INVALID_ARG;
  if (!fault_args_ok(D, M, dtype, withhold_load, wait_limit_ns)) return LA_ERR_INVALID_ARG;
  if (!ptrs_ok({q, k, v, out})) return LA_ERR_INVALID_ARG;
  const size_t need = la_forward_workspace_bytes(B, H, N, D, M, causal, dtype);
  if (workspace == nullptr || !aligned16(workspace) || workspace_bytes < need)
    return LA_ERR_WORKSPACE;
  cudaStream_t st = as_stream(stream);
  if (clear_header(workspace, st) != cudaSuccess) return LA_ERR_CUDA;
  la::FaultHook fh;
  fh.load = withhold_load;
  fh.wait_ns = wait_limit_ns;
  return from_cuda(la::tc_forward(q, k, v, out, la::StateIO{}, B * H, N, causal != 0, workspace,
                                  st, &fh));
}

int la_debug_forward_fused_fault(const void* q, const void* k, const void* v, void* out, int B,
                                 int H, int N, int D, int M, int causal, int dtype,
                                 void* workspace, size_t workspace_bytes, int withhold_load,
                                 unsigned long long wait_limit_ns, void* stream) {
  if (!valid_dims(B, H, N, D, M) || !valid_dtype(dtype) || N == 0) return LA_ERR_INVALID_ARG;
  if (!fault_args_ok(D, M, dtype, withhold_load, wait_limit_ns)) return LA_ERR_INVALID_ARG;
  if (!ptrs_ok({q, k, v, out})) return LA_ERR_INVALID_ARG;
  const size_t need = la_forward_workspace_bytes(B, H, N, D, M, causal, dtype);
  if (workspace == nullptr || !aligned16(workspace) || workspace_bytes < need)
    return LA_ERR_WORKSPACE;
  cudaStream_t st = as_stream(stream);
  if (clear_header(workspace, st) != cudaSuccess) return LA_ERR_CUDA;
  la::FaultHook fh;
  fh.load = withhold_load;
  fh.wait_ns = wait_limit_ns;
  fh.fused = true;
  return from_cuda(la::tc_forward(q, k, v, out, la::StateIO{}, B * H, N, causal != 0, workspace,
                                  st, &fh));
}

int la_debug_backward_fault(const void* q, const void* k, const void* v, const void* dout,
                            float* dq, float* dk, float* dv, int B, int H, int N, int D, int M,
                            int causal, int dtype, void* workspace, size_t workspace_bytes,
                            int withhold_load, unsigned long long wait_limit_ns, void* stream) {
  if (!valid_dims(B, H, N, D, M) || !valid_dtype(dtype) || N == 0) return LA_ERR_INVALID_ARG;
  if (!fault_args_ok(D, M, dtype, withhold_load, wait_limit_ns)) return LA_ERR_INVALID_ARG;
  if (!ptrs_ok({q, k, v, dout, dq, dk, dv})) return LA_ERR_INVALID_ARG;
  const size_t need = la_backward_workspace_bytes(B, H, N, D, M, causal, dtype);
  if (workspace == nullptr || !aligned16(workspace) || workspace_bytes < need)
    return LA_ERR_WORKSPACE;
  cudaStream_t st = as_stream(stream);
  if (clear_header(workspace, st) != cudaSuccess) return LA_ERR_CUDA;
  la::FaultHook fh;
  fh.load = withhold_load;
  fh.wait_ns = wait_limit_ns;
  return from_cuda(la::tc_backward(q, k, v, dout, dq, dk, dv, B * H, N, causal != 0, workspace,
                                   st, &fh));
}

int la_workspace_wait_site(void* workspace, size_t workspace_bytes, void* stream) {
  if (workspace == nullptr || workspace_bytes < la::kHeaderBytes) return -1;
  cudaStream_t st = as_stream(stream);
  la::WorkspaceHeader h;
  cudaError_t e = cudaMemcpyAsync(&h, workspace, sizeof(h), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return -1;
  return h.wait_site;
}

int la_workspace_status(void* workspace, size_t workspace_bytes, void* stream) {
  if (workspace == nullptr || workspace_bytes < la::kHeaderBytes) return LA_ERR_WORKSPACE;
  cudaStream_t st = as_stream(stream);
  la::WorkspaceHeader h;
  cudaError_t e = cudaMemcpyAsync(&h, workspace, sizeof(h), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return LA_ERR_CUDA;
  if (h.status != LA_OK) {
    const int zero = 0;
    e = cudaMemcpyAsync(workspace, &zero, sizeof(zero), cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return LA_ERR_CUDA;
    return (h.status == LA_ERR_TIMEOUT || h.status == LA_ERR_INVALID_ARG) ? h.status : LA_ERR_CUDA;
  }
  return LA_OK;
}

}  // extern "C"
