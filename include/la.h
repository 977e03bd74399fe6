/*
 * la.h -- C ABI of the GB300 (sm_103a) kernelized linear-attention library.
 *
 * Method: "Transformers are RNNs: Fast Autoregressive Transformers with
 * Linear Attention" (Katharopoulos et al., ICML 2020), as summarised on the
 * pages cited per entry point below:
 *   [review]  "[Paper Review] Transformers are RNNs ..." (nubint.ai), "Proposed method"
 *   [summary] "Transformers are RNNs: Fast Autoregressive Transformers with
 *             Linear Attention" (paperlayer.ai), paper sections 3.1-3.4, App. A
 *   [deck]    "Transformers are RNNs ... 解读" (zhengyuhong.cn), slides 3-4
 *
 * phi(x) = elu(x) + 1 (ELU alpha = 1): x + 1 for x > 0, exp(x) otherwise.
 * No 1/sqrt(D) scale and no epsilon are applied inside the operator.
 *
 * Layouts (all row-major, contiguous, no padding):
 *   q, k        [B][H][N][D]      element type `dtype`
 *   v, out      [B][H][N][M]      element type `dtype`
 *   dout        [B][H][N][M]      element type `dtype`
 *   dq, dk      [B][H][N][D]      float32
 *   dv          [B][H][N][M]      float32
 *   S           [B][H][D][M]      float32  (attention memory, S[d][m])
 *   Z           [B][H][D]         float32  (normalizer memory)
 *   decode q,k  [n_streams][H][D], decode v,out [n_streams][H][M]
 *
 * Ownership and threading: every pointer is device memory owned by the
 * caller; the library never allocates, frees or synchronises. All calls are
 * asynchronous on `stream` (a cudaStream_t passed as void*, NULL = legacy
 * default stream). The only process-wide state is an atomic count of kernel
 * launches (la_kernel_launches), so calls from several host threads are safe.
 * Outputs must not alias inputs (S and Z of la_decode_step are updated in
 * place by design).
 *
 * Supported shapes: B, H >= 1; N >= 0 (N == 0 is a no-op); D and M multiples
 * of 8 in [8, 128]; pointers 16-byte aligned. dtype is LA_F32 or LA_BF16;
 * accumulation and carried state are always float32. Shapes outside this
 * set return LA_ERR_INVALID_ARG before anything is launched.
 *
 * Errors: every entry point returns an int status and never throws.
 * la_status_string() maps it to a message.
 */
#ifndef LA_H_
#define LA_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

enum la_status {
  LA_OK = 0,
  LA_ERR_INVALID_ARG = 1, /* null pointer, bad dimension, unsupported D/M, misaligned pointer */
  LA_ERR_WORKSPACE = 2,   /* workspace missing or smaller than the *_workspace_bytes() size */
  LA_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed */
  LA_ERR_TIMEOUT = 4,     /* a bounded wait inside a kernel expired (see la_workspace_status) */
  LA_ERR_TOO_LARGE = 5    /* the problem needs more scratch than la_forward_noalloc holds */
};

enum la_dtype { LA_F32 = 0, LA_BF16 = 1 };

/* Human-readable text for a status code; never NULL. */
const char* la_status_string(int status);

/* Library ABI version (major * 100 + minor). */
int la_version(void);

/* Number of CUDA kernels this library has launched in this process so far
 * (all entry points, all threads; memsets are not counted). */
unsigned long long la_kernel_launches(void);

/*
 * Scratch needed by la_forward / la_prefill for this shape, in bytes (0 if
 * none). The caller allocates it (16-byte aligned, contents irrelevant) and
 * passes it in; it must not be shared by calls that may run concurrently.
 */
size_t la_forward_workspace_bytes(int B, int H, int N, int D, int M, int causal, int dtype);

/*
 * la_forward -- kernelized attention forward, out = V'.
 *
 * causal != 0: [deck slide 4], [summary §3.3]:
 *   S_i = S_{i-1} + phi(K_i) V_i^T,  Z_i = Z_{i-1} + phi(K_i),
 *   out_i = phi(Q_i)^T S_i / (phi(Q_i)^T Z_i)      (inclusive mask j <= i)
 * causal == 0: [review, "Proposed method"], [deck slide 3]:
 *   S = sum_j phi(K_j) V_j^T, Z = sum_j phi(K_j), out_i = phi(Q_i)^T S / phi(Q_i)^T Z
 *
 * q, k, v: inputs (see layouts); out: output, same dtype as the inputs.
 * workspace/workspace_bytes: caller scratch of la_forward_workspace_bytes().
 * Returns LA_OK, LA_ERR_INVALID_ARG, LA_ERR_WORKSPACE or LA_ERR_CUDA.
 */
int la_forward(const void* q, const void* k, const void* v, void* out,
               int B, int H, int N, int D, int M, int causal, int dtype,
               void* workspace, size_t workspace_bytes, void* stream);

/*
 * la_prefill -- causal forward that also writes the final recurrent state.
 *
 * [summary §3.4], [review, "Proposed method"]: a causally masked layer is an
 * RNN with attention memory s and normalizer memory z. Writes out as
 * la_forward(causal=1) and S[b][h] = S_N, Z[b][h] = Z_N (float32), which
 * la_decode_step then continues. B plays the role of independent streams.
 * Workspace: la_forward_workspace_bytes(B, H, N, D, M, 1, dtype).
 * N == 0 writes S = 0, Z = 0.
 */
int la_prefill(const void* q, const void* k, const void* v, void* out, float* S, float* Z,
               int B, int H, int N, int D, int M, int dtype,
               void* workspace, size_t workspace_bytes, void* stream);

/*
 * la_extend -- causal forward over N new tokens of B streams that continue
 * from a stored recurrent state (chunked prefill, multi-token decode).
 *
 * [deck slide 4], [summary §3.3.2, §3.4]: the causally masked layer is an RNN,
 * so a stream's next tokens depend on its past only through (S, Z). For each
 * stream b and head h, with (S, Z) the state in pool entry slots[b] (head h)
 * on entry, out[b][h][i] = phi(q_i)^T S_i / phi(q_i)^T Z_i for i = 0..N-1 with
 * S_i = S + sum_{j<=i} phi(k_j) v_j^T, Z_i = Z + sum_{j<=i} phi(k_j), and the
 * entry holds (S_{N-1}, Z_{N-1}) on return. N = 1 is one la_decode_step; a
 * zero state gives la_prefill.
 *
 * q, k: [B][H][N][D]; v, out: [B][H][N][M] in `dtype`.
 * S_pool [pool_size][H][D][M], Z_pool [pool_size][H][D] float32, caller-owned,
 * read and updated in place.
 * slots: device int[B] (4-byte aligned) naming each stream's pool entry, all
 * distinct; nullptr means entry b (then pool_size >= B). A slot outside
 * [0, pool_size) is not read or written: that stream starts from a zero state,
 * and la_workspace_status reports LA_ERR_INVALID_ARG afterwards.
 * lens: device int[B] (4-byte aligned), stream b's token count n_b (clamped to
 * [0, N]): only its first n_b tokens are read and its state advances by n_b;
 * out rows at or past n_b are unspecified, and the padding rows of q, k, v may
 * hold anything. nullptr: every stream has N tokens.
 * Workspace: la_forward_workspace_bytes(B, H, N, D, M, 1, dtype).
 * N == 0 returns LA_OK without touching the pool.
 */
int la_extend(const void* q, const void* k, const void* v, void* out,
              float* S_pool, float* Z_pool, const int* slots, const int* lens,
              int pool_size, int B, int H, int N, int D, int M, int dtype,
              void* workspace, size_t workspace_bytes, void* stream);

/*
 * la_extend_packed -- la_extend on a packed, token-major batch: B streams of
 * different lengths stored back to back with no padding (a serving batch).
 *
 * The method is la_extend's ([deck slide 4], [summary §3.3.2, §3.4]): each
 * stream continues from its pool entry's (S, Z) and the entry advances past
 * its tokens. Only the layout differs.
 *
 * q, k: [T][H][D]; v, out: [T][H][M] in `dtype` (T = total_tokens): row t
 * holds token t of every head. cu_seqlens: device int[B + 1] (4-byte
 * aligned): stream b's tokens are rows cu_seqlens[b] .. cu_seqlens[b + 1] - 1,
 * in order. max_len bounds every stream's length (it sizes the chunk grid and
 * the workspace: la_forward_workspace_bytes(B, H, max_len, D, M, 1, dtype)).
 * Out rows of a stream's tokens are written, no other row is. A stream whose
 * bounds break 0 <= cu_seqlens[b] <= cu_seqlens[b + 1] <= T is treated as empty,
 * and one longer than max_len as its first max_len tokens (rows after those are
 * not written); either makes la_workspace_status report LA_ERR_INVALID_ARG
 * afterwards. S_pool, Z_pool, slots, pool_size: as la_extend.
 * total_tokens == 0 or max_len == 0 returns LA_OK without touching the pool;
 * total_tokens above 2^30 returns LA_ERR_INVALID_ARG.
 */
int la_extend_packed(const void* q, const void* k, const void* v, void* out,
                     float* S_pool, float* Z_pool, const int* slots, const int* cu_seqlens,
                     int pool_size, int B, int H, int total_tokens, int max_len, int D, int M,
                     int dtype, void* workspace, size_t workspace_bytes, void* stream);

/* Scratch needed by la_backward for this shape, in bytes. */
size_t la_backward_workspace_bytes(int B, int H, int N, int D, int M, int causal, int dtype);

/*
 * la_backward -- gradients of sum(dout * out) w.r.t. q, k, v.
 *
 * [summary §3.3.1, App. A]: cumulative-sum gradients, never storing every S_i;
 * the phi(Q) gradient is a forward-direction scan over (S_i, Z_i), the phi(K)
 * and V gradients a reverse-direction scan over R_j = sum_{i>=j} phi(Q_i) gN_i^T
 * and r_j = sum_{i>=j} gd_i phi(Q_i), with gN_i = dout_i / den_i and
 * gd_i = -(dout_i . out_i) / den_i (the normalizer's quotient-rule terms):
 *   dphiQ_i = S_i gN_i + gd_i Z_i,  dphiK_j = R_j V_j + r_j,  dV_j = R_j^T phi(K_j),
 *   dq = dphiQ * phi'(q),  dk = dphiK * phi'(k).
 * Non-causal uses the full sums in both directions. The forward quantities are
 * recomputed, not read from a saved forward.
 *
 * q, k, v, dout: inputs in `dtype`; dq, dk, dv: float32 outputs.
 */
int la_backward(const void* q, const void* k, const void* v, const void* dout,
                float* dq, float* dk, float* dv,
                int B, int H, int N, int D, int M, int causal, int dtype,
                void* workspace, size_t workspace_bytes, void* stream);

/*
 * la_forward_poly2 -- kernelized attention with the degree-2 polynomial
 * feature map: [summary §3.2.1], the kernel sim(x, y) = (x . y)^2 has the
 * exact finite feature map phi(x) = vec(x x^T) (D^2 features), so
 *   out_i = sum_{j<=i} (q_i . k_j)^2 v_j / sum_{j<=i} (q_i . k_j)^2
 *         = phi(q_i)^T S_i / phi(q_i)^T Z_i
 * with the S/Z recurrence of la_forward over the D^2-dimensional features
 * ([deck slide 4]). Layouts and ownership as la_forward. Supported: bf16,
 * D = M = 64 (4096 features), causal != 0; anything else returns
 * LA_ERR_INVALID_ARG. Workspace: la_poly2_workspace_bytes() (the state part
 * of every numerator and denominator in float32, 260 bytes per token and head).
 */
size_t la_poly2_workspace_bytes(int B, int H, int N, int D, int M, int causal, int dtype);
int la_forward_poly2(const void* q, const void* k, const void* v, void* out,
                     int B, int H, int N, int D, int M, int causal, int dtype,
                     void* workspace, size_t workspace_bytes, void* stream);

/*
 * la_forward_rff -- kernelized attention with random Fourier features of the
 * RBF kernel. [summary §5] names them, approximating the RBF kernel, as the
 * next feature map; the pages give no definition, and the one taken is Rahimi
 * and Recht's (2007): with the F rows w_f of W and the phases b_f drawn by the
 * caller (w_f ~ N(0, sigma^-2 I), b_f ~ U[0, 2 pi) for an RBF kernel of width
 * sigma),
 *   phi(x) = sqrt(2 / F) [cos(w_1 . x + b_1), ..., cos(w_F . x + b_F)],
 * and the attention is la_forward's (causal or not) with this phi in place of
 * elu + 1. phi(q) . phi(k) is an estimate of exp(-|q - k|^2 / (2 sigma^2)) and
 * can be negative, so a denominator phi(q_i)^T Z_i near zero makes out_i
 * ill-conditioned (the plain definition behaves the same).
 * W: [F][D] in `dtype` (row-major), bias: [F] float32, device memory.
 * Supported: bf16, D = M = F = 64; else LA_ERR_INVALID_ARG. Workspace:
 * la_rff_workspace_bytes() (la_forward's, then the bf16 features of q and k).
 */
size_t la_rff_workspace_bytes(int B, int H, int N, int D, int M, int F, int causal, int dtype);
int la_forward_rff(const void* q, const void* k, const void* v, const void* W, const float* bias,
                   void* out, int B, int H, int N, int D, int M, int F, int causal, int dtype,
                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * Sequence shards. [summary §3.3, §3.3.1], [deck slide 4]: causal attention is
 * a prefix recurrence over (S, Z), and its gradient a pair of cumulative sums
 * running in opposite directions. A causal sequence cut into consecutive shards
 * (one per rank, each holding tokens [n_r, n_{r+1}) of every (b, h) sequence)
 * therefore needs exactly two exchanges, each of D*M + D float32 per head:
 *   forward:  (S0, Z0) of shard r = sum over shards before r of their own
 *             (S, Z) sums (la_state_sums), an exclusive prefix;
 *   backward: (R0, r0) of shard r = sum over shards after r of their own
 *             reverse sums (R_own, r_own from la_backward_shard_q), an
 *             exclusive suffix.
 * With those, shard r computes exactly its part of the unsharded results:
 *   la_forward_shard(S0, Z0)         -> out of its tokens,
 *   la_backward_shard_q(S0, Z0)      -> dq of its tokens, and R_own, r_own,
 *   la_backward_shard_kv(R0, r0)     -> dk, dv of its tokens.
 * The exchange itself (e.g. an all-gather of the per-shard sums) is the
 * caller's; nothing here communicates. Causal only. State layouts as S and Z
 * above ([B][H][D][M], [B][H][D] float32); R is [B][H][D][M] (R[d][m]) and r
 * [B][H][D]. Workspaces: la_forward_workspace_bytes(..., causal = 1, dtype)
 * for la_state_sums and la_forward_shard, la_backward_workspace_bytes(...) for
 * the two backward passes, which must be given the same workspace, in order,
 * with nothing in between on it.
 */

/* la_state_sums -- S = sum_j phi(k_j) v_j^T, Z = sum_j phi(k_j) of each
 * (b, h) sequence (the review's "Proposed method", deck slide 3), written to
 * S, Z. k: [B][H][N][D], v: [B][H][N][M] in `dtype`. N == 0 writes zeros. */
int la_state_sums(const void* k, const void* v, float* S, float* Z,
                  int B, int H, int N, int D, int M, int dtype,
                  void* workspace, size_t workspace_bytes, void* stream);

/* la_forward_shard -- causal forward of N tokens that follow the state
 * (S0, Z0) (read only): out_i = phi(q_i)^T S_i / phi(q_i)^T Z_i with
 * S_i = S0 + sum_{j<=i} phi(k_j) v_j^T, Z_i = Z0 + sum_{j<=i} phi(k_j). */
int la_forward_shard(const void* q, const void* k, const void* v, void* out,
                     const float* S0, const float* Z0,
                     int B, int H, int N, int D, int M, int dtype,
                     void* workspace, size_t workspace_bytes, void* stream);

/* la_backward_shard_q -- first backward pass of a shard ([summary App. A]:
 * the forward-direction sums): dq of its tokens given the state (S0, Z0)
 * before them (read only), and the shard's own reverse sums
 * R_own = sum_i phi(q_i) gN_i^T, r_own = sum_i gd_i phi(q_i) (float32,
 * written). den_i and gd_i stay in `workspace` for the second pass. N == 0
 * writes R_own = 0, r_own = 0. */
int la_backward_shard_q(const void* q, const void* k, const void* v, const void* dout,
                        float* dq, const float* S0, const float* Z0, float* R_own, float* r_own,
                        int B, int H, int N, int D, int M, int dtype,
                        void* workspace, size_t workspace_bytes, void* stream);

/* la_backward_shard_kv -- second backward pass of a shard (the reverse-
 * direction sums): dk, dv of its tokens given the reverse sums (R0, r0) of
 * the tokens after the shard (read only), with the workspace of its
 * la_backward_shard_q call. */
int la_backward_shard_kv(const void* q, const void* k, const void* v, const void* dout,
                         float* dk, float* dv, const float* R0, const float* r0,
                         int B, int H, int N, int D, int M, int dtype,
                         void* workspace, size_t workspace_bytes, void* stream);

/*
 * la_backward_from_forward -- la_backward that reuses the segment states a
 * la_forward call left in its workspace (the forward-direction sums S, Z before
 * each segment of the sequence, [summary §3.3.1]), instead of recomputing them:
 * the training order, where the backward follows the forward on the same
 * inputs. Same arguments, results and status codes as la_backward, plus
 * fwd_workspace / fwd_workspace_bytes: the workspace of a la_forward call with
 * the same q, k, B, H, N, D, M, causal and dtype, completed (or earlier on the
 * same stream) and not reused since. Where that forward keeps no states (one
 * chunk per sequence, or the CUDA-core path) they are computed as la_backward
 * does. The forward workspace is only read.
 */
int la_backward_from_forward(const void* q, const void* k, const void* v, const void* dout,
                             float* dq, float* dk, float* dv,
                             int B, int H, int N, int D, int M, int causal, int dtype,
                             const void* fwd_workspace, size_t fwd_workspace_bytes,
                             void* workspace, size_t workspace_bytes, void* stream);

/*
 * la_decode_step -- one recurrent generation step per (stream, head).
 *
 * [deck slide 4], [summary §3.3.2, §3.4]: update, then read out:
 *   S <- S + phi(k) v^T,  Z <- Z + phi(k),  out = phi(q)^T S / phi(q)^T Z.
 * q, k: [n_streams][H][D]; v, out: [n_streams][H][M] in `dtype`;
 * S [n_streams][H][D][M] and Z [n_streams][H][D] float32, updated in place.
 * Needs no workspace.
 */
int la_decode_step(const void* q, const void* k, const void* v, float* S, float* Z, void* out,
                   int n_streams, int H, int D, int M, int dtype, void* stream);

/*
 * la_forward_noalloc -- la_forward for callers that cannot allocate device
 * memory: code that only receives device pointers for its inputs and outputs
 * from a host application or framework that owns the allocator (and exposes
 * none to it), or that runs where a cudaMalloc is not permitted. The paper has
 * no counterpart; this is a deployment variant of la_forward.
 *
 * Same arguments, layouts, results and status codes as la_forward, without
 * the workspace: the scratch is a fixed array of LA_NOALLOC_SCRATCH_BYTES in
 * the library's own device memory. Every GPU that loads the library holds
 * that array until the process exits. Nothing is allocated or freed by this
 * call (no cudaMalloc/cudaFree or allocating library routine).
 *
 * - The first call on each device looks up the array's device address with
 *   that device current (the caller's current device must be the one its
 *   pointers and stream belong to). Make that first call before any stream
 *   capture.
 * - Returns LA_ERR_TOO_LARGE, launching nothing, when the shape needs more
 *   scratch than the array holds (la_forward_workspace_bytes() > capacity).
 * - All calls share the one array and it keeps the previous call's contents
 *   (each call clears what must start at zero). Calls that overlap on the GPU,
 *   from any stream or host thread, race on it: serialise them.
 */
#define LA_NOALLOC_SCRATCH_BYTES (32u << 20)
int la_forward_noalloc(const void* q, const void* k, const void* v, void* out,
                       int B, int H, int N, int D, int M, int causal, int dtype, void* stream);

/*
 * la_forward_noalloc_status -- the status word of the fixed scratch array on
 * the current device, as la_workspace_status reads a caller's workspace:
 * synchronises `stream`, returns LA_OK or the LA_ERR_TIMEOUT a bounded wait of
 * the last la_forward_noalloc call recorded (its outputs are then invalid),
 * and clears the word. Each la_forward_noalloc call clears it on entry, so it
 * describes the last call only. Allocates nothing.
 */
int la_forward_noalloc_status(void* stream);

/*
 * la_debug_noalloc_set_status -- test hook (no counterpart on the pages):
 * writes `status` and `wait_site` into the status header of the fixed scratch
 * array on the current device, as a kernel whose bounded wait ran out would,
 * so that tests can check la_forward_noalloc_status reads and clears it.
 */
int la_debug_noalloc_set_status(int status, int wait_site, void* stream);

/*
 * la_workspace_status -- synchronises `stream` and reads the status word a
 * previous la_forward / la_prefill / la_extend / la_backward left in
 * `workspace`: LA_OK; LA_ERR_TIMEOUT if a bounded wait inside a kernel (for a
 * TMA copy or a group of tensor-core MMAs) gave up, the outputs of that call
 * then being invalid; LA_ERR_INVALID_ARG if la_extend met a slot outside its
 * pool. Clears the word. Debug / test use.
 */
int la_workspace_status(void* workspace, size_t workspace_bytes, void* stream);

/*
 * la_workspace_wait_site -- synchronises `stream` and returns the code of the
 * bounded wait that last gave up in the call that used `workspace` (0 if none
 * did; -1 if the header cannot be read). The codes are internal to the
 * kernels; the two the failure test hooks below make run out are
 * LA_SITE_FORWARD_LOAD and LA_SITE_BACKWARD_LOAD. Does not clear anything.
 */
enum la_wait_site {
  LA_SITE_FORWARD_LOAD = 11,  /* forward chunk-attention kernel, waiting for a chunk's tiles */
  LA_SITE_FORWARD_FUSED_LOAD = 16, /* one-launch forward, waiting for a chunk's K, V tiles
                                      while it sums its segment's states */
  LA_SITE_BACKWARD_LOAD = 21  /* backward forward-direction kernel, waiting for a chunk's tiles */
};
int la_workspace_wait_site(void* workspace, size_t workspace_bytes, void* stream);

/*
 * Failure-detection test hooks (the pages have no counterpart; test use only).
 *
 * la_debug_forward_fault / la_debug_backward_fault run la_forward /
 * la_backward on the tensor-core path (bf16, D = M = 64) with one TMA load
 * withheld: CTA 0 of the main kernel (the forward's chunk attention, the
 * backward's forward-direction kernel) skips issuing its load number
 * `withhold_load` (counted from 0 in its own issue order), so the wait for it
 * can only run out, and bounds its main-loop waits by `wait_limit_ns`
 * (1 us .. 2 s; every other wait keeps the normal 2 s limit). Nothing faults:
 * the CTA records LA_ERR_TIMEOUT and the wait site in the workspace header,
 * waits (with the full limit) for its issued copies and MMAs, frees its tensor
 * memory and returns; the other CTAs finish normally. The outputs are then
 * invalid. If CTA 0 issues fewer loads than withhold_load + 1 nothing is
 * withheld. Returns LA_ERR_INVALID_ARG off the tensor-core path, for
 * withhold_load < 0 or a limit out of range; otherwise as la_forward /
 * la_backward.
 */
int la_debug_forward_fault(const void* q, const void* k, const void* v, void* out,
                           int B, int H, int N, int D, int M, int causal, int dtype,
                           void* workspace, size_t workspace_bytes, int withhold_load,
                           unsigned long long wait_limit_ns, void* stream);
/*
 * la_debug_forward_fused_fault: la_debug_forward_fault on the one-launch forward
 * (a thread-block cluster per sequence; la_forward takes it when a sequence has at
 * most 8 segments, and so does this hook; otherwise it is la_debug_forward_fault).
 * CTA 0, the first segment's CTA of the first sequence, withholds its load number
 * `withhold_load` (its loads of K, V while it sums the segment's states come first),
 * so its wait runs out (LA_SITE_FORWARD_FUSED_LOAD for those); the CTA still
 * reaches both of its cluster's barriers, so the cluster's other CTAs finish.
 */
int la_debug_forward_fused_fault(const void* q, const void* k, const void* v, void* out,
                                 int B, int H, int N, int D, int M, int causal, int dtype,
                                 void* workspace, size_t workspace_bytes, int withhold_load,
                                 unsigned long long wait_limit_ns, void* stream);
int la_debug_backward_fault(const void* q, const void* k, const void* v, const void* dout,
                            float* dq, float* dk, float* dv,
                            int B, int H, int N, int D, int M, int causal, int dtype,
                            void* workspace, size_t workspace_bytes, int withhold_load,
                            unsigned long long wait_limit_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* LA_H_ */
