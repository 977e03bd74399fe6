// Tensor-core backward for bf16 inputs with D = M = 64: cumulative-sum
// gradients ("Transformers are RNNs", paperlayer.ai summary §3.3.1 and
// App. A), chunked like the forward.
//
// With G = dout, den_i = phi(Q_i)^T Z_i, out_i = num_i / den_i:
//   gN_i = G_i / den_i,  gd_i = -(G_i . out_i) / den_i,
//   T_ij = V_j . gN_i + gd_i,
//   dphiQ_i = sum_{j<=i} T_ij phi(K_j)            (forward-direction sums)
//   dphiK_j = sum_{i>=j} T_ij phi(Q_i)            (reverse-direction sums)
//   dV_j    = sum_{i>=j} (phi(Q_i) . phi(K_j)) gN_i
// and dq = dphiQ * phi'(q), dk = dphiK * phi'(k). Per chunk of C = 128 tokens
// the sums split into an intra-chunk part with the masked C x C matrices
// P_L = (phi(Q) phi(K)^T) (.) L and T_L, and a state part: S_prev, Z_prev
// (state before the chunk) for dq, R_next = sum_{i after the chunk} phi(Q_i)
// gN_i^T and r_next = sum gd_i phi(Q_i) for dk and dv:
//   dphiQ = T_L phi(K) + gN S_prev^T + gd Z_prev^T
//   dphiK = T_L^T phi(Q) + V R_next^T + r_next
//   dV    = P_L^T gN + phi(K) R_next
//
// Kernels: the forward's segment-state kernel and scan give S_prev per
// segment; tc_bwd_q_kernel (forward direction) recomputes num/den, writes dq,
// den_i, gd_i and each segment's sum of phi(Q)^T gN and gd phi(Q); a suffix
// scan gives R_next per segment; tc_bwd_kv_kernel walks each segment's chunks
// from last to first and writes dk, dv.
//
// Precision: phi(k) = 1 + k for small k, and dq = sum_j T_ij phi(K_j) cancels
// the constant part (sum_j T_ij ~ 0; exactly 0 at i = j = 0). What is left is
// carried by k, so bf16 rounding of phi(K) (2^-9 absolute at 1.0) would cost
// dq ~2% normwise and ~10% on its significant elements; likewise phi(Q) for dk
// and P_L, T_L for dq. Every operand that feeds such a sum therefore enters the
// tensor cores as a bf16 hi + lo pair (phi(K) and P_L in the forward-direction
// kernel and the prefix states, phi(Q) in both kernels' R sums and T_L^T phi(Q),
// T_L / T_L^T, gN, and the carried states), and gd is added in float32.
#include "la_tc_common.cuh"

namespace la {
namespace tcx {
namespace {

// Shared memory of the reverse-direction (dk, dv) kernel.
constexpr int kBwdStages = 2;
constexpr int kSnapB = 2 * kDim * 128;  // state snapshot, hi and lo, 64 rows each
constexpr int kGnB = 2 * kTile;         // gN hi and lo, 128 rows each
constexpr int kArr = 8192;              // small float arrays
constexpr int kLoB = kTile;             // phi(Q) lo part
constexpr int kBwdSmem =
    1024 + kBwdStages * 4 * kTile + kSnapB + kGnB + kLoB + kArr + 2048;

__device__ __forceinline__ void split_bf16(float a, float b, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16(a, b);
  const float2 r = sub2(make_float2(a, b), make_float2(bf16_lo_f(hi), bf16_hi_f(hi)));
  lo = pack_bf16(r.x, r.y);
}

// 16 consecutive bf16 of row `row`, logical 16-byte chunks c0, c0+1 -> float.
__device__ __forceinline__ void load_row16(const uint8_t* tile, int row, int c0, float* out) {
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const uint4 w = *reinterpret_cast<const uint4*>(tile + sw128(row, (c0 + c) * 16));
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      out[8 * c + 2 * q] = bf16_lo_f(u[q]);
      out[8 * c + 2 * q + 1] = bf16_hi_f(u[q]);
    }
  }
}

struct BwdSmem {
  uint8_t* stages;
  uint8_t* s_hi;
  uint8_t* s_lo;
  uint8_t* gn_hi;
  uint8_t* gn_lo;
  uint8_t* qlo;
  float* arr;
  uint64_t* full;
  uint64_t* mma_bar;
  uint64_t* sbar;  // sbar[1]: the chunk's R sums (and all their issuer issued before them)
  uint64_t* drain;  // every MMA of the CTA is done (end of the kernel)
  uint32_t* tslot;
  __device__ explicit BwdSmem(uint8_t* raw) {
    uint8_t* sm =
        reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    stages = sm;
    s_hi = sm + kBwdStages * 4 * kTile;
    s_lo = s_hi + kDim * 128;
    gn_hi = s_lo + kDim * 128;
    gn_lo = gn_hi + kTile;
    qlo = gn_lo + kTile;
    arr = reinterpret_cast<float*>(qlo + kTile);
    uint8_t* misc = reinterpret_cast<uint8_t*>(arr) + kArr;
    full = reinterpret_cast<uint64_t*>(misc);
    mma_bar = full + kBwdStages;
    sbar = mma_bar + 1;
    drain = sbar + 2;
    tslot = reinterpret_cast<uint32_t*>(drain + 1);
  }
  __device__ uint8_t* tile(int stage, int which) { return stages + (stage * 4 + which) * kTile; }
};

enum { kQ = 0, kK = 1, kV = 2, kG = 3 };

// Named barrier 1 over the dk/dv kernel's 512 threads: the threads that hand data
// over arrive without waiting, the ones that take it wait.
__device__ __forceinline__ void named_arrive_all() { asm volatile("bar.arrive 1, 512;" ::: "memory"); }
__device__ __forceinline__ void named_sync_all() { asm volatile("bar.sync 1, 512;" ::: "memory"); }
// The dk/dv kernel's per-chunk R sums and its second MMA group are issued by the
// first thread of warp 2 (TMEM lanes 64-95: its slice of the P / T epilogue is
// masked out entirely and its R exchange only hands data over); thread 0 issues
// the first group (P, W).
constexpr int kG2Issuer = 64;

// The reverse-direction kernel runs 512 threads: warp w covers TMEM lane quarter
// w % 4 (rows 32 (w % 4) .. + 31) and column quarter qc = w / 4 (16 of the 64
// state columns, the 32-column slice qc of the chunk's 128), so every row is
// handled by four threads; threads 0 and 64 issue its MMAs. Where a TMEM region is
// compacted in place (fp32 P into bf16 P_L), all reads finish before a barrier
// and the writes follow it.
constexpr int kBTQ = 512;

// Quarter-row store of x[16] (columns [16 qc, 16 qc + 16)) as bf16 hi and lo rows.
__device__ __forceinline__ void store_split_quarter(uint8_t* hi_buf, uint8_t* lo_buf, int row, int qc,
                                                    const float* x) {
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    uint32_t hh[4], ll[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) split_bf16(x[8 * c + 2 * q], x[8 * c + 2 * q + 1], hh[q], ll[q]);
    const uint32_t off = sw128(row, (2 * qc + c) * 16);
    *reinterpret_cast<uint4*>(hi_buf + off) = make_uint4(hh[0], hh[1], hh[2], hh[3]);
    *reinterpret_cast<uint4*>(lo_buf + off) = make_uint4(ll[0], ll[1], ll[2], ll[3]);
  }
}

// phi on columns [16 qc, 16 qc + 16) of a tile row, rounded to bf16 in place with
// the rounding error kept as a bf16 lo part in `lo`; z gets the float32 values.
// Rows >= nvalid become zero.
template <bool MASK>
__device__ __forceinline__ void phi_quarter_split_impl(uint8_t* tile, uint8_t* lo, int row, int qc,
                                                       int nvalid, float (&z)[16]) {
  const bool valid = !MASK || row < nvalid;
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const uint32_t off = sw128(row, (2 * qc + c) * 16);
    const uint4 w = *reinterpret_cast<const uint4*>(tile + off);
    uint32_t u[4] = {w.x, w.y, w.z, w.w}, l[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float a = valid ? phi_fast(bf16_lo_f(u[q])) : 0.f;
      const float b = valid ? phi_fast(bf16_hi_f(u[q])) : 0.f;
      u[q] = pack_bf16(a, b);
      const float2 e = sub2(make_float2(a, b), make_float2(bf16_lo_f(u[q]), bf16_hi_f(u[q])));
      l[q] = pack_bf16(e.x, e.y);
      z[8 * c + 2 * q] = a;
      z[8 * c + 2 * q + 1] = b;
    }
    *reinterpret_cast<uint4*>(tile + off) = make_uint4(u[0], u[1], u[2], u[3]);
    *reinterpret_cast<uint4*>(lo + off) = make_uint4(l[0], l[1], l[2], l[3]);
  }
}

__device__ __forceinline__ void phi_quarter_split(uint8_t* tile, uint8_t* lo, int row, int qc, int nvalid,
                                                  float (&z)[16]) {
  if (nvalid >= kC)
    phi_quarter_split_impl<false>(tile, lo, row, qc, nvalid, z);
  else
    phi_quarter_split_impl<true>(tile, lo, row, qc, nvalid, z);
}

// Sum z[16] over the 32 lanes of a warp; lanes l and l + 16 end with column l % 16.
__device__ __forceinline__ float warp_column_sums16(float (&z)[16]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1) {
    const bool up = lane & w;
#pragma unroll
    for (int j = 0; j < w; ++j) {
      const float mine = up ? z[w + j] : z[j];
      const float other = up ? z[j] : z[w + j];
      z[j] = mine + __shfl_xor_sync(0xffffffffu, other, w);
    }
  }
  return z[0] + __shfl_xor_sync(0xffffffffu, z[0], 16);
}

__device__ __forceinline__ void sync_tc() {
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
}

// --------------------------------------------------- warp-specialised kernels
//
// 640 threads: warps 0-15 are the workers (warp w covers TMEM lane quarter
// w % 4 and column quarter w / 4, every tile row handled by four threads);
// warp 16 issues the MMAs and warp 17 the TMA loads and stores, one thread
// each; warps 18 and 19 complete that control warpgroup, whose registers go to
// the workers. The workers hand the MMA warp its operands through mbarriers
// (one arrival per warp), and the TMA warp the staged outputs; among themselves
// they synchronise on a named barrier. Nothing else waits for the thread that
// issues a group of MMAs, and while a chunk's second group runs the workers
// already prepare the next chunk's tiles, which the TMA warp loaded into the
// other stage.
constexpr int kWorkers = 512;
constexpr int kWsThreads = kWorkers + 128;
constexpr int kMmaWarp = 16, kTmaWarp = 17;
constexpr int kWorkerRegs = 112, kControlRegs = 32;  // 512 x 112 + 128 x 32 = 640 x 96

template <int N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// Named barrier 1 over the 512 workers, reducing a flag: true for all if any
// worker passes true (a failed wait ends the loop for every worker together).
__device__ __forceinline__ bool workers_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, 1, 512, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(v ? 1u : 0u)
      : "memory");
  return r != 0;
}

// Bounded wait of one thread that also gives up once another role has given up.
__device__ __forceinline__ bool role_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          WorkspaceHeader* hdr, int site, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      *abort = 1;
      record_timeout(hdr, site);
      return false;
    }
  }
}

// The same for a whole warp (warp-collective TMEM accesses follow).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          WorkspaceHeader* hdr, int site,
                                          uint64_t limit_ns = kWaitLimitNs) {
  return __all_sync(0xffffffffu, role_wait(bar, parity, abort, hdr, site, limit_ns));
}

// One arrival per warp on a barrier that counts the 16 worker warps, once every
// lane's writes are in.
__device__ __forceinline__ void warp_arrive(uint64_t* bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// Shared-memory descriptors as their low 32 bits (start address >> 4, leading
// byte offset >> 4): every operand here has a 1024-byte stride offset and the
// 128-byte swizzle, which make up the high half, the same for all of them.
__device__ __forceinline__ uint32_t sdesc_lo(uint32_t saddr, uint32_t lbo) {
  return ((saddr & 0x3FFFFu) >> 4) | (((lbo >> 4) & 0x3FFFu) << 16);
}
constexpr uint32_t kDescHi = (1024u >> 4) | (1u << 14) | (2u << 29);  // bits 32..63 of sdesc_lo(., .)

// D[tmem] (+)= A[smem] * B[smem] from the descriptors' low halves plus constant
// offsets (in 16-byte units), added inside the instruction sequence so that an
// unrolled run of MMAs keeps only its base descriptors in registers.
template <uint32_t AOFF, uint32_t BOFF>
__device__ __forceinline__ void mma_ss_l(uint32_t d, uint32_t a_lo, uint32_t b_lo, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b32 al, bl;\n\t.reg .b64 ra, rb;\n\t"
      "setp.ne.b32 p, %4, 0;\n\tadd.u32 al, %1, %6;\n\tadd.u32 bl, %2, %7;\n\t"
      "mov.b64 ra, {al, %5};\n\tmov.b64 rb, {bl, %5};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, p;\n\t}" ::"r"(d),
      "r"(a_lo), "r"(b_lo), "r"(idesc), "r"(accumulate), "r"(kDescHi), "n"(AOFF), "n"(BOFF)
      : "memory");
}

// The same with A in TMEM (its address offset also added in place).
template <uint32_t AOFF, uint32_t BOFF>
__device__ __forceinline__ void mma_ts_l(uint32_t d, uint32_t a_tmem, uint32_t b_lo, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b32 at, bl;\n\t.reg .b64 rb;\n\t"
      "setp.ne.b32 p, %4, 0;\n\tadd.u32 at, %1, %6;\n\tadd.u32 bl, %2, %7;\n\t"
      "mov.b64 rb, {bl, %5};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [at], rb, %3, p;\n\t}" ::"r"(d),
      "r"(a_tmem), "r"(b_lo), "r"(idesc), "r"(accumulate), "r"(kDescHi), "n"(AOFF), "n"(BOFF)
      : "memory");
}

// N MMAs over consecutive K = 16 slices, the descriptors advanced by AS / BS
// bytes per slice (32 inside a K-major swizzle atom, 2048 = 16 rows of an
// MN-major tile); acc0: whether the first one accumulates.
template <int N, uint32_t AS, uint32_t BS, int K = 0>
__device__ __forceinline__ void mma_run(uint32_t d, uint32_t a_lo, uint32_t b_lo, uint32_t idesc,
                                        uint32_t acc0) {
  if constexpr (K < N) {
    mma_ss_l<K * (AS >> 4), K * (BS >> 4)>(d, a_lo, b_lo, idesc, K == 0 ? acc0 : 1u);
    mma_run<N, AS, BS, K + 1>(d, a_lo, b_lo, idesc, acc0);
  }
}

// The same with A in TMEM (8 columns of packed bf16 per slice), accumulating.
template <int N, uint32_t BS, int K = 0>
__device__ __forceinline__ void mma_run_ts(uint32_t d, uint32_t a_tmem, uint32_t b_lo, uint32_t idesc) {
  if constexpr (K < N) {
    mma_ts_l<8 * K, K * (BS >> 4)>(d, a_tmem, b_lo, idesc, 1u);
    mma_run_ts<N, BS, K + 1>(d, a_tmem, b_lo, idesc);
  }
}

// --------------------------------------------------- forward direction: dq
//
// With W = G V^T (bf16 x bf16 products, exact in the float32 accumulator):
//   den_i   = rowsum(P_L)_i + phi(Q_i) . Z_prev
//   G.num_i = sum_j P_L,ij W_ij + G_i . (phi(Q_i) S_prev)
//   gd_i    = -(G.num_i) / den_i^2,   gN_i = G_i / den_i
//   T_ij    = W_ij / den_i + gd_i      (= (v_j - out_i) . gN_i, in float32)
// so one epilogue after the first MMA group yields T_L, gN and gd, and the
// second group accumulates dphiQ = T_L phi(K) + gN S_prev^T and the segment
// sum of phi(Q)^T gN.

// TMEM columns
constexpr uint32_t kFP = 0;     // 128: P = phi(Q) phi(K)^T; after the first epilogue, bf16 T_L
                                // hi in [0,64), lo in [64,128) (kFT)
constexpr uint32_t kFW = 128;   // 128: W = G V^T
constexpr uint32_t kFO = 256;   // 128: phi(Q) S_prev as phi(Q) S_hi (0..63) and phi(Q) S_lo (64..127);
                                // after the first epilogue, dphiQ as two 64-column parts (kFQ)
constexpr uint32_t kFT = 0;
constexpr uint32_t kFQ = 256;
constexpr uint32_t kFS = 384;   // 64: the S carry, M = 128 layout (rows d: prefix + hi parts in
                                // lanes 0-63, lo parts in 64-127)
constexpr uint32_t kFR = 448;   // 64: segment sum of phi(Q)^T gN (M = 128 layout, like dS)

// A stage holds one chunk: the loaded Q, K, V, G tiles (phi applied to Q and K
// in place) and the lo parts of phi(K) and phi(Q). gN takes the place of G (hi)
// and of the spent V (lo); dq is staged in the K and phi(K) lo tiles.
enum { kSQ = 0, kSK = 1, kSV = 2, kSG = 3, kSKL = 4, kSQL = 5, kQStageTiles = 6 };
constexpr int kQArr = 1664;  // floats: Z snapshots, column sums, den / G.num partials
constexpr int kQSmem = 1024 + 2 * kQStageTiles * kTile + 2 * kDim * 128 + kQArr * 4 + 128;

// Addresses from one aligned base and constant offsets, so that a role keeps a
// single pointer live instead of one per buffer.
struct QSmem {
  static constexpr int kSnap = 2 * kQStageTiles * kTile;  // S_prev as bf16 hi, then lo (rows d)
  static constexpr int kArrOff = kSnap + 2 * kDim * 128;
  static constexpr int kBarOff = kArrOff + kQArr * 4;
  enum {
    kFull = 0,     // [2] a stage's tiles landed
    kG1Ready = 2,  // the workers' operands of the first group are in (16 warps)
    kG2Ready,      // ... of the second group
    kStReady,      // the chunk's dq is staged, and the workers are done with its stage
    kG1Done,       // P, W, phi(Q) S_prev
    kDsDone,       // dS (the last reader of V)
    kGnFree,       // gN S_prev^T and the segment sums (the last readers of the gN tiles,
                   // the snapshot and the phi(Q) tiles)
    kG2Done,       // dphiQ
    kDqRead,       // the workers have read dphiQ (16 warps)
    kDrain,        // every MMA of the CTA is done (end of the kernel)
    kNBars
  };
  uint8_t* base;
  __device__ explicit QSmem(uint8_t* raw)
      : base(reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023))) {}
  __device__ uint8_t* tile(int s, int which) const { return base + (s * kQStageTiles + which) * kTile; }
  __device__ uint8_t* s_hi() const { return base + kSnap; }
  __device__ uint8_t* s_lo() const { return base + kSnap + kDim * 128; }
  __device__ float* arr() const { return reinterpret_cast<float*>(base + kArrOff); }
  __device__ uint64_t* bar(int i) const { return reinterpret_cast<uint64_t*>(base + kBarOff) + i; }
  __device__ int* abort() const { return reinterpret_cast<int*>(bar(kNBars)); }
  __device__ uint32_t* tslot() const { return reinterpret_cast<uint32_t*>(bar(kNBars)) + 1; }
};
static_assert(QSmem::kBarOff + QSmem::kNBars * 8 + 8 <= kQSmem - 1024, "dq kernel shared memory");

// MMA warp, one thread: per chunk the first group once the workers' phi and
// snapshot are in, the second once gN and T_L are.
template <bool CAUSAL>
__device__ __forceinline__ void bwd_q_mma(QSmem& sm, const Geometry& g, uint32_t tbase,
                                          volatile int* abort, WorkspaceHeader* hdr) {
  FullCursor c;
  c.start(g, true);
  const uint32_t ha = smem_u32(sm.s_hi()), la = smem_u32(sm.s_lo());
  long long n = 0;
  while (c.valid(g)) {
    const int s = (int)(n & 1);
    const uint32_t ph = (uint32_t)(n & 1);
    const uint32_t qa = smem_u32(sm.tile(s, kSQ)), ka = smem_u32(sm.tile(s, kSK));
    const uint32_t va = smem_u32(sm.tile(s, kSV)), ga = smem_u32(sm.tile(s, kSG));
    const uint32_t kl = smem_u32(sm.tile(s, kSKL)), ql = smem_u32(sm.tile(s, kSQL));
    if (!role_wait(sm.bar(QSmem::kG1Ready), ph, abort, hdr, 41, kWaitLimitNs)) break;
    // P overwrites the previous chunk's T_L: its second group must be done
    if (n > 0 && !role_wait(sm.bar(QSmem::kG2Done), ph ^ 1, abort, hdr, 44, kWaitLimitNs)) break;
    fence_after_sync();
    // K-major operands step 32 bytes per K = 16 slice (inside the swizzle atom),
    // MN-major ones 2048 bytes (16 rows of 128 bytes)
    if (CAUSAL) {
      const uint32_t id128 = idesc_bf16(128, 128, false, false);
      // P = phi(Q) (phi(K)_hi + phi(K)_lo)^T, W = G V^T
      mma_run<4, 32, 32>(tbase + kFP, sdesc_lo(qa, 16), sdesc_lo(ka, 16), id128, 0);
      mma_run<4, 32, 32>(tbase + kFP, sdesc_lo(qa, 16), sdesc_lo(kl, 16), id128, 1);
      mma_run<4, 32, 32>(tbase + kFW, sdesc_lo(ga, 16), sdesc_lo(va, 16), id128, 0);
    }
    // phi(Q) S_prev overwrites the previous chunk's dphiQ: the workers must have read it
    if (n > 0 && !role_wait(sm.bar(QSmem::kDqRead), ph ^ 1, abort, hdr, 45, kWaitLimitNs)) break;
    fence_after_sync();
    // phi(Q) [S_hi | S_lo]: B = the snapshot, rows d (= K), m contiguous
    // (MN-major), its hi and lo tiles the two 64-column N blocks (la - ha apart)
    mma_run<4, 32, 2048>(tbase + kFO, sdesc_lo(qa, 16), sdesc_lo(ha, la - ha),
                         idesc_bf16(128, 128, false, true), 0);
    mma_commit(sm.bar(QSmem::kG1Done));
    if (CAUSAL) {  // S += phi(K)^T V with phi(K)^T hi and lo stacked as one M = 128
                   // MN-major operand (kl - ka bytes apart); hi rows in lanes 0-63, lo 64-127
      mma_run<kC / 16, 2048, 2048>(tbase + kFS, sdesc_lo(ka, kl - ka), sdesc_lo(va, 1024),
                                   idesc_bf16(128, 64, true, true), 1);
      mma_commit(sm.bar(QSmem::kDsDone));
    }
    if (!role_wait(sm.bar(QSmem::kG2Ready), ph, abort, hdr, 42, kWaitLimitNs)) break;
    fence_after_sync();
    // gN [S_hi; S_lo]^T + gN_lo S_hi^T first: B = the snapshot, rows d (= N), m
    // contiguous (K-major), the S_lo rows after the S_hi rows (one N = 128
    // product); gN hi sits in the G tile, gN lo in the V tile. dphiQ is the sum
    // of the accumulator's two 64-column halves.
    const uint32_t gha = ga, gla = va;
    mma_run<4, 32, 32>(tbase + kFQ, sdesc_lo(gha, 16), sdesc_lo(ha, 16),
                       idesc_bf16(128, 128, false, false), 0);
    mma_run<4, 32, 32>(tbase + kFQ, sdesc_lo(gla, 16), sdesc_lo(ha, 16),
                       idesc_bf16(128, 64, false, false), 1);
    // segment sum of phi(Q)^T gN: phi(Q)^T hi and lo stacked as one M = 128
    // MN-major operand (ql - qa bytes apart) times gN hi, then gN lo; the hi-row
    // and lo-row halves (TMEM lanes 0-63 / 64-127) are summed at the segment's end
    const uint32_t idR = idesc_bf16(128, 64, true, true);
    mma_run<kC / 16, 2048, 2048>(tbase + kFR, sdesc_lo(qa, ql - qa), sdesc_lo(gha, 1024), idR,
                                 c.first() ? 0u : 1u);
    mma_run<kC / 16, 2048, 2048>(tbase + kFR, sdesc_lo(qa, ql - qa), sdesc_lo(gla, 1024), idR, 1);
    mma_commit(sm.bar(QSmem::kGnFree));
    if (CAUSAL) {
      // + T_L phi(K) with the hi*hi + hi*lo + lo*hi terms; the hi*lo partners share
      // their A operand (T_L in TMEM, 8 columns per K = 16 slice), so they sit side
      // by side in one N = 128 instruction: T_hi [phi(K)_hi | phi(K)_lo] (N blocks
      // kl - ka apart), then T_lo phi(K)_hi
      mma_run_ts<kC / 16, 2048>(tbase + kFQ, tbase + kFT, sdesc_lo(ka, kl - ka),
                                idesc_bf16(128, 128, false, true));
      mma_run_ts<kC / 16, 2048>(tbase + kFQ, tbase + kFT + 64, sdesc_lo(ka, 1024),
                                idesc_bf16(128, 64, false, true));
    }
    mma_commit(sm.bar(QSmem::kG2Done));
    ++n;
    c.advance(g);
  }
  // every MMA completes before the CTA frees TMEM (time-bounded only)
  mma_commit(sm.bar(QSmem::kDrain));
  if (!mbar_wait(sm.bar(QSmem::kDrain), 0)) record_timeout(hdr, 25);
}

// TMA warp, one thread: loads two chunks ahead of the workers, stores each
// chunk's dq once it is staged and then refills that stage.
template <bool CAUSAL>
__device__ __forceinline__ void bwd_q_tma(QSmem& sm, const Geometry& g, const CUtensorMap* tm_q,
                                          const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                                          const CUtensorMap* tm_g, const CUtensorMap* tm_dq,
                                          volatile int* abort, WorkspaceHeader* hdr) {
  const uint32_t tx = (CAUSAL ? 4 : 2) * kTile;
  FullCursor cl, cs;
  cl.start(g, true);
  cs = cl;
  long long nl = 0, ns = 0;
  auto load = [&]() {
    const int s = (int)(nl & 1);
    if (!(g.faulty() && nl == g.fault_load)) {  // test hook: this load is withheld
      const int t0 = cl.chunk * kC;
      mbar_arrive_expect_tx(sm.bar(QSmem::kFull + (s)), tx);
      tma_load_3d(sm.tile(s, kSQ), tm_q, sm.bar(QSmem::kFull + (s)), 0, t0, cl.bh);
      tma_load_3d(sm.tile(s, kSG), tm_g, sm.bar(QSmem::kFull + (s)), 0, t0, cl.bh);
      if (CAUSAL) {
        tma_load_3d(sm.tile(s, kSK), tm_k, sm.bar(QSmem::kFull + (s)), 0, t0, cl.bh);
        tma_load_3d(sm.tile(s, kSV), tm_v, sm.bar(QSmem::kFull + (s)), 0, t0, cl.bh);
      }
    }
    ++nl;
    cl.advance(g);
  };
  while (nl < 2 && cl.valid(g)) load();
  while (cs.valid(g)) {
    const int s = (int)(ns & 1);
    if (!role_wait(sm.bar(QSmem::kStReady), (uint32_t)(ns & 1), abort, hdr, 43, kWaitLimitNs)) break;
    // rows past the sequence end are clipped by the tensor map
    tma_store_3d(tm_dq, sm.tile(s, kSK), 0, cs.chunk * kC, cs.bh);
    tma_store_3d(tm_dq, sm.tile(s, kSKL), 32, cs.chunk * kC, cs.bh);
    bulk_commit();
    if (cl.valid(g)) {
      bulk_wait_read<0>();
      load();
    }
    ++ns;
    cs.advance(g);
  }
  // every issued load lands and every store completes before the CTA lets go of
  // its shared memory (time-bounded only)
  for (long long k = ns; k < nl; ++k)
    if (!(g.faulty() && k == g.fault_load) && !mbar_wait(sm.bar(QSmem::kFull + (k & 1)), (uint32_t)((k >> 1) & 1)))
      record_timeout(hdr, 26);
  bulk_wait_all<0>();
}

template <bool CAUSAL>
__device__ __forceinline__ void bwd_q_workers(QSmem& sm, const Geometry& g, uint32_t tbase,
                                              volatile int* abort, const float* __restrict__ sprefix,
                                              float* __restrict__ rpartial, float* __restrict__ den_out,
                                              float* __restrict__ gd_out, WorkspaceHeader* hdr) {
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int lq = warp & 3, qc = warp >> 2;
  const int row = lq * 32 + lane;  // query row of this thread
  // S carry: row d = 32 (lq % 2) + lane, held by the threads of TMEM lanes 0-63
  const int drow = 32 * (lq & 1) + lane;
  const bool dthread = lq < 2;
  const uint32_t tl = lane_base(tbase);
  const uint64_t wlim = g.wait_ns();  // tile waits (shortened only by the test hook)
  float* zsnap = sm.arr();        // [2][64]: Z before the chunk, by chunk parity
  float* dzk = sm.arr() + 128;    // [4][64]: column sums of the prepared chunk's phi(K)
  float* dzr = sm.arr() + 384;    // [4][64]: the chunk's column sums of gd phi(Q)
  float* rsum = sm.arr() + 640;   // [4][128]: quarter-row parts of den
  float* gnum = sm.arr() + 1152;  // [4][128]: quarter-row parts of G . num

  // phi of a stage's tiles in place, the rounding errors into the lo tiles
  auto phi_stage = [&](int s, int nvalid) {
    float z[16];
    if (CAUSAL) {
      phi_quarter_split(sm.tile(s, kSK), sm.tile(s, kSKL), row, qc, nvalid, z);
      const float cs = warp_column_sums16(z);
      if (lane < 16) dzk[lq * 64 + 16 * qc + lane] = cs;
    }
    phi_quarter_split(sm.tile(s, kSQ), sm.tile(s, kSQL), row, qc, kC, z);
    fence_proxy_async_smem();
  };
  float zrun = 0.f, zinc = 0.f, rr = 0.f;  // Z[d], the chunk's phi(K) column sums, r[d] (tid < 64)
  // The state a segment starts from: the snapshot, and the carry. The carry is the
  // dS accumulator itself: the dS MMAs of a segment add into it, its hi-part rows
  // (TMEM lanes 0-63, row d = drow) seeded with the prefix and its lo-part rows
  // (lanes 64-127) with zeros, so that S before a chunk is the sum of the two.
  auto start_item = [&](int item, int bh) {
    const float* src = sprefix + (size_t)(CAUSAL ? item : bh) * kStateFloats;
    float v[16];
    if (dthread) {  // the prefix is S^T [m][d]: column drow, rows m of this quarter
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = src[(16 * qc + j) * kDim + drow];
      store_split_quarter(sm.s_hi(), sm.s_lo(), drow, qc, v);
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = 0.f;
    }
    if (CAUSAL) {
      uint32_t u[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) u[j] = __float_as_uint(v[j]);
      tmem_st16(tl + kFS + 16 * qc, u);
    }
    if (tid < kDim) zrun = src[kDim * kDim + tid];
    fence_proxy_async_smem();
  };

  // Hand the MMA warp chunk cc's operands: Z and the state snapshot before the
  // chunk (a segment's first chunk had its state set up by start_item), phi of its
  // tiles being in already.
  auto state_in = [&](const FullCursor& c, long long nc) {
    if (tid < kDim) {
      if (CAUSAL && !c.first()) zrun += zinc;
      if (CAUSAL) zinc = (dzk[tid] + dzk[64 + tid]) + (dzk[128 + tid] + dzk[192 + tid]);
      zsnap[64 * (nc & 1) + tid] = zrun;
    }
    fence_before_sync();  // the previous chunk's TMEM reads, before this chunk's first group
    warp_arrive(sm.bar(QSmem::kG1Ready));
  };

  FullCursor cc;
  cc.start(g, true);
  FullCursor cn = cc;  // the chunk after cc
  cn.advance(g);
  long long n = 0;
  bool bad = false;
  if (cc.valid(g)) {
    if (warp_wait(sm.bar(QSmem::kFull + (0)), 0, abort, hdr, 21, wlim)) {
      phi_stage(0, min(kC, g.N - cc.chunk * kC));
      start_item(cc.item, cc.bh);
    } else {
      bad = true;
    }
  }
  // The loop is left only where all workers agree (a named-barrier reduction of
  // their failure flags): a warp whose wait ran out skips its work and its
  // arrivals until the next such point, so that no worker waits at a named
  // barrier for one that has left.
  if (!workers_any(bad)) {
    if (cc.valid(g)) state_in(cc, 0);
    while (cc.valid(g)) {
      const int item = cc.item, bh = cc.bh, t0 = cc.chunk * kC;
      const bool last = cc.last();
      const int nvalid = min(kC, g.N - t0);
      const int s = (int)(n & 1);
      const uint32_t ph = (uint32_t)(n & 1);
      uint8_t* qt = sm.tile(s, kSQ);
      uint8_t* kt = sm.tile(s, kSK);
      uint8_t* vt = sm.tile(s, kSV);
      uint8_t* gt = sm.tile(s, kSG);
      uint8_t* klt = sm.tile(s, kSKL);
      uint8_t* qlt = sm.tile(s, kSQL);
      const float* zs = zsnap + 64 * s;

      // ---- epilogue of the first group: den, G.num
      if (!bad && warp_wait(sm.bar(QSmem::kG1Done), ph, abort, hdr, 22)) {
        fence_after_sync();
        // the partial sums run in two lanes (even and odd columns), added at the end
        float2 dp = make_float2(0.f, 0.f), np = make_float2(0.f, 0.f);
        if (CAUSAL && qc <= lq) {  // warp-uniform; slice qc of P and W in two 16-column halves
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t rp[16], rw[16];
            tmem_ld16x2(tl + kFP + 32 * qc + 16 * h, rp, tl + kFW + 32 * qc + 16 * h, rw);
            if (qc < lq) {  // below the diagonal block: nothing is masked
#pragma unroll
              for (int c = 0; c < 16; c += 2) {
                const float2 pp = make_float2(__uint_as_float(rp[c]), __uint_as_float(rp[c + 1]));
                dp = add2(dp, pp);
                np = fma2(pp, make_float2(__uint_as_float(rw[c]), __uint_as_float(rw[c + 1])), np);
              }
            } else {
#pragma unroll
              for (int c = 0; c < 16; c += 2) {
                const int j = 32 * qc + 16 * h + c;
                const float2 pp = make_float2(j <= row ? __uint_as_float(rp[c]) : 0.f,
                                              j + 1 <= row ? __uint_as_float(rp[c + 1]) : 0.f);
                dp = add2(dp, pp);
                np = fma2(pp, make_float2(__uint_as_float(rw[c]), __uint_as_float(rw[c + 1])), np);
              }
            }
          }
        }
        {  // G_i . (phi(Q_i) S_prev) and phi(Q_i) . Z_prev over this quarter. The Z dot
           // uses the same bf16 phi(Q) as the MMAs for P and phi(Q) S_prev, so that
           // the rounding of phi(Q) cancels in num / den.
          uint32_t ro[16], ro2[16];
          tmem_ld16x2(tl + kFO + 16 * qc, ro, tl + kFO + 64 + 16 * qc, ro2);
          float gv[16], qv[16];
          load_row16(gt, row, 2 * qc, gv);
          load_row16(qt, row, 2 * qc, qv);
#pragma unroll
          for (int q = 0; q < 16; q += 2) {
            const float2 o = add2(make_float2(__uint_as_float(ro[q]), __uint_as_float(ro[q + 1])),
                                  make_float2(__uint_as_float(ro2[q]), __uint_as_float(ro2[q + 1])));
            np = fma2(make_float2(gv[q], gv[q + 1]), o, np);
            dp = fma2(make_float2(qv[q], qv[q + 1]), *reinterpret_cast<const float2*>(zs + 16 * qc + q), dp);
          }
        }
        const float dpart = dp.x + dp.y, npart = np.x + np.y;
        rsum[qc * 128 + row] = dpart;
        gnum[qc * 128 + row] = npart;
        fence_before_sync();
      } else {
        bad = true;
      }
      if (workers_any(bad)) break;  // partials visible; every read of P and O is done
      fence_after_sync();

      // ---- gd, gN (into the G and the spent V tiles), T_L (over the spent P)
      float gd;
      {
        const float den = (rsum[row] + rsum[128 + row]) + (rsum[256 + row] + rsum[384 + row]);
        const float inv = 1.f / den;
        gd = -((gnum[row] + gnum[128 + row]) + (gnum[256 + row] + gnum[384 + row])) * inv * inv;
        if (CAUSAL) {  // T_L = W / den + gd (j <= i), bf16 hi + lo
          uint32_t th[16], tlo[16];
          if (qc <= lq) {  // warp-uniform: full slice or diagonal slice
            uint32_t rw[16], rw2[16];
            tmem_ld16x2(tl + kFW + 32 * qc, rw, tl + kFW + 32 * qc + 16, rw2);
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              const int j0 = 32 * qc + 2 * c;
              const float2 t = fma2(make_float2(__uint_as_float(c < 8 ? rw[2 * c] : rw2[2 * c - 16]),
                                                __uint_as_float(c < 8 ? rw[2 * c + 1] : rw2[2 * c - 15])),
                                    make_float2(inv, inv), make_float2(gd, gd));
              split_bf16(qc < lq || j0 <= row ? t.x : 0.f, qc < lq || j0 + 1 <= row ? t.y : 0.f, th[c],
                         tlo[c]);
            }
          } else {
#pragma unroll
            for (int c = 0; c < 16; ++c) th[c] = tlo[c] = 0u;
          }
          tmem_st16(tl + kFT + 16 * qc, th);
          tmem_st16(tl + kFT + 64 + 16 * qc, tlo);
        }
        if (!CAUSAL || warp_wait(sm.bar(QSmem::kDsDone), ph, abort, hdr, 27)) {  // dS has read V
          float gn[16];
          load_row16(gt, row, 2 * qc, gn);
#pragma unroll
          for (int q = 0; q < 16; q += 2) {
            const float2 x = mul2(make_float2(gn[q], gn[q + 1]), make_float2(inv, inv));
            gn[q] = x.x;
            gn[q + 1] = x.y;
          }
          store_split_quarter(gt, vt, row, qc, gn);
          fence_proxy_async_smem();
          fence_before_sync();
          warp_arrive(sm.bar(QSmem::kG2Ready));
          if (qc == 0 && row < nvalid) {
            den_out[(size_t)bh * g.N + t0 + row] = den;
            gd_out[(size_t)bh * g.N + t0 + row] = gd;
          }
          // this chunk's share of r = sum_i gd_i phi(Q_i) (float32 phi = hi + lo)
          float qv[16], ql[16], z[16];
          load_row16(qt, row, 2 * qc, qv);
          load_row16(qlt, row, 2 * qc, ql);
#pragma unroll
          for (int q = 0; q < 16; q += 2) {
            const float2 x = mul2(make_float2(gd, gd), add2(make_float2(qv[q], qv[q + 1]),
                                                            make_float2(ql[q], ql[q + 1])));
            z[q] = x.x;
            z[q + 1] = x.y;
          }
          const float cs = warp_column_sums16(z);
          if (lane < 16) dzr[lq * 64 + 16 * qc + lane] = cs;
        } else {
          bad = true;
        }
      }

      // ---- while the second group runs: phi of the next chunk, the state carry
      if (!bad && cn.valid(g)) {
        if (warp_wait(sm.bar(QSmem::kFull + (s ^ 1)), (uint32_t)(((n + 1) >> 1) & 1), abort, hdr, 21, wlim))
          phi_stage(s ^ 1, min(kC, g.N - cn.chunk * kC));
        else
          bad = true;
      }
      // the V tile (gN lo) is free once the segment sums have read it: the lo-part
      // rows of dS pass through it to the carry's threads
      float4* xs = reinterpret_cast<float4*>(vt);  // [64][16] float4, XOR-swizzled rows
      if (!bad) {
        if (warp_wait(sm.bar(QSmem::kGnFree), ph, abort, hdr, 28)) {
          fence_after_sync();
          if (CAUSAL && !last && !dthread) {
            uint32_t r[16];
            tmem_ld16(tl + kFS + 16 * qc, r);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              xs[drow * 16 + ((4 * qc + j) ^ (drow & 15))] =
                  make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                              __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
          }
          // the next segment's starting state (the snapshot is no MMA's operand now)
          if (last && cn.valid(g)) start_item(cn.item, cn.bh);
        } else {
          bad = true;
        }
      }
      if (workers_any(bad)) break;
      if (tid < kDim) rr += (dzr[tid] + dzr[64 + tid]) + (dzr[128 + tid] + dzr[192 + tid]);
      if (CAUSAL && !last && dthread) {  // the next snapshot: hi rows from TMEM, lo rows exchanged
        uint32_t r[16];
        tmem_ld16(tl + kFS + 16 * qc, r);
        float v[16];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float4 lo = xs[drow * 16 + ((4 * qc + j) ^ (drow & 15))];
          v[4 * j] = __uint_as_float(r[4 * j]) + lo.x;
          v[4 * j + 1] = __uint_as_float(r[4 * j + 1]) + lo.y;
          v[4 * j + 2] = __uint_as_float(r[4 * j + 2]) + lo.z;
          v[4 * j + 3] = __uint_as_float(r[4 * j + 3]) + lo.w;
        }
        store_split_quarter(sm.s_hi(), sm.s_lo(), drow, qc, v);
      }
      // the next chunk's first group can start (it waits for dphiQ's reads below
      // only before phi(Q) S_prev)
      if (cn.valid(g)) state_in(cn, n + 1);

      // ---- dq = (dphiQ + gd Z_prev) * phi'(q), phi'(q) = min(phi(q), 1); this
      // quarter's columns, staged in 128 x 32 float32 boxes (128-byte swizzle) for
      // TMA stores in the chunk's spent K and phi(K) lo tiles
      if (warp_wait(sm.bar(QSmem::kG2Done), ph, abort, hdr, 24)) {
        fence_after_sync();
        uint32_t r[16], r2[16];
        tmem_ld16x2(tl + kFQ + 16 * qc, r, tl + kFQ + 64 + 16 * qc, r2);
        fence_before_sync();
        warp_arrive(sm.bar(QSmem::kDqRead));
        float qv[16], o[16];
        load_row16(qt, row, 2 * qc, qv);
#pragma unroll
        for (int q = 0; q < 16; q += 2) {
          const float2 t = fma2(make_float2(gd, gd), *reinterpret_cast<const float2*>(zs + 16 * qc + q),
                                add2(make_float2(__uint_as_float(r[q]), __uint_as_float(r[q + 1])),
                                     make_float2(__uint_as_float(r2[q]), __uint_as_float(r2[q + 1]))));
          const float2 x = mul2(t, make_float2(fminf(qv[q], 1.f), fminf(qv[q + 1], 1.f)));
          o[q] = x.x;
          o[q + 1] = x.y;
        }
        uint8_t* sq = qc < 2 ? kt : klt;
#pragma unroll
        for (int c = 0; c < 4; ++c)
          *reinterpret_cast<float4*>(sq + sw128(row, (qc & 1) * 64 + c * 16)) =
              make_float4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
        fence_proxy_async_smem();
        if (!last) warp_arrive(sm.bar(QSmem::kStReady));
      } else {
        bad = true;
      }
      if (last) {  // segment partial: R = sum phi(Q)^T gN (rows d), r
        // lane 32 lq + lane holds row d = 32 (lq % 2) + lane: hi part for lq < 2, lo
        // part for lq >= 2; the lo parts pass through the spent G tile
        float4* xr = reinterpret_cast<float4*>(gt);
        uint32_t r[16];
        if (!bad) {
          tmem_ld16(tl + kFR + 16 * qc, r);
          if (!dthread) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
              xr[drow * 16 + ((4 * qc + j) ^ (drow & 15))] =
                  make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                              __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
          }
        }
        if (workers_any(bad)) break;
        float* dst = rpartial + (size_t)item * kStateFloats;
        if (dthread) {
          float4* d4 = reinterpret_cast<float4*>(dst + drow * kDim + 16 * qc);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float4 lo = xr[drow * 16 + ((4 * qc + j) ^ (drow & 15))];
            d4[j] = make_float4(__uint_as_float(r[4 * j]) + lo.x, __uint_as_float(r[4 * j + 1]) + lo.y,
                                __uint_as_float(r[4 * j + 2]) + lo.z, __uint_as_float(r[4 * j + 3]) + lo.w);
          }
        }
        if (tid < kDim) {
          dst[kDim * kDim + tid] = rr;
          rr = 0.f;
        }
        warp_arrive(sm.bar(QSmem::kStReady));  // the G tile too is done with now
      }
      ++n;
      cc = cn;
      cn.advance(g);
    }
  }
}

template <bool CAUSAL>
__global__ void __launch_bounds__(kWsThreads, 1)
tc_bwd_q_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
                const __grid_constant__ CUtensorMap tm_dq, Geometry g,
                const float* __restrict__ sprefix, float* __restrict__ rpartial,
                float* __restrict__ den_out, float* __restrict__ gd_out, WorkspaceHeader* hdr) {
  extern __shared__ uint8_t smraw[];
  QSmem sm(smraw);
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  if (tid == 0) {
    mbar_init(sm.bar(QSmem::kFull + (0)), 1);
    mbar_init(sm.bar(QSmem::kFull + (1)), 1);
    mbar_init(sm.bar(QSmem::kG1Ready), kWorkers / 32);
    mbar_init(sm.bar(QSmem::kG2Ready), kWorkers / 32);
    mbar_init(sm.bar(QSmem::kStReady), kWorkers / 32);
    mbar_init(sm.bar(QSmem::kG1Done), 1);
    mbar_init(sm.bar(QSmem::kDsDone), 1);
    mbar_init(sm.bar(QSmem::kGnFree), 1);
    mbar_init(sm.bar(QSmem::kG2Done), 1);
    mbar_init(sm.bar(QSmem::kDqRead), kWorkers / 32);
    mbar_init(sm.bar(QSmem::kDrain), 1);
    *sm.abort() = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(sm.tslot(), 512);
    tmem_relinquish();
  }
  sync_tc();
  const uint32_t tbase = *sm.tslot();
  pdl_wait();
  volatile int* abort = sm.abort();
  if (warp >= kWorkers / 32) {
    regs_dec<kControlRegs>();
    if (lane == 0) {
      if (warp == kMmaWarp)
        bwd_q_mma<CAUSAL>(sm, g, tbase, abort, hdr);
      else if (warp == kTmaWarp)
        bwd_q_tma<CAUSAL>(sm, g, &tm_q, &tm_k, &tm_v, &tm_g, &tm_dq, abort, hdr);
    }
    __syncwarp();
  } else {
    regs_inc<kWorkerRegs>();
    bwd_q_workers<CAUSAL>(sm, g, tbase, abort, sprefix, rpartial, den_out, gd_out, hdr);
  }
  pdl_trigger();
  sync_tc();
  if (warp == 0) tmem_dealloc(tbase, 512);
}

// --------------------------------------------------- reverse direction: dk, dv
//
// Key rows j on the TMEM lanes: P^T = phi(K) phi(Q)^T, W^T = V G^T, and
// T^T_ji = W^T_ji / den_i + gd_i with den_i, gd_i saved by the forward-direction
// kernel.

// Masked slice sl of a 128-column fp32 TMEM matrix -> packed bf16. LOWER keeps
// j <= row (query rows), otherwise i >= row (key rows).
template <bool LOWER>
__device__ __forceinline__ void masked_pack_slice(uint32_t taddr, int sl, int lq, int row, uint32_t (&hi)[16]) {
  const bool any = LOWER ? sl <= lq : sl >= lq;
  if (any) {  // warp-uniform
    uint32_t r[32];
    tmem_ld32(taddr + 32 * sl, r);
    if (sl != lq) {  // off the diagonal block: nothing is masked
#pragma unroll
      for (int c = 0; c < 16; ++c) hi[c] = pack_bf16(__uint_as_float(r[2 * c]), __uint_as_float(r[2 * c + 1]));
    } else {
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const int j0 = 32 * sl + 2 * c;
        const bool k0 = LOWER ? j0 <= row : j0 >= row;
        const bool k1 = LOWER ? j0 + 1 <= row : j0 + 1 >= row;
        hi[c] = pack_bf16(k0 ? __uint_as_float(r[2 * c]) : 0.f, k1 ? __uint_as_float(r[2 * c + 1]) : 0.f);
      }
    }
  } else {
#pragma unroll
    for (int c = 0; c < 16; ++c) hi[c] = 0u;
  }
}

// phi with the float32 exponential on columns [16 qc, 16 qc + 16) of a tile row,
// in place; rows >= nvalid become zero.
__device__ __forceinline__ void phi_quarter_exact(uint8_t* tile, int row, int qc, int nvalid) {
  const bool valid = row < nvalid;
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    uint4* p = reinterpret_cast<uint4*>(tile + sw128(row, (2 * qc + c) * 16));
    const uint4 w = *p;
    *p = valid ? make_uint4(phi2_bf16_exact(w.x), phi2_bf16_exact(w.y), phi2_bf16_exact(w.z),
                            phi2_bf16_exact(w.w))
               : make_uint4(0, 0, 0, 0);
  }
}

// The gradients accumulate as two 64-column parts each (the hi*lo partner
// products of a hi/lo pair sit side by side in N = 128 MMAs) and are summed in
// the epilogue.
constexpr uint32_t kRP = 0;     // 128: P^T (rows keys), then bf16 P_L^T in [0, 64) and T_L^T hi in [64, 128)
constexpr uint32_t kRH = 64;    // bf16 hi part of T_L^T
constexpr uint32_t kRT = 128;   // 128: W^T = V G^T, spent by the first epilogue
constexpr uint32_t kRV = 128;   // 128: dV parts (over W^T)
constexpr uint32_t kRK = 256;   // 128: dphiK parts
constexpr uint32_t kRR = 384;   // 64: this chunk's phi(Q)^T gN (M = 64 layout)
constexpr uint32_t kRL = 448;   // 64: bf16 lo part of T_L^T

template <bool CAUSAL>
__global__ void __launch_bounds__(kBTQ, 1)
tc_bwd_kv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
                 const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                 Geometry g, const float* __restrict__ rsuffix, const float* __restrict__ den_in,
                 const float* __restrict__ gd_in, WorkspaceHeader* hdr) {
  extern __shared__ uint8_t smraw[];
  BwdSmem sm(smraw);
  // the state snapshot buffers hold R rows d (m contiguous)
  float* rsnap = sm.arr;         // 64: r before the chunk
  float* gds = sm.arr + 64;      // 128: gd_i
  float* invs = sm.arr + 192;    // 128: 1 / den_i
  float* dz = sm.arr + 320;      // [4][64]
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int lq = warp & 3, qc = warp >> 2;
  const int row = lq * 32 + lane;  // key row for the gradients, query row for gN
  // R carry: row d = 32 (lq % 2) + lane, held by the threads of TMEM lanes 0-63
  const int drow = 32 * (lq & 1) + lane;
  const bool dthread = lq < 2;
  // threads 0 and 64 issue the MMAs; the TMA loads and stores (and the waits on
  // the stores) belong to warp 1's first thread, so that they issue in parallel
  const bool tma_thread = tid == 32;

  if (tid == 0) {
    for (int s = 0; s < kBwdStages; ++s) mbar_init(&sm.full[s], 1);
    mbar_init(sm.mma_bar, 1);
    mbar_init(&sm.sbar[1], 1);
    mbar_init(sm.drain, 2);  // thread 0's and the second group's issuer's MMAs
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(sm.tslot, 512);
    tmem_relinquish();
  }
  sync_tc();
  const uint32_t tbase = *sm.tslot;
  const uint32_t tl = lane_base(tbase);
  pdl_wait();

  const uint32_t tx = (CAUSAL ? 4 : 2) * kTile;
  RevCursor cc, cp;
  cc.start(g);
  cp.start(g);
  long long issued = 0;
  auto issue = [&](RevCursor& c) {
    const int s = issued % kBwdStages;
    const int bh = c.bh, t0 = c.chunk * kC;
    mbar_arrive_expect_tx(&sm.full[s], tx);
    tma_load_3d(sm.tile(s, kK), &tm_k, &sm.full[s], 0, t0, bh);
    tma_load_3d(sm.tile(s, kV), &tm_v, &sm.full[s], 0, t0, bh);
    if (CAUSAL) {
      tma_load_3d(sm.tile(s, kQ), &tm_q, &sm.full[s], 0, t0, bh);
      tma_load_3d(sm.tile(s, kG), &tm_g, &sm.full[s], 0, t0, bh);
    }
    ++issued;
    c.advance(g);
  };
  if (tma_thread)
    for (int i = 0; i < kBwdStages - 1 && cp.valid(g); ++i) issue(cp);
  // the state terms, first into the gradient accumulators: dV = phi(K) [R_hi | R_lo]
  // (B = R rows d read MN-major, n = m contiguous; hi and lo tiles la - ha apart)
  // and dphiK = V [R_hi; R_lo]^T (B = R rows d read K-major, the lo rows after the hi)
  auto issue_state_dv = [&](uint32_t ka, uint32_t ha, uint32_t la) {
    const uint32_t idVn = idesc_bf16(128, 128, false, true);
#pragma unroll
    for (int k = 0; k < 4; ++k)
      mma_ss(tbase + kRV, sdesc(ka + k * 32, 16, 1024), sdesc(ha + k * 2048, la - ha, 1024), idVn, k);
  };
  auto issue_state_dk = [&](uint32_t va, uint32_t ha) {
    const uint32_t idKn = idesc_bf16(128, 128, false, false);
#pragma unroll
    for (int k = 0; k < 4; ++k)
      mma_ss(tbase + kRK, sdesc(va + k * 32, 16, 1024), sdesc(ha + k * 32, 16, 1024), idKn, k);
  };

  float rrun[16];  // R row drow, columns [16 qc, 16 qc + 16) (dthread)
  float rr = 0.f;  // r[d] for d = tid < 64
  long long consumed = 0;
  uint32_t ph = 0, sph = 0;
  float z[16];
  // den_i, gd_i of the chunk being processed, loaded one chunk ahead
  float nden = 1.f, ngd = 0.f;
  auto fetch_dg = [&](const RevCursor& c) {
    if (CAUSAL && tid < kC && c.valid(g)) {
      const int t = c.chunk * kC + tid;
      const bool valid = t < g.N;
      const size_t at = (size_t)c.bh * g.N + t;
      nden = valid ? den_in[at] : 1.f;
      ngd = valid ? gd_in[at] : 0.f;
    }
  };
  fetch_dg(cc);

  while (cc.valid(g)) {
    const int item = cc.item, bh = cc.bh, t0 = cc.chunk * kC;
    const bool first = cc.chunk == cc.cend - 1;  // first processed
    const int nvalid = min(kC, g.N - t0);
    if (CAUSAL && tid < kC) {
      invs[tid] = 1.f / nden;
      gds[tid] = ngd;
    }
    if (first) {
      const float* src = rsuffix + (size_t)(CAUSAL ? item : bh) * kStateFloats;
      if (dthread) {
        const float4* s4 = reinterpret_cast<const float4*>(src + drow * kDim + 16 * qc);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 x = s4[q];
          rrun[4 * q] = x.x;
          rrun[4 * q + 1] = x.y;
          rrun[4 * q + 2] = x.z;
          rrun[4 * q + 3] = x.w;
        }
      }
      if (tid < kDim) rr = src[kDim * kDim + tid];
    }
    if ((CAUSAL || first) && dthread) store_split_quarter(sm.s_hi, sm.s_lo, drow, qc, rrun);
    if (tid < kDim) rsnap[tid] = rr;
    const int s = consumed % kBwdStages;
    uint8_t* qt = sm.tile(s, kQ);
    uint8_t* kt = sm.tile(s, kK);
    uint8_t* vt = sm.tile(s, kV);
    uint8_t* gt = sm.tile(s, kG);
    if (!wait_uniform(&sm.full[s], (consumed / kBwdStages) & 1, hdr, 31)) break;
    phi_quarter_exact(kt, row, qc, nvalid);
    if (CAUSAL) {
      phi_quarter_split(qt, sm.qlo, row, qc, kC, z);
      // gN (query row = row) for this quarter, and this chunk's share of r
      const float inv = invs[row];
      const float gdr = gds[row];
      float gn[16];
      load_row16(gt, row, 2 * qc, gn);
#pragma unroll
      for (int q = 0; q < 16; q += 2) {
        const float2 x = mul2(make_float2(gn[q], gn[q + 1]), make_float2(inv, inv));
        const float2 y = mul2(make_float2(z[q], z[q + 1]), make_float2(gdr, gdr));
        gn[q] = x.x;
        gn[q + 1] = x.y;
        z[q] = y.x;
        z[q + 1] = y.y;
      }
      store_split_quarter(sm.gn_hi, sm.gn_lo, row, qc, gn);
      const float cs = warp_column_sums16(z);
      if (lane < 16) dz[lq * 64 + 16 * qc + lane] = cs;
    }
    fence_proxy_async_smem();
    sync_tc();
    if (tma_thread) {
      // the next chunk's tiles go into the previous chunk's stage, whose dk / dv
      // staging TMA stores have had this chunk's phi to finish reading it
      bulk_wait_read<0>();
      if (cp.valid(g)) issue(cp);
    }
    if (tid == 0) {
      const uint32_t qa = smem_u32(qt), ka = smem_u32(kt), va = smem_u32(vt);
      const uint32_t ha = smem_u32(sm.s_hi), la = smem_u32(sm.s_lo);
      if (CAUSAL) {
        const uint32_t idP = idesc_bf16(128, 128, false, false);
#pragma unroll
        for (int k = 0; k < 4; ++k)  // P^T = phi(K) phi(Q)^T
          mma_ss(tbase + kRP, sdesc(ka + k * 32, 16, 1024), sdesc(qa + k * 32, 16, 1024), idP, k);
        const uint32_t ga = smem_u32(gt);
#pragma unroll
        for (int k = 0; k < 4; ++k)  // W^T = V G^T
          mma_ss(tbase + kRT, sdesc(va + k * 32, 16, 1024), sdesc(ga + k * 32, 16, 1024), idP, k);
      }
      if (!CAUSAL) {  // causal: dphiK's after the R sums, dV's in the second group
        issue_state_dv(ka, ha, la);
        issue_state_dk(va, ha);
      }
      mma_commit(sm.mma_bar);
    }
    {  // the next chunk's den, gd: their latency hides behind the first MMA group
      RevCursor nx = cc;
      nx.advance(g);
      fetch_dg(nx);
    }
    // phi'(k) of this quarter row, read before the barrier that precedes the dk / dv
    // staging writes into the K tile
    float kv[16];
    if (!CAUSAL) load_row16(kt, row, 2 * qc, kv);
    if (!wait_uniform(sm.mma_bar, ph, hdr, 32)) break;
    ph ^= 1;
    fence_after_sync();

    if (CAUSAL) {
      if (tid == kG2Issuer) {
        // this chunk's phi(Q)^T gN, awaited when the state is updated, issued while
        // the other warps run the epilogue below (warp 2's slice of it, query
        // columns 0-31 of key rows 64-95, is masked out entirely): phi(Q)^T hi
        // and lo stacked as one M = 128 MN-major operand (ql - qa bytes apart)
        // times gN hi, then gN lo; rows d of the hi part in TMEM lanes 0-63, of
        // the lo part in lanes 64-127
        const uint32_t qa = smem_u32(qt), lbo = smem_u32(sm.qlo) - qa;
        const uint32_t gha = smem_u32(sm.gn_hi), gla = smem_u32(sm.gn_lo);
        const uint32_t idR = idesc_bf16(128, 64, true, true);
#pragma unroll
        for (int k = 0; k < kC / 16; ++k)
          mma_ss(tbase + kRR, sdesc(qa + k * 2048, lbo, 1024), sdesc(gha + k * 2048, 1024, 1024),
                 idR, k);
#pragma unroll
        for (int k = 0; k < kC / 16; ++k)
          mma_ss(tbase + kRR, sdesc(qa + k * 2048, lbo, 1024), sdesc(gla + k * 2048, 1024, 1024),
                 idR, 1);
        mma_commit(&sm.sbar[1]);
        // dphiK's state term (its accumulator is free: the previous chunk's dk was read)
        issue_state_dk(smem_u32(vt), smem_u32(sm.s_hi));
      }
      // key row keeps query columns i >= row; slice qc of P^T and of T^T
      uint32_t pph[16], pth[16], ptl[16];
      masked_pack_slice<false>(tl + kRP, qc, lq, row, pph);  // P_L^T enters the MMA as bf16
      // T^T_ji = W^T_ji / den_i + gd_i (column-dependent scale and shift)
      if (qc >= lq) {  // warp-uniform
        uint32_t r[32];
        tmem_ld32(tl + kRT + 32 * qc, r);
        if (qc != lq) {  // below the diagonal block: nothing is masked
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const int i0 = 32 * qc + 2 * c;
            const float2 t = fma2(make_float2(__uint_as_float(r[2 * c]), __uint_as_float(r[2 * c + 1])),
                                  *reinterpret_cast<const float2*>(invs + i0),
                                  *reinterpret_cast<const float2*>(gds + i0));
            split_bf16(t.x, t.y, pth[c], ptl[c]);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const int i0 = 32 * qc + 2 * c;
            const float2 t = fma2(make_float2(__uint_as_float(r[2 * c]), __uint_as_float(r[2 * c + 1])),
                                  *reinterpret_cast<const float2*>(invs + i0),
                                  *reinterpret_cast<const float2*>(gds + i0));
            split_bf16(i0 >= row ? t.x : 0.f, i0 + 1 >= row ? t.y : 0.f, pth[c], ptl[c]);
          }
        }
      } else {
#pragma unroll
        for (int c = 0; c < 16; ++c) pth[c] = ptl[c] = 0u;
      }
      sync_tc();  // all reads of P^T, T^T done before the bf16 parts overwrite them
      tmem_st16(tl + kRP + 16 * qc, pph);
      tmem_st16(tl + kRH + 16 * qc, pth);
      tmem_st16(tl + kRL + 16 * qc, ptl);
      sync_tc();
      {  // R_run += this chunk's phi(Q)^T gN and r += sum gd phi(Q) (the sums were
         // issued under the epilogue above); the lo-part rows (lanes 64-127) pass through
         // the chunk's G tile (no MMA reads it any more). Their threads hand them over
         // through named barrier 1 without waiting, and one of them then issues the
         // second group, so the hi-part threads' update runs under that issue.
        if (!wait_uniform(&sm.sbar[1], sph, hdr, 34)) break;
        sph ^= 1;
        fence_after_sync();
        uint32_t r[16];
        tmem_ld16(tl + kRR + 16 * qc, r);
        float4* xs = reinterpret_cast<float4*>(gt);  // [64][16] float4, XOR-swizzled rows
        if (!dthread) {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            xs[drow * 16 + ((4 * qc + j) ^ (drow & 15))] =
                make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                            __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
          named_arrive_all();
          if (tid == kG2Issuer) {
            const uint32_t qa = smem_u32(qt), ql = smem_u32(sm.qlo);
            const uint32_t gha = smem_u32(sm.gn_hi), gla = smem_u32(sm.gn_lo);
            issue_state_dv(smem_u32(kt), smem_u32(sm.s_hi), smem_u32(sm.s_lo));
            const uint32_t idV2 = idesc_bf16(128, 128, false, true), idV = idesc_bf16(128, 64, false, true);
#pragma unroll
            for (int k = 0; k < kC / 16; ++k)  // dV += P_L^T [gN_hi | gN_lo] (N blocks gla - gha apart)
              mma_ts(tbase + kRV, tbase + kRP + k * 8, sdesc(gha + k * 2048, gla - gha, 1024), idV2, 1);
#pragma unroll
            for (int k = 0; k < kC / 16; ++k)  // dphiK += T_hi^T [phi(Q)_hi | phi(Q)_lo]
              mma_ts(tbase + kRK, tbase + kRH + k * 8, sdesc(qa + k * 2048, ql - qa, 1024), idV2, 1);
#pragma unroll
            for (int k = 0; k < kC / 16; ++k)  // + T_lo^T phi(Q)_hi
              mma_ts(tbase + kRK, tbase + kRL + k * 8, sdesc(qa + k * 2048, 1024, 1024), idV, 1);
            mma_commit(sm.mma_bar);
          }
        } else {
          named_sync_all();
        }
        if (dthread) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float4 lo = xs[drow * 16 + ((4 * qc + j) ^ (drow & 15))];
            rrun[4 * j] += __uint_as_float(r[4 * j]) + lo.x;
            rrun[4 * j + 1] += __uint_as_float(r[4 * j + 1]) + lo.y;
            rrun[4 * j + 2] += __uint_as_float(r[4 * j + 2]) + lo.z;
            rrun[4 * j + 3] += __uint_as_float(r[4 * j + 3]) + lo.w;
          }
        }
        if (tid < kDim) rr += dz[tid] + dz[64 + tid] + dz[128 + tid] + dz[192 + tid];
      }
      load_row16(kt, row, 2 * qc, kv);
      if (!wait_uniform(sm.mma_bar, ph, hdr, 33)) break;
      ph ^= 1;
      fence_after_sync();
    }

    // dk = (dphiK + r_next) * phi'(k) and dv, this quarter's columns, staged in 128 x 32
    // float32 boxes (128-byte swizzle) for TMA stores in the chunk's spent tiles: dk in
    // V / G, dv in Q / K (the R MMAs that read Q ran before the second group, whose
    // completion was awaited)
    {
      uint8_t* sk = qc < 2 ? vt : gt;
      uint8_t* sv = qc < 2 ? qt : kt;
      {
        uint32_t w[16], w2[16];
        tmem_ld16x2(tl + kRV + 16 * qc, w, tl + kRV + 64 + 16 * qc, w2);
#pragma unroll
        for (int c = 0; c < 4; ++c)
          *reinterpret_cast<float4*>(sv + sw128(row, (qc & 1) * 64 + c * 16)) = make_float4(
              __uint_as_float(w[4 * c]) + __uint_as_float(w2[4 * c]),
              __uint_as_float(w[4 * c + 1]) + __uint_as_float(w2[4 * c + 1]),
              __uint_as_float(w[4 * c + 2]) + __uint_as_float(w2[4 * c + 2]),
              __uint_as_float(w[4 * c + 3]) + __uint_as_float(w2[4 * c + 3]));
      }
      uint32_t r[16], r2[16];
      tmem_ld16x2(tl + kRK + 16 * qc, r, tl + kRK + 64 + 16 * qc, r2);
      float o[16];
#pragma unroll
      for (int q = 0; q < 16; q += 2) {
        const float2 t = add2(add2(make_float2(__uint_as_float(r[q]), __uint_as_float(r[q + 1])),
                                   make_float2(__uint_as_float(r2[q]), __uint_as_float(r2[q + 1]))),
                              *reinterpret_cast<const float2*>(rsnap + 16 * qc + q));
        const float2 x = mul2(t, make_float2(fminf(kv[q], 1.f), fminf(kv[q + 1], 1.f)));
        o[q] = x.x;
        o[q + 1] = x.y;
      }
#pragma unroll
      for (int c = 0; c < 4; ++c)
        *reinterpret_cast<float4*>(sk + sw128(row, (qc & 1) * 64 + c * 16)) =
            make_float4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
    }
    fence_proxy_async_smem();
    sync_tc();
    if (tma_thread) {  // rows past the sequence end are clipped by the tensor maps
      tma_store_3d(&tm_dk, vt, 0, t0, bh);
      tma_store_3d(&tm_dk, gt, 32, t0, bh);
      tma_store_3d(&tm_dv, qt, 0, t0, bh);
      tma_store_3d(&tm_dv, kt, 32, t0, bh);
      bulk_commit();
    }
    ++consumed;
    cc.advance(g);
  }
  pdl_trigger();
  if (tma_thread) {
    while (consumed < issued) {
      const int s = consumed % kBwdStages;
      if (!mbar_wait(&sm.full[s], (consumed / kBwdStages) & 1)) record_timeout(hdr, 36);
      ++consumed;
    }
    bulk_wait_all<0>();
  }
  // every MMA of both issuing threads completes before TMEM is freed (time-bounded only)
  if (tid == 0 || tid == kG2Issuer) mma_commit(sm.drain);
  if (tid == 0 && !mbar_wait(sm.drain, 0)) record_timeout(hdr, 35);
  sync_tc();
  if (warp == 0) tmem_dealloc(tbase, 512);
}

size_t states_bytes(const Geometry& g) {
  return align_up(sizeof(float) * kStateFloats * (size_t)g.n_items(), 256);
}

}  // namespace
}  // namespace tcx

using namespace tcx;

size_t tc_backward_workspace(int BH, int N) {
  const Geometry g = make_geometry(BH, N);
  return kHeaderBytes + 4 * states_bytes(g) + 2 * align_up(sizeof(float) * (size_t)BH * N, 256);
}

namespace {

// The backward's workspace: header, then per-segment states (S partials and
// prefix, R partials and suffix), then den_i and gd_i per token.
struct BwdWork {
  WorkspaceHeader* hdr;
  float *spartial, *sprefix, *rpartial, *rsuffix, *den, *gd;
  BwdWork(void* ws, const Geometry& g, int BH, int N) {
    hdr = static_cast<WorkspaceHeader*>(ws);
    char* base = static_cast<char*>(ws) + kHeaderBytes;
    const size_t sb = states_bytes(g);
    spartial = reinterpret_cast<float*>(base);
    sprefix = reinterpret_cast<float*>(base + sb);
    rpartial = reinterpret_cast<float*>(base + 2 * sb);
    rsuffix = reinterpret_cast<float*>(base + 3 * sb);
    den = reinterpret_cast<float*>(base + 4 * sb);
    gd = den + align_up(sizeof(float) * (size_t)BH * N, 256) / sizeof(float);
  }
};

}  // namespace

cudaError_t tc_backward_q(const void* q, const void* k, const void* v, const void* dout,
                          float* dq, const StateIO* pre, const StateIO* own, int BH, int N,
                          bool causal, void* ws, cudaStream_t st, const FaultHook* fault,
                          const float* fwd_prefix) {
  const Geometry g = make_geometry(BH, N);
  Geometry gq = g;  // the forward-direction kernel's copy, with the test hook if any
  if (fault != nullptr) {
    gq.fault_load = fault->load;
    gq.fault_wait_ns = fault->wait_ns;
  }
  BwdWork w(ws, g, BH, N);
  CUtensorMap tq, tk, tv, tg, tdq;
  const uint64_t n = (uint64_t)N, bh = (uint64_t)BH;
  if (!make_tmap_bf16_3d(&tq, q, kDim, n, bh, kDim, kC, 1) ||
      !make_tmap_bf16_3d(&tk, k, kDim, n, bh, kDim, kC, 1) ||
      !make_tmap_bf16_3d(&tv, v, kDim, n, bh, kDim, kC, 1) ||
      !make_tmap_bf16_3d(&tg, dout, kDim, n, bh, kDim, kC, 1) ||
      !make_tmap_f32_3d(&tdq, dq, kDim, n, bh, 32, kC, 1))
    return cudaErrorInvalidValue;

  // the segment states before each segment: the forward's (same geometry, same inputs), or
  // computed here (segment increments in the psi form, then the prefix / total scan)
  const float* sprefix = fwd_prefix;
  cudaError_t e = cudaSuccess;
  if (sprefix == nullptr) {
    e = launch_segment_states(&tk, &tv, g, w.spartial, w.hdr, st);
    if (e != cudaSuccess) return e;
    e = launch_scan(w.spartial, w.sprefix, g, causal ? kScanPrefix : kScanTotal,
                    pre != nullptr ? *pre : StateIO{}, w.hdr, st);
    if (e != cudaSuccess) return e;
    sprefix = w.sprefix;
  }
  auto run_q = [&](auto kern) {
    cudaError_t err = configure(kern, kQSmem);
    if (err != cudaSuccess) return err;
    const int ctas = min(g.n_items(), resident_ctas(kern, kQSmem, kWsThreads) * sm_count());
    err = launch_pdl(kern, dim3(ctas), dim3(kWsThreads), kQSmem, st, tq, tk, tv, tg, tdq, gq,
                     sprefix, w.rpartial, w.den, w.gd, w.hdr);
    count_launches(1);
    return err != cudaSuccess ? err : cudaGetLastError();
  };
  e = causal ? run_q(tc_bwd_q_kernel<true>) : run_q(tc_bwd_q_kernel<false>);
  if (e != cudaSuccess || own == nullptr) return e;
  // the shard's own reverse sums: the total over its segments (rsuffix is scratch here)
  return launch_scan(w.rpartial, w.rsuffix, g, kScanTotal, *own, w.hdr, st);
}

cudaError_t tc_backward_kv(const void* q, const void* k, const void* v, const void* dout,
                           float* dk, float* dv, const StateIO* suf, int BH, int N, bool causal,
                           void* ws, cudaStream_t st) {
  const Geometry g = make_geometry(BH, N);
  BwdWork w(ws, g, BH, N);
  CUtensorMap tq, tk, tv, tg, tdk, tdv;
  const uint64_t n = (uint64_t)N, bh = (uint64_t)BH;
  if (!make_tmap_bf16_3d(&tq, q, kDim, n, bh, kDim, kC, 1) ||
      !make_tmap_bf16_3d(&tk, k, kDim, n, bh, kDim, kC, 1) ||
      !make_tmap_bf16_3d(&tv, v, kDim, n, bh, kDim, kC, 1) ||
      !make_tmap_bf16_3d(&tg, dout, kDim, n, bh, kDim, kC, 1) ||
      !make_tmap_f32_3d(&tdk, dk, kDim, n, bh, 32, kC, 1) ||
      !make_tmap_f32_3d(&tdv, dv, kDim, n, bh, 32, kC, 1))
    return cudaErrorInvalidValue;
  cudaError_t e = launch_scan(w.rpartial, w.rsuffix, g, causal ? kScanSuffix : kScanTotal,
                              suf != nullptr ? *suf : StateIO{}, w.hdr, st);
  if (e != cudaSuccess) return e;
  auto run_kv = [&](auto kern) {
    cudaError_t err = configure(kern, kBwdSmem);
    if (err != cudaSuccess) return err;
    const int ctas = min(g.n_items(), resident_ctas(kern, kBwdSmem, kBTQ) * sm_count());
    err = launch_pdl(kern, dim3(ctas), dim3(kBTQ), kBwdSmem, st, tq, tk, tv, tg, tdk, tdv, g,
                     (const float*)w.rsuffix, (const float*)w.den, (const float*)w.gd, w.hdr);
    count_launches(1);
    return err != cudaSuccess ? err : cudaGetLastError();
  };
  return causal ? run_kv(tc_bwd_kv_kernel<true>) : run_kv(tc_bwd_kv_kernel<false>);
}

cudaError_t tc_backward(const void* q, const void* k, const void* v, const void* dout, float* dq,
                        float* dk, float* dv, int BH, int N, bool causal, void* ws,
                        cudaStream_t st, const FaultHook* fault) {
  cudaError_t e = tc_backward_q(q, k, v, dout, dq, nullptr, nullptr, BH, N, causal, ws, st, fault);
  if (e != cudaSuccess) return e;
  return tc_backward_kv(q, k, v, dout, dk, dv, nullptr, BH, N, causal, ws, st);
}

}  // namespace la
