// Tensor-core (tcgen05 + TMEM + TMA) forward for bf16 inputs with D = M = 64.
//
// The sequence of each (batch, head) is cut into chunks of C = 128 tokens and
// the chunks into segments. Three kernels:
//
//  1. tc_state_kernel: per segment, the state increment
//       dS^T = V^T phi(K), dZ = sum_t phi(K_t)
//     ("Transformers are RNNs": S = sum_j phi(K_j) V_j^T, Z = sum_j phi(K_j);
//     nubint.ai review, "Proposed method"; zhengyuhong.cn deck, slide 3),
//     taken as phi(K) = 1 + psi(K): one tcgen05 group per chunk,
//     [V^T; 1^T] [psi(K) | 1] (M = 128 and N = 80 with stacked blocks of ones),
//     gives V^T psi(K), the column sums of V, and sum_t psi(K_t); then
//     dS^T[m][d] = (V^T psi(K))[m][d] + sum_t V[t][m], dZ[d] = sum_t psi + count.
//  2. state_scan_kernel: exclusive prefix over segments (causal; deck slide 4:
//     S_i = S_{i-1} + phi(K_i) V_i^T) or the full sum (non-causal), in float32;
//     optionally the final state for prefill.
//  3. tc_attend_kernel: per chunk, with S_prev / Z_prev the state before it,
//       causal:     num = (phi(Q) phi(K)^T (.) L) V + phi(Q) S_prev,
//                   den = rowsum((phi(Q) phi(K)^T) (.) L) + phi(Q) Z_prev
//       non-causal: num = phi(Q) S, den = phi(Q) Z
//     out = num / den. L is the inclusive lower-triangular mask (j <= i). The
//     chunk form is the parallel reading of the S/Z recurrence (paperlayer.ai
//     summary §3.3.2: training stays parallel); it equals it up to rounding.
//
// phi is applied in shared memory right after each TMA tile lands (bf16 in,
// float32 math, bf16 out). The carried state is float32; the read-out takes it
// rounded to bf16 (each element independently).
#include <cuda_bf16.h>

#include <map>
#include <mutex>
#include <utility>

#include "la_tc_common.cuh"

namespace la {
namespace tcx {

// ------------------------------------------------------- 1. segment states

constexpr int kStateWorkers = 256;  // two threads per tile row (column halves)
constexpr int kStateThreads = kStateWorkers + 32;  // + one control warp; 2 CTAs per SM
// Eight worker warps apply psi to the K tiles as they land; one control thread
// issues the loads and the MMAs, each as soon as what it needs is done (a
// stage is refilled once the MMAs that read it are done). A segment's sums land
// in one of two TMEM accumulators and are read out while the next one fills.
constexpr int kStateStages = 3;
constexpr int kStateStageBytes = 2 * kTile;  // K, V
constexpr int kStateSmem = 1024 + kStateStages * kStateStageBytes + 2048 + 256;

// IDENT: the K tiles hold the features f already (the identity feature map): the
// group then gives V^T f and sum_t f directly (features centred on zero, nothing
// to split off). Else inputs to which the elu + 1 map applies, in the psi form.
// VARLEN: per-stream lengths (lens or the packed layout); the items are then dealt
// by tickets: the control thread takes them as its loads reach them, the workers
// read each from the ring once its first tiles have landed and learn of the end
// from `loaded`.
template <bool IDENT, bool VARLEN>
__global__ void __launch_bounds__(kStateThreads, 2)
tc_state_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                Geometry g, float* __restrict__ partial, WorkspaceHeader* hdr) {
  constexpr int S = kStateStages, SB = kStateStageBytes;
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = sm;                        // [stage][K tile | V tile]
  uint8_t* ones = stages + S * SB;             // 16 x 64 bf16 ones (the stacked blocks)
  uint64_t* full = reinterpret_cast<uint64_t*>(ones + 2048);  // S: tiles landed
  uint64_t* empty = full + S;                  // S: the chunk's MMAs are done with the stage
  uint64_t* phid = empty + S;                  // S: every worker's psi of the stage is in
  uint64_t* segbar = phid + S;                 // 2: a segment's last MMAs are done
  uint64_t* drain = segbar + 2;                // every MMA of the CTA is done
  volatile int* abort = reinterpret_cast<volatile int*>(drain + 1);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(drain + 1) + 1;
  volatile int* ring = reinterpret_cast<volatile int*>(tslot + 1);  // kRing items (tickets)
  volatile int* loaded = ring + kRing;  // tickets: chunks loaded in all, once known (else -1)

  constexpr bool TICKETS = VARLEN;  // items dealt by tickets (else round robin)
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int q4 = warp & 3, h = (warp >> 2) & 1;
  const int trow = q4 * 32 + lane;  // tile row of this worker (column half h)
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&phid[s], kStateWorkers);
    }
    mbar_init(&segbar[0], 1);
    mbar_init(&segbar[1], 1);
    mbar_init(drain, 1);
    *abort = 0;
    *loaded = -1;
    fence_mbar_init();
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
  }
  for (int e = tid; e < 2048 / 16; e += blockDim.x)
    reinterpret_cast<uint4*>(ones)[e] = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
  fence_proxy_async_smem();
  if (warp == kStateWorkers / 32) {
    tmem_alloc(tslot, 256);  // accumulator p (segment parity) in columns [128 p, 128 p + 80)
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tbase = *tslot;
  pdl_wait();

  if (warp == kStateWorkers / 32) {
    // ------------------------------------------------------------- control
    if (lane == 0) {
      CursorT<VARLEN> cl, cm;  // next chunk to load, next chunk to multiply
      if constexpr (TICKETS) {
        cl.ring = cm.ring = ring;
        cl.counter = &hdr->tickets[0];
      }
      cl.start(g);
      cm.start(g);
      long long total = 0;  // chunks to process (with tickets not known in advance)
      if constexpr (TICKETS) {
        if (!cl.valid(g)) *loaded = 0;
      } else {
        for (CursorT<VARLEN> c = cl; c.valid(g); c.advance(g)) ++total;
      }
      long long nl = 0, nm = 0;
      int nseg = 0;
      const uint32_t oa = smem_u32(ones);
      uint64_t idle_since = globaltimer_ns();
      while (TICKETS ? (nm < nl || cl.valid(g)) : nm < total) {
        bool moved = false;
        if (nm < nl && mbar_test_wait(&phid[nm % S], (uint32_t)((nm / S) & 1))) {
          fence_after_sync();
          const int s = (int)(nm % S);
          const bool first = cm.first();
          const bool last = cm.last();
          const uint32_t acc = tbase + 128 * (nseg & 1);
          const uint32_t ka = smem_u32(stages + s * SB), va = ka + kTile;
          // [V^T; 1^T] (M = 128 MN-major, rows 64.. from the ones block) times
          // [psi(K) | 1] (N = 80 MN-major, columns 64.. from the ones block):
          // lanes 0-63 get (V^T psi(K))[m][d] in columns [0, 64) and the column
          // sum of V[:, m] in column 64; lanes 64-127 get sum_t psi(K)[t][d]. The
          // ones block of an operand is 16 token rows: every K step of 16 tokens
          // reads the same block, its descriptor's leading byte offset measured
          // from that step's start (oa - (va + 2048 k)).
          const uint32_t idS = idesc_bf16(128, 80, true, true);
#pragma unroll
          for (int k = 0; k < kC / 16; ++k)
            mma_ss(acc, sdesc(va + k * 2048, oa - (va + k * 2048), 1024),
                   sdesc(ka + k * 2048, oa - (ka + k * 2048), 1024), idS,
                   (first && k == 0) ? 0u : 1u);
          mma_commit(&empty[s]);
          if (last) mma_commit(&segbar[nseg++ & 1]);
          cm.advance(g);
          ++nm;
          moved = true;
        }
        if ((TICKETS ? cl.valid(g) : nl < total) &&
            (nl < S || mbar_test_wait(&empty[nl % S], (uint32_t)(((nl - S) / S) & 1)))) {
          const int s = (int)(nl % S);
          uint8_t* st = stages + s * SB;
          mbar_arrive_expect_tx(&full[s], 2 * kTile);
          int y, z;
          cl.tile_yz(g, y, z);
          tma_load_3d(st, &tm_k, &full[s], 0, y, z);
          tma_load_3d(st + kTile, &tm_v, &full[s], 0, y, z);
          cl.advance(g);
          ++nl;
          if constexpr (TICKETS) {
            if (!cl.valid(g)) *loaded = (int)nl;
          }
          moved = true;
        }
        if (moved) {
          idle_since = globaltimer_ns();
        } else if (*abort) {
          break;
        } else if (globaltimer_ns() - idle_since > kWaitLimitNs) {
          *abort = 1;
          record_timeout(hdr, 4);
          break;
        } else {
          __nanosleep(32);
        }
      }
      // every issued load lands and every MMA completes before the CTA lets go of
      // its shared memory and TMEM (time-bounded only: not cut short by the abort flag)
      for (long long k = nl > S ? nl - S : 0; k < nl; ++k)
        if (!mbar_wait(&full[k % S], (uint32_t)((k / S) & 1))) record_timeout(hdr, 3);
      mma_commit(drain);
      if (!mbar_wait(drain, 0)) record_timeout(hdr, 5);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------- workers
    // a segment's sums -> partial[item]: S^T [m][d], then Z [d]
    auto readout = [&](int item, int p) {
      float* dst = partial + (size_t)item * kStateFloats;
      const uint32_t acc = lane_base(tbase) + 128 * p;
      uint32_t r[32];
      tmem_ld32(acc + h * 32, r);
      // lanes 0..63: row m = lane of V^T psi(K) (columns d) plus the column sum of
      // V[:, m] (column 64); lanes 64..127: sum_t psi(K)[t][d] (every lane alike),
      // plus the segment's count of valid tokens. This thread writes columns
      // [32h, 32h + 32) of its row.
      if (q4 < 2 || (q4 == 2 && lane == 0)) {
        float add = 0.f;  // identity features: the sums are the state itself
        if (q4 < 2) {
          uint32_t r16[16];
          tmem_ld16(acc + 64, r16);
          if (!IDENT) add = __uint_as_float(r16[0]);
        } else if (!IDENT) {
          const int c0 = g.chunk_begin(item), c1 = g.chunk_end(item);
          add = (float)max(0, min(g.len(g.bh_of(item)) - c0 * kC, (c1 - c0) * kC));
        }
        float4* d4 = reinterpret_cast<float4*>(dst + (q4 < 2 ? (32 * q4 + lane) * kDim : kDim * kDim) + h * 32);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          d4[j] = make_float4(__uint_as_float(r[4 * j]) + add, __uint_as_float(r[4 * j + 1]) + add,
                              __uint_as_float(r[4 * j + 2]) + add, __uint_as_float(r[4 * j + 3]) + add);
      }
    };

    CursorT<VARLEN> cc;
    if constexpr (TICKETS)
      cc.ring = ring;
    else
      cc.start(g);
    bool fresh = TICKETS;             // the next chunk starts an item still to be read
    long long consumed = 0;
    int nseg = 0;                    // segments whose last chunk has passed
    int pend_item = -1, pend_p = 0;  // segment awaiting its readout
    uint32_t pend_phase = 0;
    bool ok = true;
    while (TICKETS || cc.valid(g)) {
      // the chunk's item (with tickets known only once its tiles have landed)
      int item = 0, bh = 0, nvalid = 0;
      bool last = false;
      if constexpr (!TICKETS) {
        item = cc.item;
        bh = cc.bh;
        nvalid = min(kC, (VARLEN ? cc.n : g.N) - cc.chunk * kC);
        last = cc.last();
      }
      const int s = consumed % S;
      uint8_t* kt = stages + s * SB;
      uint8_t* vt = kt + kTile;
      if constexpr (TICKETS) {
        const int r = mbar_wait_warp_or_end(&full[s], (uint32_t)((consumed / S) & 1), abort, hdr, 1,
                                            loaded, consumed);
        if (r == 0) {
          ok = false;
          break;
        }
        if (r == 2) break;
        if (fresh) {
          cc.take(g);
          fresh = false;
        }
        item = cc.item;
        bh = cc.bh;
        nvalid = min(kC, cc.n - cc.chunk * kC);
        last = cc.last();
      } else if (!mbar_wait_warp(&full[s], (uint32_t)((consumed / S) & 1), abort, hdr, 1)) {
        ok = false;
        break;
      }
      if (IDENT)
        zero_half_if_past(kt, trow, h, nvalid);
      else
        psi_half(kt, trow, h, nvalid);
      if (nvalid < kC) zero_half_if_past(vt, trow, h, nvalid);
      fence_proxy_async_smem();
      mbar_arrive(&phid[s]);
      // the segment that ended with the previous chunk: its accumulator is not the
      // one this chunk's MMAs use
      if (pend_item >= 0) {
        if (!mbar_wait_warp(&segbar[pend_p], pend_phase, abort, hdr, 2)) {
          ok = false;
          break;
        }
        fence_after_sync();
        readout(pend_item, pend_p);
        fence_before_sync();
        pend_item = -1;
      }
      if (last) {
        pend_item = item;
        pend_p = nseg & 1;
        pend_phase = (uint32_t)((nseg >> 1) & 1);
        ++nseg;
      }
      ++consumed;
      if constexpr (!TICKETS)
        cc.advance(g);
      else if (last)
        fresh = true;
      else
        ++cc.chunk;
    }
    if (ok && pend_item >= 0 && mbar_wait_warp(&segbar[pend_p], pend_phase, abort, hdr, 2)) {
      fence_after_sync();
      readout(pend_item, pend_p);
      fence_before_sync();
    }
  }
  pdl_trigger();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (warp == kStateWorkers / 32) tmem_dealloc(tbase, 256);
}

// ----------------------------------------------------------- 2. segment scan

// mode kScanPrefix:  out[seg][bh] = S0 + sum_{s < seg} partial[s][bh]  (causal, forward)
// mode kScanTotal:   out[bh]      = sum_s partial[s][bh]               (non-causal)
// mode kScanSuffix:  out[seg][bh] = S0 + sum_{s > seg} partial[s][bh]  (causal, reverse)
// S0 is the entry's initial state when io.read_init (prefix and suffix modes),
// else 0; with io.S set and io.write_final the full sum (S0 + all segments) is
// written to the entry: S [d][m], Z [d]. The partials are S^T [m][d] (the
// segment-state kernel's) or, with io.rows_are_d, R [d][m] (the backward's).
// Two forms. Few sequences: one thread per state element; the segment loads are
// issued in batches of 8 so the walk over segments is not a chain of dependent
// global loads. Many sequences (short ones, as in a serving batch): a block per
// sequence, each thread holding 9 elements and the entry passed through shared
// memory whole (read and written in its own [d][m] order), so that a block's few
// dependent loads (slot, entry, partials) cover a whole state.
constexpr int kScanThreads = 128;
constexpr int kScanSeqThreads = 512;
constexpr int kScanPer = (kStateFloats + kScanSeqThreads - 1) / kScanSeqThreads;  // 9

// the sequence's state entry (prefill, extend); a slot outside the pool is reported
__device__ __forceinline__ bool scan_entry(const StateIO& io, int bh, bool report,
                                           WorkspaceHeader* hdr, size_t& entry) {
  entry = (size_t)bh;
  if (io.S == nullptr) return false;
  if (io.slots == nullptr) return true;
  const int slot = io.slots[bh / io.H];
  entry = (size_t)slot * io.H + bh % io.H;
  const bool ok = slot >= 0 && slot < io.pool;
  if (!ok && report) atomicExch(&hdr->status, (int)LA_ERR_INVALID_ARG);
  return ok;
}

// the segments that hold tokens: with per-stream lengths, the segments past the
// stream's last chunk were skipped by the segment-state kernel (their sums are zero
// and never written)
__device__ __forceinline__ int scan_segments(const Geometry& g, int bh) {
  if (g.lens == nullptr && g.cu == nullptr) return g.n_seg;
  return min(g.n_seg, ((g.len(bh) + kC - 1) / kC + g.seg_chunks - 1) / g.seg_chunks);
}

__global__ void __launch_bounds__(kScanThreads)
state_scan_kernel(const float* __restrict__ partial, float* __restrict__ out, Geometry g,
                  int mode, StateIO io, WorkspaceHeader* hdr) {
  const int bh = blockIdx.y;
  const int e = blockIdx.x * kScanThreads + threadIdx.x;
  const int BH = g.BH;
  pdl_wait();
  if (e >= kStateFloats) return;
  const int n_seg = scan_segments(g, bh);
  size_t entry;
  const bool entry_ok = scan_entry(io, bh, e == 0, hdr, entry);
  // e < 4096: S^T [m][d] (or R [d][m]); else Z [e - 4096]
  const int m = io.rows_are_d ? e % kDim : e / kDim, d = io.rows_are_d ? e / kDim : e % kDim;
  float* cell = !entry_ok ? nullptr
                          : (e < kDim * kDim ? io.S + entry * kDim * kDim + d * kDim + m
                                             : io.Z + entry * kDim + (e - kDim * kDim));
  float run = (cell != nullptr && io.read_init && mode != kScanTotal) ? *cell : 0.f;
  const bool rev = mode == kScanSuffix;
  // a forward prefix with no entry to write needs no sums of the last segment
  const int n_read = (mode == kScanPrefix && io.S == nullptr) ? n_seg - 1 : n_seg;
  for (int s0 = 0; s0 < n_seg; s0 += 8) {
    float x[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int sg = rev ? n_seg - 1 - (s0 + j) : s0 + j;
      x[j] = s0 + j < n_read ? partial[((size_t)sg * BH + bh) * kStateFloats + e] : 0.f;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (s0 + j < n_seg) {
        const int sg = rev ? n_seg - 1 - (s0 + j) : s0 + j;
        if (mode != kScanTotal) out[((size_t)sg * BH + bh) * kStateFloats + e] = run;
        run += x[j];
      }
    }
  }
  if (mode == kScanTotal) out[(size_t)bh * kStateFloats + e] = run;
  if (cell != nullptr && io.write_final) *cell = run;
}

// The per-sequence form: block bh, elements t + 512 i (i < 9) in the partials' order.
__global__ void __launch_bounds__(kScanSeqThreads)
state_scan_seq_kernel(const float* __restrict__ partial, float* __restrict__ out, Geometry g,
                      int mode, StateIO io, WorkspaceHeader* hdr) {
  __shared__ float st[kDim * (kDim + 1) + kDim];  // the entry: S [d][m] (rows padded), then Z
  const int bh = blockIdx.x, t = threadIdx.x;
  const int BH = g.BH;
  pdl_wait();
  const int n_seg = scan_segments(g, bh);
  size_t entry;
  const bool entry_ok = scan_entry(io, bh, t == 0, hdr, entry);
  // element e -> its cell of the entry in shared memory
  auto cell = [&](int e) {
    if (e >= kDim * kDim) return kDim * (kDim + 1) + (e - kDim * kDim);
    const int m = io.rows_are_d ? e % kDim : e / kDim, d = io.rows_are_d ? e / kDim : e % kDim;
    return d * (kDim + 1) + m;
  };
  float run[kScanPer];
  const bool init = entry_ok && io.read_init && mode != kScanTotal;
  if (init) {
    const float* S = io.S + entry * kDim * kDim;
#pragma unroll
    for (int i = 0; i < kScanPer; ++i) {
      const int p = t + kScanSeqThreads * i;  // entry order: S [d][m], then Z
      if (p < kDim * kDim)
        st[(p / kDim) * (kDim + 1) + p % kDim] = S[p];
      else if (p < kStateFloats)
        st[kDim * (kDim + 1) + (p - kDim * kDim)] = io.Z[entry * kDim + (p - kDim * kDim)];
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < kScanPer; ++i) {
    const int e = t + kScanSeqThreads * i;
    run[i] = (init && e < kStateFloats) ? st[cell(e)] : 0.f;
  }
  const bool rev = mode == kScanSuffix;
  // a forward prefix with no entry to write needs no sums of the last segment
  const int n_read = (mode == kScanPrefix && io.S == nullptr) ? n_seg - 1 : n_seg;
  for (int j = 0; j < n_seg; ++j) {
    const int sg = rev ? n_seg - 1 - j : j;
    const float* src = partial + ((size_t)sg * BH + bh) * kStateFloats;
    float* dst = out + ((size_t)sg * BH + bh) * kStateFloats;
    float x[kScanPer];
#pragma unroll
    for (int i = 0; i < kScanPer; ++i) {
      const int e = t + kScanSeqThreads * i;
      x[i] = (e < kStateFloats && j < n_read) ? src[e] : 0.f;
    }
#pragma unroll
    for (int i = 0; i < kScanPer; ++i) {
      const int e = t + kScanSeqThreads * i;
      if (e < kStateFloats) {
        if (mode != kScanTotal) dst[e] = run[i];
        run[i] += x[i];
      }
    }
  }
#pragma unroll
  for (int i = 0; i < kScanPer; ++i) {
    const int e = t + kScanSeqThreads * i;
    if (mode == kScanTotal && e < kStateFloats) out[(size_t)bh * kStateFloats + e] = run[i];
  }
  if (entry_ok && io.write_final) {
    if (init) __syncthreads();  // every read of the staged entry is done
#pragma unroll
    for (int i = 0; i < kScanPer; ++i) {
      const int e = t + kScanSeqThreads * i;
      if (e < kStateFloats) st[cell(e)] = run[i];
    }
    __syncthreads();
    float* S = io.S + entry * kDim * kDim;
#pragma unroll
    for (int i = 0; i < kScanPer; ++i) {
      const int p = t + kScanSeqThreads * i;
      if (p < kDim * kDim)
        S[p] = st[(p / kDim) * (kDim + 1) + p % kDim];
      else if (p < kStateFloats)
        io.Z[entry * kDim + (p - kDim * kDim)] = st[kDim * (kDim + 1) + (p - kDim * kDim)];
    }
  }
}

// --------------------------------------------------------- 3. chunk attention

constexpr int kAttStages = 2;  // 2 CTAs per SM
// S^T rows (64), then [Z; 0 x 15] rows (16): together the N = 80 B operand of
// phi(Q) [S^T; Z; 0]^T; then 16 rows of ones (the stacked block that adds the
// row sums of P_L and the column sums of phi(K) to the MMAs that need them)
constexpr int kSnapBytes = kDim * 128 + 16 * 128 + 16 * 128;
constexpr int kAttSmem = 1024 + kAttStages * 3 * kTile + kSnapBytes + 2048;

// TMEM columns (256 per CTA, two CTAs per SM). P is written first, and the
// second group, issued once P is read, writes the output over P's dead upper
// half; the state increment has columns of its own, so that it can be formed
// while P is read and read while the second group runs.
constexpr uint32_t kColP = 0;     // 128: phi(Q) phi(K)^T; then bf16 P_L in [0, 64)
constexpr uint32_t kColS = 192;   // 64: dS^T [m][d] in lanes 0-63, dZ[d] in lanes 64-127
constexpr uint32_t kColO = 64;    // 80: numerator in [64, 128), denominator in column 128
constexpr uint32_t kTmemCols = 256;

// 256 threads: warp w covers TMEM lane quarter w % 4 (rows 32 (w % 4) .. + 31)
// and half h = w / 4 of each row's columns, so every row is shared by two
// threads; two CTAs per SM. P is compacted in place (fp32 to bf16): all reads
// finish before a barrier, the writes follow it.
constexpr int kAttThreads = 256;
// the fused forward: clusters of one CTA per segment (the portable cluster size)
constexpr int kMaxFusedSegments = 8;

// VARLEN: per-stream lengths (lens or the packed layout): the items are dealt by
// tickets (the TMA thread takes them, a chunk ahead, and every thread reads them
// from the ring once a block barrier has passed since they were written), and in
// the packed layout a stream's last rows are stored one by one.
// FUSED: the whole forward in one launch for sequences of at most 8 segments: a
// thread-block cluster per sequence, one CTA per segment (the cluster rank). Each
// CTA first sums its segment's states in the psi form (what the segment-state
// kernel does), the CTAs then read the sums they need from each other's shared
// memory (causal: the segments before their own, in order; non-causal: all), and
// each attends over its own segment from that state; the states also go to the
// workspace, where the scan would have put them.
template <bool CAUSAL, bool IDENT, bool VARLEN, bool FUSED>
__global__ void __launch_bounds__(kAttThreads, 2)
tc_attend_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                 Geometry g, float* __restrict__ prefix, StateIO io, bool direct,
                 WorkspaceHeader* hdr) {
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = sm;  // [stage][Q | K | V]
  uint8_t* snap = sm + kAttStages * 3 * kTile;
  uint8_t* s_hi = snap;
  uint8_t* zrow = snap + kDim * 128;
  uint8_t* ones = zrow + 16 * 128;
  uint8_t* misc = snap + kSnapBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(misc);  // kAttStages
  uint64_t* mma_bar = full + kAttStages;
  uint64_t* drain = mma_bar + 1;  // every MMA of the CTA is done (end of the kernel)
  uint64_t* sbar = drain + 1;     // the chunk's state increment
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sbar + 1);
  volatile int* ring = reinterpret_cast<volatile int*>(tslot + 1);  // kRing items (tickets)

  constexpr bool TICKETS = VARLEN;  // items dealt by tickets (else round robin)
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int q4 = warp & 3, h = warp >> 2;
  const int row = q4 * 32 + lane;   // chunk row (query) of this thread
  // the state carry: lane quarters 0, 1 hold S^T row m = row, the first lane
  // of quarter 2 holds Z (the TMEM lanes the stacked increment lands in)
  const bool sthread = q4 < 2;
  const bool zthread = q4 == 2 && lane == 0;
  // thread 0 issues the MMAs but the state increment's, which warp 4's first
  // thread issues while the others read P (warp 4's share of that epilogue, key
  // columns 64-127 of query rows 0-31, is masked out entirely); the TMA loads
  // and stores (and the waits on the stores) belong to warp 1's first thread
  const bool tma_thread = tid == 32;
  constexpr int kSIssuer = 128;
  // the per-stream-length kernels keep the increment in thread 0's first group
  // and read it with P (the later read costs them registers they do not have)
  constexpr bool kLateS = !VARLEN;
  if (tid == 0) {
    for (int s = 0; s < kAttStages; ++s) mbar_init(&full[s], 1);
    mbar_init(mma_bar, 1);
    mbar_init(sbar, 1);
    mbar_init(drain, 2);  // the MMAs of both issuing threads
    fence_mbar_init();
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_o);
    if (CAUSAL) {
      prefetch_tensormap(&tm_k);
      prefetch_tensormap(&tm_v);
    }
  }
  // rows 1..15 of the [Z; 0...] operand stay zero; the ones operand is constant
  for (int e = tid; e < 16 * 128 / 16; e += blockDim.x) {
    reinterpret_cast<uint4*>(zrow)[e] = make_uint4(0, 0, 0, 0);
    reinterpret_cast<uint4*>(ones)[e] = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
  }
  if (warp == 0) {
    tmem_alloc(tslot, kTmemCols);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tbase = *tslot;
  const uint32_t tl = lane_base(tbase);
  pdl_wait();

  // bad row offsets (or a stream longer than N) and, on the one-chunk path, slots
  // outside the pool are reported for every stream, also for those without tokens
  // (whose items the cursor skips)
  if (VARLEN && (g.cu != nullptr || (direct && io.slots != nullptr))) {
    for (int b = blockIdx.x * kAttThreads + tid; b < g.BH / g.H; b += gridDim.x * kAttThreads) {
      bool bad = g.cu != nullptr && !g.span_ok(b * g.H);
      if (direct && io.slots != nullptr) bad |= io.slots[b] < 0 || io.slots[b] >= io.pool;
      if (bad) atomicExch(&hdr->status, (int)LA_ERR_INVALID_ARG);
    }
  }
  const uint32_t tx_bytes = CAUSAL ? 3 * kTile : kTile;
  const uint64_t wlim = g.wait_ns();  // main-loop wait limit (shortened only by the test hook)
  // items last to first: the segment-state kernel just streamed k and v first to last
  // (with tickets first to last: the items past short streams' ends, which hold no
  // chunk, are then the last ones handed out)
  CursorT<VARLEN> cc, cp;
  if constexpr (TICKETS) {
    cc.ring = cp.ring = ring;
    cp.counter = &hdr->tickets[1];
  } else if constexpr (!FUSED) {
    cc.start(g, true);
    cp.start(g, true);
  }
  // [V^T; 1^T] (M = 128 MN-major, rows 64.. from the ones block) times phi(K)
  // (N = 64 MN-major): dS^T [m][d] in lanes 0-63, dZ[d] in lanes 64-127
  auto issue_ds = [&](uint32_t va, uint32_t ka, uint32_t oa) {
    const uint32_t idS = idesc_bf16(128, 64, true, true);
#pragma unroll
    for (int k = 0; k < kC / 16; ++k)
      mma_ss(tbase + kColS, sdesc(va + k * 2048, oa - (va + k * 2048), 1024),
             sdesc(ka + k * 2048, 1024, 1024), idS, k);
  };
  long long issued = 0;
  auto issue = [&](CursorT<VARLEN>& c) {
    if (g.faulty() && issued == g.fault_load) {  // test hook: this load is withheld
      ++issued;
      c.advance(g);
      return;
    }
    const int s = issued % kAttStages;
    uint8_t* st = stages + s * 3 * kTile;
    int y, z;
    c.tile_yz(g, y, z);
    mbar_arrive_expect_tx(&full[s], tx_bytes);
    tma_load_3d(st, &tm_q, &full[s], 0, y, z);
    if (CAUSAL) {
      tma_load_3d(st + kTile, &tm_k, &full[s], 0, y, z);
      tma_load_3d(st + 2 * kTile, &tm_v, &full[s], 0, y, z);
    }
    ++issued;
    c.advance(g);
  };
  if (!FUSED && tma_thread) {
    if constexpr (TICKETS) cp.start(g);
    for (int i = 0; i < kAttStages - 1 && cp.valid(g); ++i) issue(cp);
  }
  if constexpr (TICKETS) {
    __syncthreads();
    cc.start(g);
  }

  // running state: S^T row `row` (sthread) or Z (zthread), columns [32h, 32h + 32)
  float srun[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) srun[j] = 0.f;

  bool ok = true;
  long long consumed = 0;
  uint32_t mma_phase = 0, s_phase = 0;
  if constexpr (FUSED) {
    // ---------------------------------------------------------------- fused
    const int nseg = g.n_seg, seg = (int)cluster_ctarank(), bh = blockIdx.x / nseg;
    const int item = seg * g.BH + bh;
    const int c0 = g.chunk_begin(item), c1 = g.chunk_end(item);
    // the segment's sums, fp32 in the partials' layout: S^T [m][d] in stage 0's Q
    // slot, Z [d] in the snapshot area (both free until the attention starts)
    float* pS = reinterpret_cast<float*>(stages);
    float* pZ = reinterpret_cast<float*>(s_hi);
    // causal: nobody reads the last segment's sums
    if (!CAUSAL || seg + 1 < nseg) {
      auto load_kv = [&](int c) {
        if (g.faulty() && issued == g.fault_load) {  // test hook: this load is withheld
          ++issued;
          return;
        }
        const int st = issued % kAttStages;
        uint8_t* base = stages + st * 3 * kTile;
        mbar_arrive_expect_tx(&full[st], 2 * kTile);
        tma_load_3d(base + kTile, &tm_k, &full[st], 0, c * kC, bh);
        tma_load_3d(base + 2 * kTile, &tm_v, &full[st], 0, c * kC, bh);
        ++issued;
      };
      int nl = c0;
      if (tma_thread)
        for (int i = 0; i < kAttStages && nl < c1; ++i) load_kv(nl++);
      for (int c = c0; c < c1; ++c) {
        const int s = consumed % kAttStages;
        uint8_t* kt = stages + s * 3 * kTile + kTile;
        uint8_t* vt = kt + kTile;
        if (!wait_uniform(&full[s], (consumed / kAttStages) & 1, hdr, 16, wlim)) {
          ok = false;
          break;
        }
        const int nvalid = min(kC, g.N - c * kC);
        psi_half(kt, row, h, nvalid);
        if (nvalid < kC) zero_half_if_past(vt, row, h, nvalid);
        fence_proxy_async_smem();
        fence_before_sync();
        __syncthreads();
        fence_after_sync();
        if (tid == 0) {
          // [V^T; 1^T] [psi(K) | 1] (M = 128, N = 80, both MN-major, the ones block
          // standing in for rows 64.. and columns 64..): lanes 0-63 get
          // (V^T psi(K))[m][d] and the column sum of V[:, m] (column 64), lanes
          // 64-127 the column sums of psi(K)
          const uint32_t ka = smem_u32(kt), va = smem_u32(vt), oa = smem_u32(ones);
          const uint32_t idS = idesc_bf16(128, 80, true, true);
#pragma unroll
          for (int k = 0; k < kC / 16; ++k)
            mma_ss(tbase + kColP, sdesc(va + k * 2048, oa - (va + k * 2048), 1024),
                   sdesc(ka + k * 2048, oa - (ka + k * 2048), 1024), idS,
                   (c == c0 && k == 0) ? 0u : 1u);
          mma_commit(mma_bar);
        }
        // (waiting here for the chunk's MMAs, and refilling its stage right after,
        // measured faster than deferring both by a chunk)
        if (!wait_uniform(mma_bar, mma_phase, hdr, 17, wlim)) {
          ok = false;
          break;
        }
        mma_phase ^= 1;
        fence_after_sync();
        ++consumed;
        if (tma_thread && nl < c1) load_kv(nl++);  // into the stage just released
      }
      if (ok) {  // the sums -> pS, pZ (this thread's row m or Z, columns [32h, 32h + 32))
        uint32_t r[32];
        tmem_ld32(tl + kColP + 32 * h, r);
        if (sthread || zthread) {
          float add;
          if (sthread) {
            uint32_t r16[16];
            tmem_ld16(tl + kColP + 64, r16);
            add = __uint_as_float(r16[0]);  // sum of V[:, m]: the constant part of phi
          } else {
            add = (float)max(0, min(g.N - c0 * kC, (c1 - c0) * kC));  // the segment's tokens
          }
          float4* d4 = reinterpret_cast<float4*>(sthread ? pS + row * kDim + 32 * h : pZ + 32 * h);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            d4[j] = make_float4(__uint_as_float(r[4 * j]) + add, __uint_as_float(r[4 * j + 1]) + add,
                                __uint_as_float(r[4 * j + 2]) + add, __uint_as_float(r[4 * j + 3]) + add);
        }
      }
    }
    fence_before_sync();
    __syncwarp();
    cluster_sync();  // every CTA's sums are in its shared memory
    // the starting states, a slice of the state's elements per CTA: CTA q reads its
    // slice from every CTA's sums, adds them in segment order (as the scan kernel
    // does) and writes each CTA's starting state (causal: the sum over the segments
    // before it; non-causal: the total) into that CTA's shared memory and into the
    // workspace; every CTA then reads its own state locally
    float* rS = reinterpret_cast<float*>(stages + 3 * kTile);  // stage 1's Q slot
    float* rZ = pZ + kDim;
    {
      const int per = (kStateFloats + nseg - 1) / nseg;
      const int e1 = min(kStateFloats, (seg + 1) * per);
      for (int e = seg * per + tid; e < e1; e += kAttThreads) {
        const uint32_t src = smem_u32(e < kDim * kDim ? pS + e : pZ + (e - kDim * kDim));
        const uint32_t dst = smem_u32(e < kDim * kDim ? rS + e : rZ + (e - kDim * kDim));
        float x[kMaxFusedSegments];
#pragma unroll
        for (int r = 0; r < kMaxFusedSegments; ++r)
          x[r] = r < nseg ? ld_cluster_f32(cluster_map(src, (uint32_t)r)) : 0.f;
        float run = 0.f;
#pragma unroll
        for (int r = 0; r < kMaxFusedSegments; ++r) {
          if (r < nseg) {
            if (CAUSAL) {
              st_cluster_f32(cluster_map(dst, (uint32_t)r), run);
              prefix[((size_t)r * g.BH + bh) * kStateFloats + e] = run;
            }
            run += x[r];
          }
        }
        if (!CAUSAL) {
          for (int r = 0; r < nseg; ++r) st_cluster_f32(cluster_map(dst, (uint32_t)r), run);
          prefix[(size_t)bh * kStateFloats + e] = run;
        }
      }
    }
    __syncwarp();
    cluster_sync();  // every CTA's starting state is in its shared memory
    if (sthread || zthread) {
      const float4* s4 = reinterpret_cast<const float4*>(sthread ? rS + row * kDim + 32 * h : rZ + 32 * h);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float4 x = s4[j];
        srun[4 * j] = x.x;
        srun[4 * j + 1] = x.y;
        srun[4 * j + 2] = x.z;
        srun[4 * j + 3] = x.w;
      }
    }
    // the starting states were written into this CTA's stage memory through the
    // generic proxy (by other CTAs as well); the TMA loads that refill it below are
    // ordered after those writes
    fence_proxy_async_smem();
    fence_before_sync();
    __syncthreads();  // the stages are refilled only after these reads
    fence_after_sync();
    // the attention over this segment: one item per CTA
    cc.item = cp.item = item;
    cc.step = cp.step = (int)gridDim.x;
    cc.set_item(g);
    cp.set_item(g);
    cc.chunk = cp.chunk = c0;
    if (tma_thread && ok)
      for (int i = 0; i < kAttStages - 1 && cp.valid(g); ++i) issue(cp);
  }
  while (cc.valid(g) && ok) {
    const int item = cc.item;
    const int bh = cc.bh;
    const int t0 = cc.chunk * kC;
    const bool first = cc.first();
    const int nvalid = min(kC, (VARLEN ? cc.n : g.N) - t0);
    if (!CAUSAL && tma_thread && cp.valid(g)) {  // causal: issued with the first MMA group
      bulk_wait_read<0>();  // the stage being refilled was last read by an output store
      issue(cp);
    }
    // direct (causal, one chunk per sequence): the state before the chunk is the
    // sequence's entry in io (or zero), and the state after it goes back there
    size_t entry = (size_t)bh;
    bool entry_ok = direct && io.S != nullptr;
    if (entry_ok && io.slots != nullptr) {
      const int slot = io.slots[bh / io.H];
      entry_ok = slot >= 0 && slot < io.pool;
      entry = (size_t)slot * io.H + bh % io.H;
      if (!entry_ok && tid == 0) atomicExch(&hdr->status, (int)LA_ERR_INVALID_ARG);
    }
    if (direct) {  // S [entry][d][m]: this thread's row m = row, columns d of its half
      const bool init = entry_ok && io.read_init;
      if (sthread) {
        const float* src = io.S + entry * kDim * kDim + (size_t)(32 * h) * kDim + row;
#pragma unroll
        for (int j = 0; j < 32; ++j) srun[j] = init ? src[(size_t)j * kDim] : 0.f;
      } else if (zthread) {
#pragma unroll
        for (int j = 0; j < 32; ++j) srun[j] = init ? io.Z[entry * kDim + 32 * h + j] : 0.f;
      }
    } else if (!FUSED && first && (sthread || zthread)) {  // state before this segment
      const float* src = prefix + (size_t)(CAUSAL ? item : bh) * kStateFloats;
      const float4* s4 = reinterpret_cast<const float4*>(src + (sthread ? row * kDim : kDim * kDim) + 32 * h);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float4 x = s4[j];
        srun[4 * j] = x.x;
        srun[4 * j + 1] = x.y;
        srun[4 * j + 2] = x.z;
        srun[4 * j + 3] = x.w;
      }
    }
    const int s = consumed % kAttStages;
    uint8_t* qt = stages + s * 3 * kTile;
    uint8_t* kt = qt + kTile;
    uint8_t* vt = qt + 2 * kTile;
    // snapshot of the float32 state before this chunk, rounded to bf16, as
    // one K-major B operand of 80 rows: S^T rows m, then Z, then zero rows.
    // Each S element is rounded independently, so over the D-term dot
    // product phi(Q_i) . S[:, m] the rounding averages to ~2^-9 / sqrt(D).
    if ((CAUSAL || first) && (sthread || zthread)) {
      uint8_t* dst = sthread ? s_hi : zrow;
      const int r0 = sthread ? row : 0;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t hi[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) hi[q] = pack_bf16(srun[8 * c + 2 * q], srun[8 * c + 2 * q + 1]);
        *reinterpret_cast<uint4*>(dst + sw128(r0, (4 * h + c) * 16)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      }
    }
    if (!wait_uniform(&full[s], (consumed / kAttStages) & 1, hdr, 11, wlim)) {
      ok = false;
      break;
    }
    // phi(Q) with the packed-bf16 exponential: its rounding enters numerator and
    // denominator alike and largely cancels in out = num / den; phi(K) exact, since
    // the state sums phi(K) v^T over random-sign v (padded query rows are never stored)
    if (IDENT) {  // the tiles hold the features: only the rows past the end are cleared
      if (CAUSAL && nvalid < kC) {
        zero_half_if_past(kt, row, h, nvalid);
        zero_half_if_past(vt, row, h, nvalid);
      }
    } else {
      phi_half(qt, row, h, kC);
      if (CAUSAL) {
        phi_half<true>(kt, row, h, nvalid);
        if (nvalid < kC) zero_half_if_past(vt, row, h, nvalid);
      }
    }
    fence_proxy_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    // The ones block of an operand is 16 token rows: every K step of 16 tokens
    // reads the same block, its descriptor's leading byte offset measured from
    // that step's start (oa - (va + 2048 k)).
    if (tid == 0) {
      const uint32_t qa = smem_u32(qt), ka = smem_u32(kt), va = smem_u32(vt);
      const uint32_t ha = smem_u32(s_hi), oa = smem_u32(ones);
      if (CAUSAL) {
        const uint32_t idP = idesc_bf16(128, 128, false, false);
#pragma unroll
        for (int k = 0; k < 4; ++k)  // P = phi(Q) phi(K)^T
          mma_ss(tbase + kColP, sdesc(qa + k * 32, 16, 1024), sdesc(ka + k * 32, 16, 1024), idP, k);
        if (!kLateS) issue_ds(va, ka, oa);
      } else {  // num and den = phi(Q) [S^T; Z; 0]^T, the state being the total
        const uint32_t idO = idesc_bf16(128, 80, false, false);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_ss(tbase + kColO, sdesc(qa + k * 32, 16, 1024), sdesc(ha + k * 32, 16, 1024), idO, k);
      }
      mma_commit(mma_bar);
    }
    // causal: the next chunk's tiles are issued here, while thread 0 issues the
    // first MMA group, rather than at the top of the iteration, so that the output
    // store last read from that stage (issued at the end of the previous iteration)
    // has drained by now
    if (CAUSAL && tma_thread && cp.valid(g)) {
      bulk_wait_read<0>();
      issue(cp);
    }
    if (!wait_uniform(mma_bar, mma_phase, hdr, 12, wlim)) {
      ok = false;
      break;
    }
    mma_phase ^= 1;
    fence_after_sync();

    if (CAUSAL) {
      if (kLateS && tid == kSIssuer) {
        issue_ds(smem_u32(vt), smem_u32(kt), smem_u32(ones));
        mma_commit(sbar);
      }
      // masked P row -> bf16, written back over the first 64 TMEM columns; its
      // row sums (the intra-chunk part of den) come from an MMA with ones
      uint32_t pk[2][16];
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const int sl = 2 * h + t;
        if (sl <= q4) {  // warp-uniform: slices past the diagonal are all zero
          uint32_t r[32];
          tmem_ld32(tl + kColP + 32 * sl, r);
          if (sl < q4) {  // below the diagonal block: nothing is masked
#pragma unroll
            for (int c = 0; c < 16; ++c)
              pk[t][c] = pack_bf16(__uint_as_float(r[2 * c]), __uint_as_float(r[2 * c + 1]));
          } else {
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              const int j0 = 32 * sl + 2 * c;
              pk[t][c] = pack_bf16(j0 <= row ? __uint_as_float(r[2 * c]) : 0.f,
                                   j0 + 1 <= row ? __uint_as_float(r[2 * c + 1]) : 0.f);
            }
          }
        } else {
#pragma unroll
          for (int c = 0; c < 16; ++c) pk[t][c] = 0u;
        }
      }
      if (!kLateS && q4 <= 2) {  // state update: S^T += dS^T (row `row`), Z += dZ (TMEM lane 64)
        uint32_t r[32];
        tmem_ld32(tl + kColS + 32 * h, r);
        if (sthread || zthread) {
#pragma unroll
          for (int j = 0; j < 32; ++j) srun[j] += __uint_as_float(r[j]);
        }
      }
      fence_before_sync();
      __syncthreads();  // every read of fp32 P (and of the increment) is done before P_L overwrites it
      fence_after_sync();
#pragma unroll
      for (int t = 0; t < 2; ++t) tmem_st16(tl + kColP + 16 * (2 * h + t), pk[t]);
      fence_before_sync();
      __syncthreads();
      fence_after_sync();
      if (tid == 0) {
        const uint32_t va = smem_u32(vt), qa = smem_u32(qt), ha = smem_u32(s_hi);
        const uint32_t oa = smem_u32(ones);
        // phi(Q) [S^T; Z; 0]^T + P_L [V | 1] (N = 80; V's columns 64.. from the ones
        // block): the numerator in columns [0, 64) of kColO and the denominator
        // phi(Q) . Z_prev + rowsum(P_L) in column 64, from the same bf16 weights
        const uint32_t idO = idesc_bf16(128, 80, false, false);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_ss(tbase + kColO, sdesc(qa + k * 32, 16, 1024), sdesc(ha + k * 32, 16, 1024), idO, k);
        const uint32_t idPV = idesc_bf16(128, 80, false, true);
#pragma unroll
        for (int k = 0; k < kC / 16; ++k)
          mma_ts(tbase + kColO, tbase + kColP + k * 8, sdesc(va + k * 2048, oa - (va + k * 2048), 1024),
                 idPV, 1);
        mma_commit(mma_bar);
      }
      // state update while the second group runs: S^T += dS^T (row `row`), Z += dZ
      // (TMEM lane 64), this half's columns; a warp whose wait runs out leaves the
      // loop at the barrier below with the others
      bool sok = true;
      if (kLateS && q4 <= 2) {  // warp-uniform
        sok = __all_sync(0xffffffffu, mbar_wait(sbar, s_phase, wlim));
        if (sok) {
          fence_after_sync();
          uint32_t r[32];
          tmem_ld32(tl + kColS + 32 * h, r);
          if (sthread || zthread) {
#pragma unroll
            for (int j = 0; j < 32; ++j) srun[j] += __uint_as_float(r[j]);
          }
        }
      }
      if (kLateS) s_phase ^= 1;
      const bool gok = mbar_wait(mma_bar, mma_phase, wlim);
      if (!__syncthreads_and(sok && gok ? 1 : 0)) {
        if (tid == 0) record_timeout(hdr, sok ? 13 : 18);
        ok = false;
        break;
      }
      mma_phase ^= 1;
      fence_after_sync();
      if (entry_ok && io.write_final) {  // direct: the state after the sequence's only chunk
        if (sthread) {
          float* dst = io.S + entry * kDim * kDim + (size_t)(32 * h) * kDim + row;
#pragma unroll
          for (int j = 0; j < 32; ++j) dst[(size_t)j * kDim] = srun[j];
        } else if (zthread) {
#pragma unroll
          for (int j = 0; j < 32; ++j) io.Z[entry * kDim + 32 * h + j] = srun[j];
        }
      }
    }

    // out = num / den -> bf16, this half's columns, staged in the Q slot (all
    // MMAs reading it are done)
    {
      uint32_t oz[16], r[32];
      tmem_ld16_32(tl + kColO + 64, oz, tl + kColO + 32 * h, r);
      const float inv = 1.f / __uint_as_float(oz[0]);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 x = mul2(make_float2(__uint_as_float(r[8 * c + 2 * q]),
                                            __uint_as_float(r[8 * c + 2 * q + 1])),
                                make_float2(inv, inv));
          o[q] = pack_bf16(x.x, x.y);
        }
        *reinterpret_cast<uint4*>(qt + sw128(row, (4 * h + c) * 16)) = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
    fence_proxy_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (!VARLEN || g.cu == nullptr || nvalid == kC) {
      if (tma_thread) {
        int y, z;
        cc.tile_yz(g, y, z);
        tma_store_3d(&tm_o, qt, 0, y, z);
        bulk_commit();
      }
    } else if (nvalid > 0) {
      // packed layout, the stream's last chunk: its rows past the end belong to
      // the next stream, so only the valid rows are stored, 16 bytes at a time
      const size_t rs = (size_t)g.H * kDim;  // elements between token rows
      __nv_bfloat16* dst = g.out_rows + (size_t)(cc.r0 + t0) * rs + (size_t)cc.head * kDim;
      for (int u = tid; u < nvalid * 8; u += kAttThreads) {
        const int r = u >> 3, c = u & 7;
        *reinterpret_cast<uint4*>(dst + r * rs + 8 * c) =
            *reinterpret_cast<const uint4*>(qt + sw128(r, 16 * c));
      }
    }
    ++consumed;
    cc.advance(g);
  }
  pdl_trigger();
  if (tma_thread) {
    while (consumed < issued) {  // loads still in flight after an early exit
      const int s = consumed % kAttStages;
      if (!(g.faulty() && consumed == g.fault_load) &&
          !mbar_wait(&full[s], (consumed / kAttStages) & 1))
        record_timeout(hdr, 14);
      ++consumed;
    }
    bulk_wait_all<0>();
  }
  // every MMA of both issuing threads completes before TMEM is freed (time-bounded only)
  if (tid == 0 || tid == kSIssuer) mma_commit(drain);
  if (tid == 0 && !mbar_wait(drain, 0)) record_timeout(hdr, 15);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (warp == 0) tmem_dealloc(tbase, kTmemCols);
}

int sm_count() {
  static int n = [] {
    int dev = 0, v = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    return v > 0 ? v : 148;
  }();
  return n;
}

namespace {

// Items (segment-major: item = seg * BH + bh) are dealt round robin to G persistent
// CTAs. Returns the largest number of chunks and of items any CTA gets when each
// sequence of n_chunks chunks is cut into segments of s chunks (the last one shorter).
void deal(long long BH, long long n_chunks, long long s, long long G, long long& max_chunks,
          long long& max_items) {
  const long long n_seg = (n_chunks + s - 1) / s, last = n_chunks - (n_seg - 1) * s;
  const long long items = BH * n_seg, lo = items - BH;  // [lo, items): the short last segments
  max_chunks = max_items = 0;
  for (long long c = 0; c < G && c < items; ++c) {
    const long long n = (items - 1 - c) / G + 1;
    // items c + kG in [lo, items)
    const long long k0 = lo > c ? (lo - c + G - 1) / G : 0;
    const long long n_short = n > k0 ? n - k0 : 0;
    const long long chunks = n * s - n_short * (s - last);
    max_chunks = chunks > max_chunks ? chunks : max_chunks;
    max_items = n > max_items ? n : max_items;
  }
}

}  // namespace

// Segment length: the one that minimises a model of a forward + backward's time. The
// forward's kernels run two CTAs per SM, the backward's one; a CTA's time is its chunk
// count (the backward's chunks cost ~4x the forward's) plus a little per item (state
// loads, read-outs), and every item adds its states to the scans' traffic.
int choose_segment(int BH, int n_chunks) {
  const long long sms = sm_count();
  double best = 1e300;
  int best_s = 1;
  for (int s = 1; s <= n_chunks && s <= 64; ++s) {
    long long fc, fi, bc, bi;
    deal(BH, n_chunks, s, 2 * sms, fc, fi);
    deal(BH, n_chunks, s, sms, bc, bi);
    const long long items = (long long)BH * ((n_chunks + s - 1) / s);
    const double cost = 3.9 * fc + 15.0 * bc + 0.2 * fi + 0.5 * bi + 0.02 * items;
    if (cost <= best) {  // ties go to the longer segment
      best = cost;
      best_s = s;
    }
  }
  return best_s;
}

Geometry make_geometry(int BH, int N) {
  Geometry g;
  g.BH = BH;
  g.N = N;
  g.n_chunks = (N + kC - 1) / kC;
  // the choice is a pure function of (BH, n_chunks) and the SM count; it is
  // remembered so that a call (and its workspace query) pays for the search once
  static std::mutex mu;
  static std::map<std::pair<int, int>, int> memo;
  int s = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = memo.find({BH, g.n_chunks});
    if (it != memo.end()) s = it->second;
  }
  if (s == 0) {
    s = choose_segment(BH, g.n_chunks);
    std::lock_guard<std::mutex> lock(mu);
    if (memo.size() > 4096) memo.clear();
    memo[{BH, g.n_chunks}] = s;
  }
  g.seg_chunks = s;
  g.n_seg = (g.n_chunks + g.seg_chunks - 1) / g.seg_chunks;
  return g;
}

cudaError_t launch_segment_states(const CUtensorMap* tk, const CUtensorMap* tv, const Geometry& g,
                                  float* partial, WorkspaceHeader* hdr, cudaStream_t st,
                                  bool identity) {
  auto run = [&](auto kern) {
    cudaError_t e = configure(kern, kStateSmem);
    if (e != cudaSuccess) return e;
    const int ctas = min(g.n_items(), resident_ctas(kern, kStateSmem, kStateThreads) * sm_count());
    e = launch_pdl(kern, dim3(ctas), dim3(kStateThreads), kStateSmem, st, *tk, *tv, g, partial, hdr);
    count_launches(1);
    return e != cudaSuccess ? e : cudaGetLastError();
  };
  if (g.lens != nullptr || g.cu != nullptr)  // per-stream lengths (never identity features)
    return identity ? cudaErrorInvalidValue : run(tc_state_kernel<false, true>);
  return identity ? run(tc_state_kernel<true, false>) : run(tc_state_kernel<false, false>);
}

cudaError_t launch_scan(const float* partial, float* out, const Geometry& g, int mode,
                        const StateIO& io, WorkspaceHeader* hdr, cudaStream_t st) {
  // many short sequences: a block per sequence (a few dependent loads cover a whole state)
  const cudaError_t e =
      g.BH >= 2 * sm_count()
          ? launch_pdl(state_scan_seq_kernel, dim3(g.BH), dim3(kScanSeqThreads), 0, st, partial,
                       out, g, mode, io, hdr)
          : launch_pdl(state_scan_kernel, dim3((kStateFloats + kScanThreads - 1) / kScanThreads, g.BH),
                       dim3(kScanThreads), 0, st, partial, out, g, mode, io, hdr);
  count_launches(1);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// Whether clusters of `n` CTAs of the fused kernel `kern` can be resident (the query
// remembered per kernel and n); configures the kernel's shared memory on every call.
template <typename K>
bool fused_fits(K kern, int n) {
  if (configure(kern, kAttSmem) != cudaSuccess) return false;
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, bool> memo;
  const std::pair<const void*, int> key{reinterpret_cast<const void*>(kern), n};
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = memo.find(key);
    if (it != memo.end()) return it->second;
  }
  bool fits = false;
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(n);
    cfg.blockDim = dim3(kAttThreads);
    cfg.dynamicSmemBytes = kAttSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = n;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) == cudaSuccess)
      fits = clusters > 0;
    else
      cudaGetLastError();  // a refused query leaves no error behind
  }
  std::lock_guard<std::mutex> lock(mu);
  memo[key] = fits;
  return fits;
}

}  // namespace tcx

using namespace tcx;

bool tc_forward_supported(int D, int M, int dtype) { return dtype == LA_BF16 && D == 64 && M == 64; }

size_t tc_forward_workspace(int BH, int N) {
  const Geometry g = make_geometry(BH, N);
  return kHeaderBytes + 2 * align_up(sizeof(float) * kStateFloats * (size_t)g.n_items(), 256);
}

const float* tc_forward_prefix(const void* fwd_ws, int BH, int N, bool causal) {
  const Geometry g = make_geometry(BH, N);
  if (causal && g.n_chunks == 1) return nullptr;  // the direct path: no segment states
  const float* partial = reinterpret_cast<const float*>(static_cast<const char*>(fwd_ws) + kHeaderBytes);
  return partial + align_up(sizeof(float) * kStateFloats * (size_t)g.n_items(), 256) / 4;
}

cudaError_t tc_state_sums(const void* k, const void* v, const StateIO& io, int BH, int N, void* ws,
                          cudaStream_t st) {
  const Geometry g = make_geometry(BH, N);
  WorkspaceHeader* hdr = static_cast<WorkspaceHeader*>(ws);
  float* partial = reinterpret_cast<float*>(static_cast<char*>(ws) + kHeaderBytes);
  float* total = partial + align_up(sizeof(float) * kStateFloats * (size_t)g.n_items(), 256) / 4;
  CUtensorMap tk, tv;
  const uint64_t n = (uint64_t)N, bh = (uint64_t)BH;
  if (!make_tmap_bf16_3d(&tk, k, kDim, n, bh, kDim, kC, 1) ||
      !make_tmap_bf16_3d(&tv, v, kDim, n, bh, kDim, kC, 1))
    return cudaErrorInvalidValue;
  cudaError_t e = launch_segment_states(&tk, &tv, g, partial, hdr, st);
  if (e != cudaSuccess) return e;
  return launch_scan(partial, total, g, kScanTotal, io, hdr, st);
}

cudaError_t tc_forward(const void* q, const void* k, const void* v, void* out, const StateIO& io,
                       int BH, int N, bool causal, void* ws, cudaStream_t st,
                       const FaultHook* fault, bool identity) {
  Geometry g = make_geometry(BH, N);
  g.lens = io.lens;
  g.H = io.H;
  g.cu = io.cu;
  g.T = io.T;
  g.out_rows = static_cast<__nv_bfloat16*>(out);
  if (fault != nullptr) {  // read by the attend kernel only
    g.fault_load = fault->load;
    g.fault_wait_ns = fault->wait_ns;
  }
  WorkspaceHeader* hdr = static_cast<WorkspaceHeader*>(ws);
  float* partial = reinterpret_cast<float*>(static_cast<char*>(ws) + kHeaderBytes);
  float* prefix = partial + align_up(sizeof(float) * kStateFloats * (size_t)g.n_items(), 256) / 4;
  CUtensorMap tq, tk, tv, to;
  // [BH][N][D] as (d, token, sequence); the packed [T][H][D] as (d, head, row),
  // a chunk being 128 rows of one head (the same 128-byte rows in shared memory)
  const bool packed = io.cu != nullptr;
  const uint64_t d1 = packed ? (uint64_t)io.H : (uint64_t)N;
  const uint64_t d2 = packed ? (uint64_t)io.T : (uint64_t)BH;
  const uint32_t b1 = packed ? 1 : kC, b2 = packed ? kC : 1;
  if (!make_tmap_bf16_3d(&tq, q, kDim, d1, d2, kDim, b1, b2) ||
      !make_tmap_bf16_3d(&tk, k, kDim, d1, d2, kDim, b1, b2) ||
      !make_tmap_bf16_3d(&tv, v, kDim, d1, d2, kDim, b1, b2) ||
      !make_tmap_bf16_3d(&to, out, kDim, d1, d2, kDim, b1, b2))
    return cudaErrorInvalidValue;

  // causal with one chunk per sequence, continuing a stored state: no segment
  // states or scan; the attend kernel takes the state from io (or zero) and
  // writes the final state there. A fresh prefill takes the segment path, whose
  // state increment is the psi form (see tc_state_kernel): the attend kernel's
  // own increment rounds phi(K) to bf16, which a sum from a zero state over
  // random-sign v leaves at ~2% on the state's significant elements.
  const bool direct = causal && g.n_chunks == 1 && !(io.S != nullptr && !io.read_init);
  // a plain forward of sequences of at most 8 segments: one launch, a cluster per sequence,
  // when all of its CTAs are resident at once (with more, each CTA would pay its setup for
  // one item, where the persistent kernels pay it once: B256 H8 N1024 took 0.44 ms so
  // against 0.36 ms)
  if (!direct && !identity && io.S == nullptr && io.lens == nullptr && io.cu == nullptr &&
      (fault == nullptr || fault->fused) && g.n_seg <= kMaxFusedSegments) {
    auto fused = [&](auto kern) -> cudaError_t {
      if (!fused_fits(kern, g.n_seg) ||
          g.n_items() > resident_ctas(kern, kAttSmem, kAttThreads) * sm_count())
        return cudaErrorNotSupported;
      const cudaError_t err = launch_cluster_pdl(kern, dim3(g.n_items()), dim3(kAttThreads), kAttSmem,
                                                 st, g.n_seg, tq, tk, tv, to, g, prefix, StateIO{},
                                                 false, hdr);
      count_launches(1);
      return err != cudaSuccess ? err : cudaGetLastError();
    };
    const cudaError_t fe = causal ? fused(tc_attend_kernel<true, false, false, true>)
                                  : fused(tc_attend_kernel<false, false, false, true>);
    if (fe != cudaErrorNotSupported) return fe;
  }
  cudaError_t e = cudaSuccess;
  if (!direct) {
    // causal with no state to write back: the last segment's sums would only feed the
    // sequence's final state, so the segment-state pass stops one segment short
    Geometry gs = g;
    if (causal && io.S == nullptr) gs.n_seg = g.n_seg - 1;
    if (gs.n_items() > 0) {
      e = launch_segment_states(&tk, &tv, gs, partial, hdr, st, identity);
      if (e != cudaSuccess) return e;
    }
    e = launch_scan(partial, prefix, g, causal ? kScanPrefix : kScanTotal, io, hdr, st);
    if (e != cudaSuccess) return e;
  }
  const int sms = sm_count();

  // non-causal: one item per chunk range of the readout, all reading prefix[bh]
  auto attend = [&](auto kern, const StateIO& kio, bool kdirect) {
    cudaError_t err = configure(kern, kAttSmem);
    if (err != cudaSuccess) return err;
    const int ctas = min(g.n_items(), resident_ctas(kern, kAttSmem, kAttThreads) * sms);
    err = launch_pdl(kern, dim3(ctas), dim3(kAttThreads), kAttSmem, st, tq, tk, tv, to, g,
                     prefix, kio, kdirect, hdr);
    count_launches(1);
    return err != cudaSuccess ? err : cudaGetLastError();
  };
  if (io.lens != nullptr || io.cu != nullptr)  // per-stream lengths: causal, elu + 1 only
    return causal && !identity ? attend(tc_attend_kernel<true, false, true, false>, io, direct)
                               : cudaErrorInvalidValue;
  if (causal)
    return identity ? attend(tc_attend_kernel<true, true, false, false>, io, direct)
                    : attend(tc_attend_kernel<true, false, false, false>, io, direct);
  return identity ? attend(tc_attend_kernel<false, true, false, false>, StateIO{}, false)
                  : attend(tc_attend_kernel<false, false, false, false>, StateIO{}, false);
}

}  // namespace la
