// Shared pieces of the tensor-core kernels (forward and backward): chunk
// geometry, the per-CTA work cursor, phi on swizzled tiles and bounded waits.
#pragma once

#include <cuda_bf16.h>

#include "la_common.cuh"
#include "la_internal.h"
#include "la_tc.cuh"

namespace la {
namespace tcx {

using namespace tc;

constexpr int kC = 128;            // tokens per chunk
constexpr int kDim = 64;           // D = M
constexpr int kTile = kC * kDim * 2;  // 16 KB bf16 tile
constexpr int kThreadsTC = 128;
constexpr int kStateFloats = kDim * kDim + kDim;  // S^T [m][d] then Z [d]

// ------------------------------------------------------------------ helpers

struct Geometry {
  int BH, N, n_chunks, seg_chunks, n_seg;
  // forward only: stream b = bh / H uses its first lens[b] tokens (nullptr: all N)
  const int* lens = nullptr;
  int H = 1;
  // Failure test hook (la_debug_*_fault): CTA 0 withholds its TMA load number
  // fault_load (no copy is issued, so the wait for it can only run out) and
  // bounds its main-loop waits by fault_wait_ns. -1: off (every launch but the
  // test hook's).
  int fault_load = -1;
  unsigned long long fault_wait_ns = 0;
  __device__ bool faulty() const { return fault_load >= 0 && blockIdx.x == 0; }
  __device__ uint64_t wait_ns() const { return faulty() ? fault_wait_ns : kWaitLimitNs; }
  // forward only, packed token-major layout [T][H][D] (cu != nullptr): stream
  // b = bh / H holds rows cu[b] .. cu[b + 1] - 1 of every head (its first N at
  // most); bounds outside 0 <= cu[b] <= cu[b + 1] <= T give the stream no tokens
  const int* cu = nullptr;
  int T = 0;
  __nv_bfloat16* out_rows = nullptr;  // the packed output (rows stored one by one)
  __device__ void span(int bh, int& r0, int& n) const {
    const int b = bh / H, s = cu[b], e = cu[b + 1];
    const bool ok = 0 <= s && s <= e && e <= T;
    r0 = ok ? s : T;
    n = ok ? min(e - s, N) : 0;
  }
  // the stream's bounds are consistent and its length is at most N
  __device__ bool span_ok(int bh) const {
    const int b = bh / H, s = cu[b], e = cu[b + 1];
    return 0 <= s && s <= e && e <= T && e - s <= N;
  }
  __device__ int len(int bh) const {
    if (cu != nullptr) {
      int r0, n;
      span(bh, r0, n);
      return n;
    }
    return lens ? max(0, min(lens[bh / H], N)) : N;
  }

  __host__ __device__ int n_items() const { return BH * n_seg; }
  // item -> (bh, seg): segment-major so that a segment's predecessors were
  // scheduled earlier
  __host__ __device__ int bh_of(int item) const { return item % BH; }
  __host__ __device__ int seg_of(int item) const { return item / BH; }
  __host__ __device__ int chunk_begin(int item) const { return seg_of(item) * seg_chunks; }
  __host__ __device__ int chunk_end(int item) const {
    return min(chunk_begin(item) + seg_chunks, n_chunks);
  }
};

// Walks (item, chunk) pairs of this CTA in processing order: the CTA's items
// blockIdx.x, blockIdx.x + gridDim.x, ... first to last, or (back) last to
// first, each item's chunks in order. A kernel that re-reads what a kernel
// before it streamed walks its items back, so that it starts on the tiles the
// other read last (the ones still in L2). The item's (batch, head) index and
// chunk range are worked out once per item (they take integer divisions by
// runtime sizes), not per chunk.
// With per-stream lengths (LENS: lens or the packed layout, forward only) an item's
// range stops at the last chunk that holds tokens of its stream, and items with
// none are skipped: a stream shorter than N costs only its own chunks. The items
// are then dealt by tickets rather than round robin, since their sizes differ:
// one thread per CTA (the producer) takes the next ticket from a counter in the
// workspace header when it reaches the end of an item and passes the item on
// through a ring in shared memory, which the CTA's other cursors (consumers) read
// in the same order; -1 there ends the walk.
constexpr int kRing = 8;

template <bool LENS>
struct CursorT {
  int item, chunk;
  int bh, cbeg, cend;  // of `item`
  int n;               // LENS: its stream's token count
  int r0, head;        // LENS, packed layout: the stream's first row, the item's head
  int step;            // +-gridDim.x
  int* counter = nullptr;        // dealt by tickets: the producer's ticket counter
  volatile int* ring = nullptr;  // dealt by tickets: the ring (producer and consumers)
  int rpos = 0;
  int ahead = -1;  // producer: the ticket requested while the previous item ran
  bool back = false;
  __device__ void set_item(const Geometry& g) {
    bh = g.bh_of(item);
    cbeg = g.chunk_begin(item);
    cend = g.chunk_end(item);
    if (LENS && g.cu != nullptr) {
      g.span(bh, r0, n);
      head = bh % g.H;
      cend = min(cend, (n + kC - 1) / kC);
    } else if (LENS && g.lens != nullptr) {
      n = g.len(bh);
      cend = min(cend, (n + kC - 1) / kC);
    }
  }
  // TMA coordinates (y, z) of the current chunk: (first token, sequence) in the
  // [BH][N][D] layout, (head, row) in the packed one; a chunk wholly past the
  // stream's end points past row T (the copy reads only fill values)
  __device__ void tile_yz(const Geometry& g, int& y, int& z) const {
    const int t0 = chunk * kC;
    if (LENS && g.cu != nullptr) {
      y = head;
      z = t0 < n ? r0 + t0 : g.T;
    } else {
      y = t0;
      z = bh;
    }
  }
  // the first item from `item` on (in steps of `step`) with a chunk to process
  __device__ void seek(const Geometry& g) {
    chunk = 0;
    for (; valid(g); item += step) {
      set_item(g);
      if (cbeg < cend) {
        chunk = cbeg;
        return;
      }
    }
  }
  // dealt by tickets: the next item with a chunk to process (producer: from the
  // counter, recorded in the ring; consumer: the ring's next entry)
  __device__ void take(const Geometry& g) {
    chunk = 0;
    if (counter != nullptr) {
      for (;;) {
        // each ticket is requested one item ahead, so that the atomic's round trip
        // overlaps the item's work instead of stalling the thread that takes it
        const int t = ahead >= 0 ? ahead : atomicAdd(counter, 1);
        ahead = atomicAdd(counter, 1);
        item = t < g.n_items() ? (back ? g.n_items() - 1 - t : t) : -1;
        if (item < 0) break;
        set_item(g);
        if (cbeg < cend) break;
      }
      ring[rpos++ % kRing] = item;
    } else {
      item = ring[rpos++ % kRing];
    }
    if (item >= 0) {
      set_item(g);
      chunk = cbeg;
    }
  }
  __device__ void start(const Geometry& g, bool back_ = false) {
    if (LENS && ring != nullptr) {
      back = back_;
      take(g);
      return;
    }
    item = blockIdx.x;
    step = back_ ? -(int)gridDim.x : (int)gridDim.x;
    if (back_ && item < g.n_items()) item += (g.n_items() - 1 - item) / (int)gridDim.x * (int)gridDim.x;
    if constexpr (LENS) {
      seek(g);
    } else {
      chunk = 0;
      if (valid(g)) {
        set_item(g);
        chunk = cbeg;
      }
    }
  }
  __device__ bool valid(const Geometry& g) const { return (unsigned)item < (unsigned)g.n_items(); }
  __device__ bool first() const { return chunk == cbeg; }
  __device__ bool last() const { return chunk + 1 == cend; }
  __device__ void advance(const Geometry& g) {
    if (++chunk >= cend) {
      if (LENS && ring != nullptr) {
        take(g);
        return;
      }
      item += step;
      if constexpr (LENS) {
        seek(g);
      } else if (valid(g)) {
        set_item(g);
        chunk = cbeg;
      }
    }
  }
};

using Cursor = CursorT<true>;       // the forward's kernels
using FullCursor = CursorT<false>;  // every sequence N tokens long (the backward's)

// Same items as FullCursor, but each item's chunks from last to first.
struct RevCursor {
  int item, chunk;
  int bh, cbeg, cend;  // of `item`
  __device__ void set_item(const Geometry& g) {
    bh = g.bh_of(item);
    cbeg = g.chunk_begin(item);
    cend = g.chunk_end(item);
  }
  __device__ void start(const Geometry& g) {
    item = blockIdx.x;
    chunk = 0;
    if (item < g.n_items()) {
      set_item(g);
      chunk = cend - 1;
    }
  }
  __device__ bool valid(const Geometry& g) const { return item < g.n_items(); }
  __device__ void advance(const Geometry& g) {
    if (--chunk < cbeg) {
      item += gridDim.x;
      if (item < g.n_items()) {
        set_item(g);
        chunk = cend - 1;
      }
    }
  }
};

// Two float32 lanes at once (one packed instruction, each lane rounded as alone).
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(d)
      : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)),
        "l"(*reinterpret_cast<uint64_t*>(&c)));
  return *reinterpret_cast<float2*>(&d);
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;"
      : "=l"(d)
      : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)));
  return *reinterpret_cast<float2*>(&d);
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;"
      : "=l"(d)
      : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)));
  return *reinterpret_cast<float2*>(&d);
}
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;"
      : "=l"(d)
      : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)));
  return *reinterpret_cast<float2*>(&d);
}

__device__ __forceinline__ float bf16_lo_f(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi_f(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

__device__ __forceinline__ void record_timeout(WorkspaceHeader* hdr, int site) {
  atomicExch(&hdr->status, (int)LA_ERR_TIMEOUT);
  atomicExch(&hdr->wait_site, site);
}

// phi(x) = exp(min(x, 0)) + max(x, 0): the elu + 1 map without a branch, with
// the hardware exp2 (its few-ulp float32 error vanishes in the bf16 rounding
// of the result).
__device__ __forceinline__ float phi_fast(float x) {
  return __expf(fminf(x, 0.f)) + fmaxf(x, 0.f);
}

// phi on two packed bf16 values, exp(min(x, 0)) + max(x, 0), in bf16x2
// arithmetic throughout: t = min(x, 0) log2(e) as one fused multiply-add with
// log2(e) split into two bf16 parts (t = m L_hi + bf16(m L_lo), rounded once),
// the packed base-2 exponential of t, and the final add. Besides the rounding
// of the result, the exponential carries the rounding of t: a relative error
// of at most 2^-9 |t| ln 2 (below one bf16 ulp for |x| < 2).
__device__ __forceinline__ uint32_t phi2_bf16(uint32_t u) {
  const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162*>(&u);
  const __nv_bfloat162 zero = __float2bfloat162_rn(0.f);
  const __nv_bfloat162 l_hi = __float2bfloat162_rn(1.4453125f);           // bf16(log2 e)
  const __nv_bfloat162 l_lo = __float2bfloat162_rn(-0.0026174591110366f);  // log2 e - l_hi
  const __nv_bfloat162 m = __hmin2(x, zero);
  const __nv_bfloat162 t = __hfma2(m, l_hi, __hmul2(m, l_lo));
  const uint32_t tu = *reinterpret_cast<const uint32_t*>(&t);
  uint32_t eu;
  asm("ex2.approx.ftz.bf16x2 %0, %1;" : "=r"(eu) : "r"(tu));
  const __nv_bfloat162 e = *reinterpret_cast<const __nv_bfloat162*>(&eu);
  const __nv_bfloat162 r = __hadd2(e, __hmax2(x, zero));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// phi on two packed bf16 values with a float32 exponential (each result is
// phi of the exact input, rounded once): the backward's variant, where dq and
// dk cancel the constant part of phi and keep only what k and q add to it.
__device__ __forceinline__ uint32_t phi2_bf16_exact(uint32_t u) {
  __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162*>(&u);
  const __nv_bfloat162 zero = __float2bfloat162_rn(0.f);
  const float2 f = __bfloat1622float2(__hmin2(x, zero));
  const __nv_bfloat162 e = __floats2bfloat162_rn(__expf(f.x), __expf(f.y));
  __nv_bfloat162 r = __hadd2(e, __hmax2(x, zero));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// Half-row variants for kernels where two warpgroups share each row: half h
// owns the logical 16-byte chunks [4h, 4h + 4), i.e. columns [32h, 32h + 32).
template <bool EXACT, bool MASK>
__device__ __forceinline__ void phi_half_impl(uint8_t* tile, int row, int h, int nvalid) {
  const bool valid = !MASK || row < nvalid;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint4* p = reinterpret_cast<uint4*>(tile + sw128(row, (4 * h + c) * 16));
    const uint4 w = *p;
    uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) u[q] = valid ? (EXACT ? phi2_bf16_exact(u[q]) : phi2_bf16(u[q])) : 0u;
    *p = make_uint4(u[0], u[1], u[2], u[3]);
  }
}

// (the row mask is applied only in a tile with padding rows; nvalid is the
// same for the whole CTA, so the branch is uniform)
template <bool EXACT = false>
__device__ __forceinline__ void phi_half(uint8_t* tile, int row, int h, int nvalid) {
  if (nvalid >= kC)
    phi_half_impl<EXACT, false>(tile, row, h, nvalid);
  else
    phi_half_impl<EXACT, true>(tile, row, h, nvalid);
}

// psi(x) = phi(x) - 1 (x for x > 0, exp(x) - 1 otherwise) on two packed bf16
// values, each rounded once. phi(k) = 1 + psi(k) with |psi| << 1 for the small
// inputs of attention, so a sum over phi(k) splits into an exact count (or an
// exact column sum) and a sum over psi(k) whose bf16 rounding is ~10x smaller
// than that of phi(k) itself.
__device__ __forceinline__ uint32_t psi2_bf16(uint32_t u) {
  const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162*>(&u);
  const __nv_bfloat162 zero = __float2bfloat162_rn(0.f);
  const float2 m = __bfloat1622float2(__hmin2(x, zero));
  const float2 p = __bfloat1622float2(__hmax2(x, zero));
  const float2 e = add2(sub2(make_float2(__expf(m.x), __expf(m.y)), make_float2(1.f, 1.f)), p);
  const __nv_bfloat162 r = __floats2bfloat162_rn(e.x, e.y);
  return *reinterpret_cast<const uint32_t*>(&r);
}

// psi on this thread's half of tile row `row`, in place; rows >= nvalid become 0.
__device__ __forceinline__ void psi_half(uint8_t* tile, int row, int h, int nvalid) {
  const bool valid = row < nvalid;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint4* p = reinterpret_cast<uint4*>(tile + sw128(row, (4 * h + c) * 16));
    const uint4 w = *p;
    *p = valid ? make_uint4(psi2_bf16(w.x), psi2_bf16(w.y), psi2_bf16(w.z), psi2_bf16(w.w))
               : make_uint4(0, 0, 0, 0);
  }
}

// Zeroes this thread's half of tile row `row` (columns [32h, 32h + 32)) when the
// row is past the valid rows: rows beyond a sequence's length may hold any bits
// (even NaN), and a zero weight times NaN is still NaN.
__device__ __forceinline__ void zero_half_if_past(uint8_t* tile, int row, int h, int nvalid) {
  if (row < nvalid) return;
#pragma unroll
  for (int c = 0; c < 4; ++c)
    *reinterpret_cast<uint4*>(tile + sw128(row, (4 * h + c) * 16)) = make_uint4(0, 0, 0, 0);
}

template <bool MASK>
__device__ __forceinline__ void phi_half_split_impl(uint8_t* tile, uint8_t* lo, int row, int h,
                                                    int nvalid, float (&z)[32]) {
  const bool valid = !MASK || row < nvalid;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint32_t off = sw128(row, (4 * h + c) * 16);
    uint4* p = reinterpret_cast<uint4*>(tile + off);
    const uint4 w = *p;
    uint32_t u[4] = {w.x, w.y, w.z, w.w}, l[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float a = valid ? phi_fast(bf16_lo_f(u[q])) : 0.f;
      const float b = valid ? phi_fast(bf16_hi_f(u[q])) : 0.f;
      u[q] = pack_bf16(a, b);
      l[q] = pack_bf16(a - bf16_lo_f(u[q]), b - bf16_hi_f(u[q]));
      z[8 * c + 2 * q] = a;
      z[8 * c + 2 * q + 1] = b;
    }
    *p = make_uint4(u[0], u[1], u[2], u[3]);
    *reinterpret_cast<uint4*>(lo + off) = make_uint4(l[0], l[1], l[2], l[3]);
  }
}

__device__ __forceinline__ void phi_half_split(uint8_t* tile, uint8_t* lo, int row, int h,
                                               int nvalid, float (&z)[32]) {
  if (nvalid >= kC)
    phi_half_split_impl<false>(tile, lo, row, h, nvalid, z);
  else
    phi_half_split_impl<true>(tile, lo, row, h, nvalid, z);
}

// Bounded wait that also gives up once another thread of the CTA has given up
// (a shared abort flag), so that one timeout winds the whole CTA down; for
// kernels whose warps wait on different barriers at different times.
__device__ __forceinline__ bool mbar_wait_abort(uint64_t* bar, uint32_t parity, volatile int* abort,
                                                WorkspaceHeader* hdr, int site) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      *abort = 1;
      record_timeout(hdr, site);
      return false;
    }
  }
}

// The same, agreed by the whole warp (warp-collective TMEM accesses follow).
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, volatile int* abort,
                                               WorkspaceHeader* hdr, int site) {
  return __all_sync(0xffffffffu, mbar_wait_abort(bar, parity, abort, hdr, site));
}

// A worker warp's wait for a stage's tiles when items are dealt by tickets: 1 when
// the tiles of chunk n have landed, 2 when the CTA's work ended before chunk n (the
// producer, having run out of items, stored the number of chunks it loaded in
// `total`, -1 until then; no load for chunk n is then coming), 0 when the wait ran
// out or the CTA is winding down. Agreed by the warp (the lowest outcome wins).
__device__ __forceinline__ int mbar_wait_warp_or_end(uint64_t* bar, uint32_t parity,
                                                     volatile int* abort, WorkspaceHeader* hdr,
                                                     int site, volatile int* total, long long n) {
  int r = 0;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) {
      r = 1;
      break;
    }
    const int tot = *total;
    if (tot >= 0 && n >= tot) {
      r = 2;
      break;
    }
    if (*abort) break;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      *abort = 1;
      record_timeout(hdr, site);
      break;
    }
  }
  return __reduce_min_sync(0xffffffffu, r);
}

// Block-uniform bounded wait: every thread waits, then all agree on the outcome
// (a timeout seen by any thread ends the loop for the whole CTA together).
__device__ __forceinline__ bool wait_uniform(uint64_t* bar, uint32_t parity, WorkspaceHeader* hdr,
                                             int site, uint64_t limit_ns = kWaitLimitNs) {
  const bool all = __syncthreads_and(mbar_wait(bar, parity, limit_ns) ? 1 : 0) != 0;
  if (!all && threadIdx.x == 0) record_timeout(hdr, site);
  return all;
}

// End of a kernel whose thread 0 issued tcgen05 MMAs: one commit after all of
// them, waited for with the full limit, so that TMEM is never freed (nor shared
// memory released) under an MMA still in flight, whatever made the loop end.
__device__ __forceinline__ void drain_mmas(uint64_t* drain, WorkspaceHeader* hdr, int site) {
  if (threadIdx.x == 0) {
    mma_commit(drain);
    if (!mbar_wait(drain, 0)) record_timeout(hdr, site);
  }
}

__device__ __forceinline__ uint32_t lane_base(uint32_t tbase) {
  return tbase + ((uint32_t)((threadIdx.x / 32) % 4 * 32) << 16);
}


// Opt in to the dynamic shared memory `kernel` needs and to the largest
// shared-memory carveout (so several CTAs fit per SM).
template <typename K>
inline cudaError_t configure(K kernel, int smem) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                              (int)cudaSharedmemCarveoutMaxShared);
}

// CTAs of `kernel` that fit on one SM (at least 1): the larger of the runtime's
// occupancy answer and a count from the kernel's registers and shared memory
// against the SM's register file and shared memory (1 KB reserved per CTA).
template <typename K>
inline int resident_ctas(K kernel, int smem, int threads = kThreadsTC) {
  int api = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&api, kernel, threads, smem) != cudaSuccess)
    api = 0;
  int dev = 0, smem_sm = 0, regs_sm = 0;
  cudaFuncAttributes fa;
  int manual = 1;
  if (cudaGetDevice(&dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) ==
          cudaSuccess &&
      cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev) ==
          cudaSuccess &&
      cudaFuncGetAttributes(&fa, kernel) == cudaSuccess) {
    const int regs_warp = ((fa.numRegs + 7) / 8 * 8) * 32;
    const int regs_cta = regs_warp * (threads / 32);
    const int by_smem = smem_sm / (smem + (int)fa.sharedSizeBytes + 1024);
    const int by_regs = regs_cta > 0 ? regs_sm / regs_cta : 1;
    manual = by_smem < by_regs ? by_smem : by_regs;
  }
  const int n = api > manual ? api : manual;
  return n > 0 ? n : 1;
}

int sm_count();
Geometry make_geometry(int BH, int N);

// Launch with programmatic stream serialization: the kernel may start while
// the previous kernel in the stream drains; every kernel launched this way
// calls pdl_wait() before its first global-memory access.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// launch_pdl for a grid of thread-block clusters of `cluster_x` CTAs along x
template <typename... KArgs, typename... Args>
inline cudaError_t launch_cluster_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                      cudaStream_t st, int cluster_x, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster_x;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

enum ScanMode { kScanPrefix = 0, kScanTotal = 1, kScanSuffix = 2 };

// Segment increments dS^T = V^T phi(K), dZ = sum phi(K) into partial[item].
// identity: the K tiles hold the features f already (summed as they are), else the
// elu + 1 map (summed in the psi form).
cudaError_t launch_segment_states(const CUtensorMap* tk, const CUtensorMap* tv, const Geometry& g,
                                  float* partial, WorkspaceHeader* hdr, cudaStream_t st,
                                  bool identity = false);
// Prefix / total / suffix of the per-segment states (see ScanMode).
// With io.S set, the prefix / total also starts from io's initial state (when
// io.read_init) and the full sum is written to io's entries (prefill, extend).
cudaError_t launch_scan(const float* partial, float* out, const Geometry& g, int mode,
                        const StateIO& io, WorkspaceHeader* hdr, cudaStream_t st);

}  // namespace tcx
}  // namespace la
