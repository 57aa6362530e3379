// Schedule: index inversion and work list, entirely on the device.
//
// "Sparse Attention" (dinara-dl), Chapter 5, "Reverse index": the selector gives
// each query its blocks; the KV-centric kernel needs, for each block, the queries
// that chose it, plus the block's place in each query's list, and popular blocks
// are split into several tasks.  "Kernel optimization for MiniMax M3", load-
// balancing section: one on-device pass flattens all (kv_head, kv_block, query)
// work into a sequence and hands each CTA a contiguous slice; shapes are fixed so
// nothing is read back to the host.
//
// Determinism without atomics deciding order: every (row, query) entry sets one
// bit of a [row][query / 32] bitmask (atomicOr is order-independent).  A query's
// rank inside its row is then the popcount of the bits below it, so the scatter
// that follows is a pure function of the input and rows come out sorted by query.
//
// Kernels, in stream order:
//   mark              bits for every valid entry; bad ids -> a bit in the header's pad[1].
//                     k_mark_cols: a CTA per (32-query bitmask column, KV head) ORs its
//                     queries' bits per block in shared memory and stores each nonzero word
//                     once; k_mark (entries<mark>, one thread per list slot, global atomics)
//                     where the blocks are many and the columns few
//   rowscan           per row: exclusive popcount prefix over words, row count, tiles
//                     per (window, row) segment; each bitmask word is copied to mcopy
//                     (what the scatter reads) and cleared, and pad[1] becomes the
//                     header's status, so the next build of the same schedule starts
//                     from a zero bitmask and header without a memset (the first build,
//                     and every build into the no-allocation scratch, zero them with two
//                     memsets, which also break the launches' programmatic dependencies)
//   scan_small        one CTA: offsets, E, nsb, the Q-outer / KV-outer decision and the
//                     exclusive scan of the segment tile counts (at most 32768 segments);
//                     more segments: scan_rows + seg_reduce / seg_top / seg_down
//   entries<scatter>  qlist, slot, cmap, blist  } one launch (scatter_tiles): the two only
//   tiles             the work list, window-major, 8-entry tiles  } read what the scans wrote
// Tiny inputs (decode sizes) take one CTA instead: schedule_one runs the same phases
// with CTA barriers in between and writes the same arrays, in one launch instead of two
// memsets and four kernels.
#include "msa_internal.h"
#include "ptx.cuh"

namespace msa {
namespace {

template <int NT>
__device__ int block_exclusive_scan(int v, int* total, int* warp_buf) {
  static_assert(NT % 32 == 0 && NT <= 1024, "block size");
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_buf[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int w = lane < NT / 32 ? warp_buf[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < NT / 32) warp_buf[lane] = w;
  }
  __syncthreads();
  const int prefix = wid ? warp_buf[wid - 1] : 0;
  *total = warp_buf[NT / 32 - 1];
  __syncthreads();
  return prefix + x - v;
}

// One thread per list slot; each CTA stages whole lists in shared memory.  Slot k of
// list (query i, group g) with own block lb is an entry iff its id b satisfies
// 0 <= b <= lb and b does not occur in an earlier slot of the same list.  Ids >= nblocks
// or < -1 are errors: ignored, and (mark pass) the sticky status bit is set.
//   kScatter = false (mark): set bit (row g * nblocks + b, query i) of the bitmask.
//   kScatter = true: the entry's CSR position p = offsets[row] + (entries of the row
//   with a smaller query) -> qlist[p] = i, slot[p] = k; every slot gets cmap (p or -1)
//   and blist (b or -1).
constexpr int kEntThreads = 256;

// Body of entries<>: CTA bid of nbid (the scatter shares its launch with the tiles).
template <bool kScatter>
__device__ __forceinline__ void entries_body(const int32_t* __restrict__ idx, int N, int Hkv, int topK, int nblocks,
                                             int Lkv, int C, int lists_per_cta, uint32_t* __restrict__ mask,
                                             const int32_t* __restrict__ rowbase, const int32_t* __restrict__ offsets,
                                             int32_t* __restrict__ qlist, int32_t* __restrict__ slot,
                                             int32_t* __restrict__ cmap, int32_t* __restrict__ blist, SchedHeader* hdr,
                                             int bid, int nbid) {
  __shared__ int32_t s_idx[kEntThreads];
  const int64_t nl = static_cast<int64_t>(N) * Hkv;
  const int t = threadIdx.x;
  bool bad = false;
  for (int64_t L0 = static_cast<int64_t>(bid) * lists_per_cta; L0 < nl;
       L0 += static_cast<int64_t>(nbid) * lists_per_cta) {
    const int64_t e0 = L0 * topK;
    const int nle = static_cast<int>(min(static_cast<int64_t>(lists_per_cta), nl - L0)) * topK;
    const int b = t < nle ? idx[e0 + t] : -1;
    s_idx[t] = b;
    __syncthreads();
    if (t < nle) {
      const int lk = t / topK, k = t - lk * topK;
      const int64_t L = L0 + lk;
      const int i = static_cast<int>(L / Hkv), g = static_cast<int>(L % Hkv);
      const int lb = (Lkv - N + i) / kBlock;
      bool entry = true;
      if (b < -1 || b >= nblocks) {
        bad = true;
        entry = false;
      } else if (b < 0 || b > lb) {
        entry = false;
      } else {
        for (int k2 = 0; k2 < k; ++k2)
          if (s_idx[lk * topK + k2] == b) {
            entry = false;
            break;
          }
      }
      const size_t r = static_cast<size_t>(g) * nblocks + (entry ? b : 0);
      if constexpr (!kScatter) {
        if (entry) atomicOr(&mask[r * C + (i >> 5)], 1u << (i & 31));
      } else {
        int p = -1;
        if (entry) {
          const uint32_t word = mask[r * C + (i >> 5)];
          p = offsets[r] + rowbase[r * (C + 1) + (i >> 5)] + __popc(word & ((1u << (i & 31)) - 1u));
          if (dbg_ok(p >= 0 && static_cast<int64_t>(p) < static_cast<int64_t>(N) * Hkv * topK, &hdr->status)) {
            qlist[p] = i;
            slot[p] = k;
          } else {
            p = -1;
          }
        }
        cmap[e0 + t] = p;
        blist[e0 + t] = entry ? b : -1;
      }
    }
    __syncthreads();
  }
  if (!kScatter && bad) atomicOr(&hdr->pad[1], kStatusBadIndex);  // the row scan moves it into status
}

__global__ void __launch_bounds__(kEntThreads)
k_mark(const int32_t* __restrict__ idx, int N, int Hkv, int topK, int nblocks, int Lkv, int C, int lists_per_cta,
       uint32_t* __restrict__ mask, SchedHeader* hdr) {
  griddep_wait();
  griddep_launch();
  entries_body<false>(idx, N, Hkv, topK, nblocks, Lkv, C, lists_per_cta, mask, nullptr, nullptr, nullptr, nullptr,
                      nullptr, nullptr, hdr, blockIdx.x, gridDim.x);
}

// The mark pass's bad-index bit becomes the status of this build (status and pad[1] are
// read and written by one thread of the row scan only).
__device__ __forceinline__ void take_mark_status(SchedHeader* hdr) {
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    hdr->status = hdr->pad[1];
    hdr->pad[1] = 0;
  }
}

// Mark by bitmask columns: CTA (w, g) takes the lists of queries 32 w .. 32 w + 31 in KV
// head g, ORs each entry's query bit into a shared-memory word per block, and stores each
// nonzero word once, with no global atomics (this CTA is the only writer of word w of the
// head's rows; the bitmask is zero beforehand: cleared by the previous build's row scan, or
// by a memset).  The entry rule is entries<>'s.  Shared memory: nblocks words, then the
// 32 * topK list slots.
constexpr int kMarkThreads = 256;
constexpr size_t kMarkColsMaxSmem = 96 * 1024;
__global__ void __launch_bounds__(kMarkThreads)
k_mark_cols(const int32_t* __restrict__ idx, int N, int Hkv, int topK, int nblocks, int Lkv, int C,
            uint32_t* __restrict__ mask, SchedHeader* hdr) {
  griddep_wait();
  griddep_launch();
  extern __shared__ uint32_t s_bits[];
  int32_t* s_idx = reinterpret_cast<int32_t*>(s_bits + nblocks);
  const int w = blockIdx.x / Hkv, g = blockIdx.x - (blockIdx.x / Hkv) * Hkv;
  const int t = threadIdx.x, nsl = 32 * topK;
  for (int b = t; b < nblocks; b += kMarkThreads) s_bits[b] = 0u;
  for (int e = t; e < nsl; e += kMarkThreads) {
    const int qi = e / topK, k = e - qi * topK, i = 32 * w + qi;
    s_idx[e] = i < N ? idx[(static_cast<int64_t>(i) * Hkv + g) * topK + k] : -1;
  }
  __syncthreads();
  bool bad = false;
  for (int e = t; e < nsl; e += kMarkThreads) {
    const int qi = e / topK, k = e - qi * topK, i = 32 * w + qi;
    if (i >= N) continue;
    const int b = s_idx[e];
    if (b < -1 || b >= nblocks) {
      bad = true;
      continue;
    }
    if (b < 0 || b > (Lkv - N + i) / kBlock) continue;
    bool first = true;
    for (int k2 = 0; k2 < k; ++k2)
      if (s_idx[qi * topK + k2] == b) {
        first = false;
        break;
      }
    if (first) atomicOr(&s_bits[b], 1u << qi);
  }
  if (bad) atomicOr(&hdr->pad[1], kStatusBadIndex);  // the row scan moves it into status
  __syncthreads();
  for (int b = t; b < nblocks; b += kMarkThreads) {
    const uint32_t v = s_bits[b];
    if (v) mask[(static_cast<size_t>(g) * nblocks + b) * C + w] = v;
  }
}

template <int NT>
__global__ void __launch_bounds__(NT) k_rowscan(uint32_t* __restrict__ mask, int R, int C, int nW,
                                                int32_t* __restrict__ rowbase, int32_t* __restrict__ counts,
                                                int32_t* __restrict__ segtiles, uint32_t* __restrict__ mcopy,
                                                SchedHeader* hdr) {
  griddep_wait();
  griddep_launch();
  take_mark_status(hdr);
  __shared__ int warp_buf[32];
  constexpr int kCpw = kWindow / kChunk;
  constexpr int kWarps = NT / 32;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  // warp wid scans the words [s0, s1) of the row, lane l taking words s0 + 32 j + l (coalesced)
  const int seg = ((C + kWarps - 1) / kWarps + 31) & ~31;
  const int s0 = min(wid * seg, C), s1 = min(s0 + seg, C);
  for (int r = blockIdx.x; r < R; r += gridDim.x) {
    uint32_t* m = mask + static_cast<size_t>(r) * C;
    uint32_t* mc = mcopy + static_cast<size_t>(r) * C;
    int32_t* rb = rowbase + static_cast<size_t>(r) * (C + 1);
    int sum = 0;
    for (int c = s0 + lane; c < s1; c += 32) sum += __popc(m[c]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane == 0) warp_buf[wid] = sum;
    __syncthreads();
    int run = 0, total = 0;  // this warp's prefix and the row total
#pragma unroll
    for (int q = 0; q < kWarps; ++q) {
      const int v = warp_buf[q];
      run += q < wid ? v : 0;
      total += v;
    }
    for (int c0 = s0; c0 < s1; c0 += 32) {  // warp-uniform trip count (the shuffles below)
      const int c = c0 + lane;
      const uint32_t w = c < s1 ? m[c] : 0u;
      const int v = __popc(w);
      int inc = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
      }
      if (c < s1) {
        rb[c] = run + inc - v;
        mc[c] = w;
        m[c] = 0u;
      }
      run += __shfl_sync(0xffffffffu, inc, 31);
    }
    if (threadIdx.x == 0) {
      rb[C] = total;
      counts[r] = total;
    }
    __syncthreads();
    for (int w = threadIdx.x; w < nW; w += NT) {
      const int cw0 = w * kCpw, cw1 = min(cw0 + kCpw, C);
      const int cnt = rb[cw1] - rb[cw0];
      segtiles[static_cast<size_t>(w) * R + r] = (cnt + kTileQ - 1) / kTileQ;
    }
    __syncthreads();
  }
}

// k_rowscan for rows of at most 32 bitmask words (N <= 1024 queries: decode and
// low-reuse sizes, where rows are many and short): one warp per row instead of a CTA.
__global__ void __launch_bounds__(256) k_rowscan_warp(uint32_t* __restrict__ mask, int R, int C, int nW,
                                                      int32_t* __restrict__ rowbase, int32_t* __restrict__ counts,
                                                      int32_t* __restrict__ segtiles, uint32_t* __restrict__ mcopy,
                                                      SchedHeader* hdr) {
  griddep_wait();
  griddep_launch();
  take_mark_status(hdr);
  constexpr int kCpw = kWindow / kChunk;
  const int lane = threadIdx.x & 31;
  for (int64_t r = blockIdx.x * 8ll + (threadIdx.x >> 5); r < R; r += gridDim.x * 8ll) {
    const uint32_t w = lane < C ? mask[r * C + lane] : 0u;
    const int v = __popc(w);
    if (lane < C) {
      mcopy[r * C + lane] = w;
      mask[r * C + lane] = 0u;
    }
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    const int total = __shfl_sync(0xffffffffu, inc, 31);
    int32_t* rb = rowbase + r * (C + 1);
    if (lane < C) rb[lane] = inc - v;
    if (lane == 0) {
      rb[C] = total;
      counts[r] = total;
    }
    for (int w0 = 0; w0 < nW; w0 += 32) {  // warp-uniform trip count: the shuffles below
      const int w = w0 + lane;
      const int cw0 = min(w * kCpw, C), cw1 = min(cw0 + kCpw, C);
      const int a = __shfl_sync(0xffffffffu, inc - v, cw0 & 31), b = __shfl_sync(0xffffffffu, inc - v, cw1 & 31);
      const int e0 = cw0 >= C ? total : a, e1 = cw1 >= C ? total : b;
      if (w < nW) segtiles[static_cast<size_t>(w) * R + r] = (e1 - e0 + kTileQ - 1) / kTileQ;
    }
  }
}

template <int NT>
__global__ void __launch_bounds__(NT) k_scan_rows(const int32_t* __restrict__ counts, int R, int N,
                                                  int32_t* __restrict__ offsets, SchedHeader* hdr) {
  griddep_wait();
  griddep_launch();
  __shared__ int warp_buf[32];
  const int per = (R + NT - 1) / NT;
  const int r0 = min(static_cast<int>(threadIdx.x) * per, R), r1 = min(r0 + per, R);
  int sum = 0, nz = 0;
  for (int r = r0; r < r1; ++r) {
    sum += counts[r];
    nz += counts[r] > 0;
  }
  int total, nsb;
  int run = block_exclusive_scan<NT>(sum, &total, warp_buf);
  block_exclusive_scan<NT>(nz, &nsb, warp_buf);
  for (int r = r0; r < r1; ++r) {
    offsets[r] = run;
    run += counts[r];
  }
  if (threadIdx.x == 0) {
    offsets[R] = total;
    hdr->entries = total;
    hdr->nsb = nsb;
    hdr->path = dispatch_path(total, nsb);  // (msa_internal.h)
  }
}

// Exclusive scan of in[0, n) into out (in place allowed) by one CTA of NT threads, in chunks
// of NT * 8 elements staged in shared memory: coalesced loads and stores, a serial scan of 8
// consecutive elements per thread (indices padded by one word per 32 against bank conflicts)
// and one block scan per chunk.  Returns the total; *nz (if given) counts the nonzero inputs;
// window_tiles (if given) receives out[q] for every q that is a multiple of R.
constexpr int kScanItems = 8;
template <int NT>
__device__ int block_scan_array(const int32_t* in, int32_t* out, int n, int* sm, int* warp_buf, int* nz,
                                int32_t* window_tiles, int R) {
  constexpr int kCh = NT * kScanItems;
  auto pad = [](int i) { return i + (i >> 5); };
  const int t = threadIdx.x;
  int carry = 0, nzc = 0;
  for (int base = 0; base < n; base += kCh) {
#pragma unroll
    for (int k = 0; k < kScanItems; ++k) {
      const int i = base + k * NT + t;
      sm[pad(k * NT + t)] = i < n ? in[i] : 0;
    }
    __syncthreads();
    int v[kScanItems], sum = 0;
#pragma unroll
    for (int j = 0; j < kScanItems; ++j) {
      v[j] = sm[pad(t * kScanItems + j)];
      sum += v[j];
      nzc += v[j] > 0;
    }
    int total;
    int run = carry + block_exclusive_scan<NT>(sum, &total, warp_buf);  // (its barriers order sm)
#pragma unroll
    for (int j = 0; j < kScanItems; ++j) {
      sm[pad(t * kScanItems + j)] = run;
      run += v[j];
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kScanItems; ++k) {
      const int i = base + k * NT + t;
      if (i < n) {
        const int e = sm[pad(k * NT + t)];
        out[i] = e;
        if (window_tiles && i % R == 0) window_tiles[i / R] = e;
      }
    }
    carry += total;
    __syncthreads();
  }
  if (nz) {
    int nzt;
    block_exclusive_scan<NT>(nzc, &nzt, warp_buf);
    *nz = nzt;
  }
  return carry;
}

constexpr int kRegItems = 16;  // values per thread of the one-pass scan of both small arrays

// Rows (as k_scan_rows) and, in the same CTA, the exclusive scan of the per-(window,
// row) segment tile counts when there are few segments (at most NT * kSmallSegPer).
constexpr int kSmallSegPer = 32;

template <int NT>
__device__ void scan_small_body(const int32_t* __restrict__ counts, int R, int N, int32_t* __restrict__ offsets,
                                int32_t* __restrict__ seg, int nseg, int32_t* __restrict__ window_tiles, int nW,
                                SchedHeader* hdr, int* warp_buf, int* sm) {
  // The one-pass scan pays where the chunked one needs more than two passes (measured on
  // GB300: 16,384 rows and segments, 0.1877 -> 0.1852 ms per low-reuse step; at 256 rows and
  // 1,024 segments, one chunk each, it was 1.5 us slower than the chunked scan)
  constexpr int kCh = NT * kScanItems;
  if (R <= NT * kRegItems && nseg <= NT * kRegItems && (R + kCh - 1) / kCh + (nseg + kCh - 1) / kCh > 2) {
    // both arrays held in registers, their loads issued together: warp w owns the
    // 32 * kRegItems consecutive values from w * 32 * kRegItems, lane l the ones at
    // offsets 32 j + l (coalesced), scanned per j across the lanes with a running carry;
    // one cross-warp scan of the warp totals (row entries, segment tiles, nonempty rows)
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int base = w * 32 * kRegItems;
    int c[kRegItems], g[kRegItems];
#pragma unroll
    for (int j = 0; j < kRegItems; ++j) {
      const int i = base + 32 * j + lane;
      c[j] = i < R ? counts[i] : 0;
      g[j] = i < nseg ? seg[i] : 0;
    }
    int cx = 0, cy = 0, cz = 0;  // warp carries
    const bool has = base < R || base < nseg;  // warp-uniform: warps past both arrays skip the scan
#pragma unroll
    for (int j = 0; j < kRegItems && has; ++j) {
      int x = c[j], y = g[j];
      cz += __popc(__ballot_sync(0xffffffffu, c[j] > 0));
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int a = __shfl_up_sync(0xffffffffu, x, o), b = __shfl_up_sync(0xffffffffu, y, o);
        if (lane >= o) {
          x += a;
          y += b;
        }
      }
      c[j] = cx + x - c[j];  // exclusive, within the warp
      g[j] = cy + y - g[j];
      cx += __shfl_sync(0xffffffffu, x, 31);
      cy += __shfl_sync(0xffffffffu, y, 31);
    }
    if (lane == 0) {
      warp_buf[w] = cx;
      warp_buf[32 + w] = cy;
      warp_buf[64 + w] = cz;
    }
    __syncthreads();
    if (w < 3) {  // warp k: exclusive scan of the k-th total over the warps
      const int v = lane < NT / 32 ? warp_buf[32 * w + lane] : 0;
      int x = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int a = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += a;
      }
      if (lane < NT / 32) warp_buf[32 * w + lane] = x - v;
      if (lane == 31) warp_buf[96 + w] = x;  // the CTA total
    }
    __syncthreads();
    const int ox = warp_buf[w], oy = warp_buf[32 + w];
#pragma unroll
    for (int j = 0; j < kRegItems; ++j) {
      const int i = base + 32 * j + lane;
      if (i < R) offsets[i] = ox + c[j];
      if (i < nseg) {
        const int e = oy + g[j];
        seg[i] = e;
        if (i % R == 0) window_tiles[i / R] = e;
      }
    }
    if (threadIdx.x == 0) {
      const int E = warp_buf[96], tiles = warp_buf[97], nsb = warp_buf[98];
      offsets[R] = E;
      hdr->entries = E;
      hdr->nsb = nsb;
      hdr->path = dispatch_path(E, nsb);  // (msa_internal.h)
      seg[nseg] = tiles;
      window_tiles[nW] = tiles;
      hdr->ntiles = tiles;
    }
    return;
  }
  int nsb = 0;
  const int total = block_scan_array<NT>(counts, offsets, R, sm, warp_buf, &nsb, nullptr, R);
  if (threadIdx.x == 0) {
    offsets[R] = total;
    hdr->entries = total;
    hdr->nsb = nsb;
    hdr->path = dispatch_path(total, nsb);  // (msa_internal.h)
  }
  const int tiles = block_scan_array<NT>(seg, seg, nseg, sm, warp_buf, nullptr, window_tiles, R);
  if (threadIdx.x == 0) {
    seg[nseg] = tiles;
    window_tiles[nW] = tiles;
    hdr->ntiles = tiles;
  }
}

template <int NT>
__global__ void __launch_bounds__(NT) k_scan_small(const int32_t* __restrict__ counts, int R, int N,
                                                   int32_t* __restrict__ offsets, int32_t* __restrict__ seg,
                                                   int nseg, int32_t* __restrict__ window_tiles, int nW,
                                                   SchedHeader* hdr) {
  griddep_wait();
  griddep_launch();
  __shared__ int warp_buf[4 * 32];
  __shared__ int sm[NT * kScanItems + NT * kScanItems / 32];
  scan_small_body<NT>(counts, R, N, offsets, seg, nseg, window_tiles, nW, hdr, warp_buf, sm);
}

template <int NT>
__global__ void __launch_bounds__(NT) k_seg_reduce(const int32_t* __restrict__ seg, int64_t nseg,
                                                   int32_t* __restrict__ sums) {
  griddep_wait();
  griddep_launch();
  __shared__ int warp_buf[32];
  constexpr int per = kSegScanBlock / NT;
  const int64_t s0 = static_cast<int64_t>(blockIdx.x) * kSegScanBlock + threadIdx.x * per;
  int sum = 0;
  for (int j = 0; j < per; ++j)
    if (s0 + j < nseg) sum += seg[s0 + j];
  int total;
  block_exclusive_scan<NT>(sum, &total, warp_buf);
  if (threadIdx.x == 0) sums[blockIdx.x] = total;
}

template <int NT>
__global__ void __launch_bounds__(NT) k_seg_top(int32_t* __restrict__ sums, int nb, int32_t* __restrict__ segoff,
                                                int64_t nseg, int32_t* __restrict__ window_tiles, int nW,
                                                SchedHeader* hdr) {
  griddep_wait();
  griddep_launch();
  __shared__ int warp_buf[32];
  const int per = (nb + NT - 1) / NT;
  const int b0 = min(static_cast<int>(threadIdx.x) * per, nb), b1 = min(b0 + per, nb);
  int sum = 0;
  for (int b = b0; b < b1; ++b) sum += sums[b];
  int total;
  int run = block_exclusive_scan<NT>(sum, &total, warp_buf);
  for (int b = b0; b < b1; ++b) {
    const int v = sums[b];
    sums[b] = run;
    run += v;
  }
  if (threadIdx.x == 0) {
    sums[nb] = total;
    segoff[nseg] = total;
    window_tiles[nW] = total;
    hdr->ntiles = total;
  }
}

template <int NT>
__global__ void __launch_bounds__(NT) k_seg_down(int32_t* __restrict__ seg, int64_t nseg,
                                                 const int32_t* __restrict__ sums, int R,
                                                 int32_t* __restrict__ window_tiles) {
  griddep_wait();
  griddep_launch();
  __shared__ int warp_buf[32];
  constexpr int per = kSegScanBlock / NT;
  const int64_t s0 = static_cast<int64_t>(blockIdx.x) * kSegScanBlock + threadIdx.x * per;
  int v[per];
  int sum = 0;
#pragma unroll
  for (int j = 0; j < per; ++j) {
    v[j] = (s0 + j < nseg) ? seg[s0 + j] : 0;
    sum += v[j];
  }
  int total;
  int run = block_exclusive_scan<NT>(sum, &total, warp_buf) + sums[blockIdx.x];
#pragma unroll
  for (int j = 0; j < per; ++j) {
    const int64_t s = s0 + j;
    if (s < nseg) {
      seg[s] = run;
      if (s % R == 0) window_tiles[s / R] = run;
    }
    run += v[j];
  }
}

// Work-list tiles of the segments, CTA bid of nbid (256 threads): one warp per (window, row)
// segment, its lanes writing the segment's tiles (a segment holds up to kWindow / kTileQ tiles)
__device__ __forceinline__ void tiles_body(const int32_t* __restrict__ segoff, int64_t nseg, int R, int C,
                                           const int32_t* __restrict__ rowbase, const int32_t* __restrict__ offsets,
                                           int4* __restrict__ tiles, int64_t cap_tiles, int32_t* status,
                                           int bid, int nbid) {
  constexpr int kCpw = kWindow / kChunk;
  constexpr int kWarps = kEntThreads / 32;
  const int lane = threadIdx.x & 31;
  for (int64_t s = bid * static_cast<int64_t>(kWarps) + (threadIdx.x >> 5); s < nseg;
       s += static_cast<int64_t>(nbid) * kWarps) {
    const int t0 = segoff[s], n = segoff[s + 1] - t0;
    if (n == 0) continue;
    const int w = static_cast<int>(s / R), r = static_cast<int>(s % R);
    const int cw0 = w * kCpw, cw1 = min(cw0 + kCpw, C);
    const int32_t* rb = rowbase + static_cast<size_t>(r) * (C + 1);
    const int first = offsets[r] + rb[cw0];
    const int cnt = rb[cw1] - rb[cw0];
    for (int j = lane; j < n; j += 32)
      if (dbg_ok(t0 + j >= 0 && t0 + j < cap_tiles, status))
        tiles[t0 + j] = make_int4(r, first + kTileQ * j, min(kTileQ, cnt - kTileQ * j), w);
  }
}

// scatter (entries<true>) on CTAs [0, ent_grid), the work-list tiles on the rest: both
// only read what the scans wrote, so one launch serves both
__global__ void __launch_bounds__(kEntThreads)
k_scatter_tiles(const int32_t* __restrict__ idx, int N, int Hkv, int topK, int nblocks, int Lkv, int C,
                int lists_per_cta, int ent_grid, const uint32_t* __restrict__ mask,
                const int32_t* __restrict__ rowbase, const int32_t* __restrict__ offsets,
                int32_t* __restrict__ qlist, int32_t* __restrict__ slot, int32_t* __restrict__ cmap,
                int32_t* __restrict__ blist, const int32_t* __restrict__ segoff, int64_t nseg, int R,
                int4* __restrict__ tiles, int64_t cap_tiles, SchedHeader* hdr) {
  griddep_wait();
  griddep_launch();
  const int b = blockIdx.x;
  if (b < ent_grid)
    entries_body<true>(idx, N, Hkv, topK, nblocks, Lkv, C, lists_per_cta, const_cast<uint32_t*>(mask), rowbase,
                       offsets, qlist, slot, cmap, blist, hdr, b, ent_grid);
  else
    tiles_body(segoff, nseg, R, C, rowbase, offsets, tiles, cap_tiles, &hdr->status, b - ent_grid,
               static_cast<int>(gridDim.x) - ent_grid);
}

// The whole schedule in one CTA (small inputs).  Phases, separated by CTA barriers:
// zero the bitmask and the header; mark (entries<mark>); per row the popcount prefix,
// the count and the segment tile counts (rowscan); the scans (scan_small); scatter
// (entries<scatter>); tiles.  An entry is what entries<> calls one (valid id, not in
// the future, first occurrence in its list), so every array equals the multi-kernel
// schedule's.  The bitmask, built with atomics, is read back through L2.
constexpr int kOneThreads = 1024;

__device__ __forceinline__ bool slot_entry(const int32_t* __restrict__ lst, int k, int b, int lb, int nblocks,
                                           bool& bad) {
  if (b < -1 || b >= nblocks) {
    bad = true;
    return false;
  }
  if (b < 0 || b > lb) return false;
  for (int k2 = 0; k2 < k; ++k2)
    if (lst[k2] == b) return false;
  return true;
}

__global__ void __launch_bounds__(kOneThreads, 1)
k_schedule_one(const int32_t* __restrict__ idx, int N, int Hkv, int topK, int nblocks, int Lkv, int R, int C, int nW,
               SchedDev d, int64_t cap_tiles) {
  griddep_wait();
  griddep_launch();
  __shared__ int warp_buf[4 * 32];
  __shared__ int s_bad;
  __shared__ int sm[kOneThreads * kScanItems + kOneThreads * kScanItems / 32];
  constexpr int kCpw = kWindow / kChunk;
  const int t = threadIdx.x;
  const int64_t nmask = static_cast<int64_t>(R) * C;
  for (int64_t q = t; q < nmask; q += kOneThreads) d.mask[q] = 0u;
  if (t < static_cast<int>(sizeof(SchedHeader) / sizeof(int32_t))) reinterpret_cast<int32_t*>(d.hdr)[t] = 0;
  if (t == 0) s_bad = 0;
  __syncthreads();
  const int64_t nslot = static_cast<int64_t>(N) * Hkv * topK;
  bool bad = false;
  for (int64_t e = t; e < nslot; e += kOneThreads) {
    const int64_t L = e / topK;
    const int k = static_cast<int>(e - L * topK);
    const int i = static_cast<int>(L / Hkv), g = static_cast<int>(L % Hkv);
    const int b = idx[e];
    const int lb = (Lkv - N + i) / kBlock;
    if (slot_entry(idx + L * topK, k, b, lb, nblocks, bad))
      atomicOr(&d.mask[(static_cast<size_t>(g) * nblocks + b) * C + (i >> 5)], 1u << (i & 31));
  }
  if (bad) s_bad = 1;
  __syncthreads();
  for (int r = t; r < R; r += kOneThreads) {
    const uint32_t* m = d.mask + static_cast<size_t>(r) * C;
    int32_t* rb = d.rowbase + static_cast<size_t>(r) * (C + 1);
    int run = 0;
    for (int c = 0; c < C; ++c) {
      rb[c] = run;
      run += __popc(__ldcg(m + c));
    }
    rb[C] = run;
    d.counts[r] = run;
    for (int w = 0; w < nW; ++w) {
      const int cw0 = w * kCpw, cw1 = min(cw0 + kCpw, C);
      const int cnt = rb[cw1] - rb[cw0];
      d.segoff[static_cast<size_t>(w) * R + r] = (cnt + kTileQ - 1) / kTileQ;
    }
  }
  __syncthreads();
  const int nseg = nW * R;
  scan_small_body<kOneThreads>(d.counts, R, N, d.offsets, d.segoff, nseg, d.window_tiles, nW, d.hdr, warp_buf, sm);
  __syncthreads();
  for (int64_t e = t; e < nslot; e += kOneThreads) {
    const int64_t L = e / topK;
    const int k = static_cast<int>(e - L * topK);
    const int i = static_cast<int>(L / Hkv), g = static_cast<int>(L % Hkv);
    const int b = idx[e];
    const int lb = (Lkv - N + i) / kBlock;
    bool unused = false;
    int p = -1;
    const bool entry = slot_entry(idx + L * topK, k, b, lb, nblocks, unused);
    if (entry) {
      const size_t r = static_cast<size_t>(g) * nblocks + b;
      const uint32_t word = __ldcg(d.mask + r * C + (i >> 5));
      p = d.offsets[r] + d.rowbase[r * (C + 1) + (i >> 5)] + __popc(word & ((1u << (i & 31)) - 1u));
      if (dbg_ok(p >= 0 && p < nslot, &d.hdr->status)) {
        d.qlist[p] = i;
        d.slot[p] = k;
      } else {
        p = -1;
      }
    }
    d.cmap[e] = p;
    d.blist[e] = entry ? b : -1;
  }
  for (int q = t; q < nseg; q += kOneThreads) {
    const int t0 = d.segoff[q], n = d.segoff[q + 1] - t0;
    if (n == 0) continue;
    const int w = q / R, r = q % R;
    const int cw0 = w * kCpw, cw1 = min(cw0 + kCpw, C);
    const int32_t* rb = d.rowbase + static_cast<size_t>(r) * (C + 1);
    const int first = d.offsets[r] + rb[cw0];
    const int cnt = rb[cw1] - rb[cw0];
    for (int j = 0; j < n; ++j)
      if (dbg_ok(t0 + j >= 0 && t0 + j < cap_tiles, &d.hdr->status))
        d.tiles[t0 + j] = make_int4(r, first + kTileQ * j, min(kTileQ, cnt - kTileQ * j), w);
  }
  if (t == 0 && s_bad) atomicOr(&d.hdr->status, kStatusBadIndex);
}

// One CTA is latency-bound (its loops run serially per thread): it wins only while the
// lists and the rows are few.  Measured on GB300, graph-replayed decode steps: N = 1 and
// 16 (64 and 1024 slots, 4096 rows) 49.6 -> 43.0 and 56 -> 52 us; at 4096 slots it was
// 21 us slower than the multi-kernel path, at 16384 slots 130 us slower.
constexpr int64_t kOneMaxSlots = 1024, kOneMaxMaskWords = 8192, kOneMaxSegments = 8192;

int grid_for(int64_t n, int threads, int cap) {
  int64_t g = (n + threads - 1) / threads;
  if (g < 1) g = 1;
  if (g > cap) g = cap;
  return static_cast<int>(g);
}

}  // namespace

cudaError_t enqueue_schedule(msa_schedule* s, const int32_t* indices, cudaStream_t st) {
  const SchedDev& d = s->d;
  const int Lkv = s->nblocks * kBlock;
  const int64_t nl = static_cast<int64_t>(s->N) * s->Hkv;
  const int lists_per_cta = kEntThreads / s->topK;  // topK <= 64
  const int ent_grid = grid_for(nl, lists_per_cta, 1 << 20);
  cudaError_t e;
  // tiny inputs: one CTA (limits keep its serial per-thread loops short); it zeroes the
  // bitmask itself and leaves it set
  if (nl * s->topK <= kOneMaxSlots && static_cast<int64_t>(s->R) * s->C <= kOneMaxMaskWords && s->C <= 64 &&
      s->nseg <= kOneMaxSegments) {
    s->mask_clean = false;
    MSA_LAUNCH(k_schedule_one, 1, kOneThreads, 0, st, indices, s->N, s->Hkv, s->topK, s->nblocks, Lkv, s->R, s->C, s->nW, d,
               s->cap_tiles);
    return cudaGetLastError();
  }
  // the bitmask and the header start at zero: left so by the previous build's row scan, or
  // zeroed here (first build, or after a build whose launches did not all go through)
  const bool clean = s->mask_clean;
  s->mask_clean = false;
  if (!clean) {
    if ((e = cudaMemsetAsync(d.mask, 0, sizeof(uint32_t) * static_cast<size_t>(s->R) * s->C, st))) return e;
    if ((e = cudaMemsetAsync(d.hdr, 0, sizeof(SchedHeader), st))) return e;
  }
  // the column mark clears and scans nblocks shared words per CTA: where that is more than four
  // times the CTA's 32 * topK list slots (few, wide columns: 256 queries over 4096 blocks took
  // 1.8 us longer per step than with the atomic mark), the atomic mark stays.  Measured per
  // step on GB300 against the atomic mark: M3 -1.3 us, the long workload -11 us, fp8 -37 us.
  const size_t mark_smem = sizeof(uint32_t) * (static_cast<size_t>(s->nblocks) + 32 * static_cast<size_t>(s->topK));
  if (mark_smem <= kMarkColsMaxSmem && s->nblocks <= 4 * 32 * s->topK) {
    static std::atomic<uint64_t> mark_attr{0};
    if ((e = set_smem_limit(k_mark_cols, static_cast<int>(kMarkColsMaxSmem), mark_attr))) return e;
    MSA_LAUNCH(k_mark_cols, s->C * s->Hkv, kMarkThreads, mark_smem, st, indices, s->N, s->Hkv, s->topK, s->nblocks, Lkv,
               s->C, d.mask, d.hdr);
  } else {
    MSA_LAUNCH(k_mark, ent_grid, kEntThreads, 0, st, indices, s->N, s->Hkv, s->topK, s->nblocks, Lkv, s->C,
               lists_per_cta, d.mask, d.hdr);
  }
  if (s->C <= 32)
    MSA_LAUNCH(k_rowscan_warp, grid_for(s->R, 8, 1 << 20), 256, 0, st, d.mask, s->R, s->C, s->nW, d.rowbase, d.counts,
               d.segoff, d.mcopy, d.hdr);
  else
    MSA_LAUNCH(k_rowscan<256>, grid_for(s->R, 1, 1 << 20), 256, 0, st, d.mask, s->R, s->C, s->nW, d.rowbase, d.counts,
               d.segoff, d.mcopy, d.hdr);
  if (s->nseg <= 1024 * kSmallSegPer) {
    MSA_LAUNCH(k_scan_small<1024>, 1, 1024, 0, st, d.counts, s->R, s->N, d.offsets, d.segoff, static_cast<int>(s->nseg),
                                           d.window_tiles, s->nW, d.hdr);
  } else {
    MSA_LAUNCH(k_scan_rows<1024>, 1, 1024, 0, st, d.counts, s->R, s->N, d.offsets, d.hdr);
    const int nb = static_cast<int>(s->nseg_blocks);
    MSA_LAUNCH(k_seg_reduce<256>, nb, 256, 0, st, d.segoff, s->nseg, d.seg_sums);
    MSA_LAUNCH(k_seg_top<1024>, 1, 1024, 0, st, d.seg_sums, nb, d.segoff, s->nseg, d.window_tiles, s->nW, d.hdr);
    MSA_LAUNCH(k_seg_down<256>, nb, 256, 0, st, d.segoff, s->nseg, d.seg_sums, s->R, d.window_tiles);
  }
  const int tiles_grid = grid_for(s->nseg, kEntThreads / 32, 1 << 16);  // a warp per segment
  MSA_LAUNCH(k_scatter_tiles, ent_grid + tiles_grid, kEntThreads, 0, st, 
      indices, s->N, s->Hkv, s->topK, s->nblocks, Lkv, s->C, lists_per_cta, ent_grid, d.mcopy, d.rowbase, d.offsets,
      d.qlist, d.slot, d.cmap, d.blist, d.segoff, s->nseg, s->R, d.tiles, s->cap_tiles, d.hdr);
  e = cudaGetLastError();
  // every launch went through: the row scan has cleared what the next build needs at zero
  s->mask_clean = e == cudaSuccess;
  return e;
}

}  // namespace msa
