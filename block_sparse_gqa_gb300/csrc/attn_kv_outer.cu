// KV-outer (KV-stationary) attention kernel, bf16 or fp8 E4M3, tcgen05 + TMA, persistent.
//
// "Kernel optimization for MiniMax M3 on NVIDIA Blackwell" (kernel stages): a CTA
// owns one KV block at a time and attends every query that chose it; because each
// tile sees a single block there is exactly one softmax step and no rescale of a
// running output; the softmax warps write the row statistics (m, l) directly and
// the output warps evacuate the raw P V accumulator, so the two never wait on each
// other; partial outputs are written tile-ordered and contiguous, and the combine
// kernel gathers them.  "Sparse Attention", Chapter 5: the KV-centric kernel writes,
// per query and head, a partial output and its softmax statistics.
//
// Work unit (tile): up to 8 consecutive CSR entries of one (group g, block b) row,
// i.e. 8 queries x 16 heads = 128 MMA rows (the head-packed "box" of one query is
// 16 rows).  The schedule lists tiles window by window (2048 queries per window).
// CTAs take chunks of 8 consecutive tiles from that list with one atomicAdd on a
// per-launch counter: all CTAs move through the windows together (Q and K/V of the
// current windows stay in L2) and a slow SM simply takes fewer chunks.  Each tile
// writes fixed output rows, so results do not depend on which CTA ran it.
//
// Warp roles (512 threads = 4 warpgroups, one CTA per SM; a warp reaches TMEM
// lanes 32 * (warp % 4) .. + 31, so a warpgroup covers all 128 rows):
//   warp 0       scheduler, all 32 lanes: claims chunks, reads the next chunk's
//                tile info and query ids ahead of time, gathers each tile's Q into Q
//                stage t % 4 (four stages) once S(t - 4) has read it -- one TMA box per
//                query, the 16 heads of its group (4 KB bf16, 2 KB E4M3), landing in the
//                128-byte-swizzled MMA layout through a 5-D (bf16) or 3-D (E4M3) view of
//                Q -- and publishes each tile in a shared-memory ring for the other roles
//   warp 2       K/V loader: on a row change loads K_b into the next of two K
//                buffers and V_b into the V buffer (TMA; E4M3: V as f16, into the next of
//                two V buffers); a ring slot is reused only after both this warp and
//                the output warps have released it
//   warp 1       TMEM allocation (512 columns = four regions R0..R3 of 128) and issue of
//                S = Q K^T (tcgen05, smem x smem) for tile t into region t % 4, once the
//                output warps have read O of tile t - 3 from it
//   warp 3       issue of O = P V into region (t + 3) % 4 -- where tile t - 1's P was --
//                with P read from TMEM (it overwrites S of region t % 4 in
//                place).  Two issuing threads: S of tile t + 1 never waits behind
//                the P V of tile t (its softmax, or an E4M3 V block being widened)
//   warps 4-7    softmax of even tiles
//   warps 8-11   softmax of odd tiles
//                (The Q gather used to be 16-byte cp.async copies issued by the softmax
//                warpgroups after each softmax: the load/store unit throttled their
//                issue to ~1.3 us per 32 KB tile, half of a warpgroup's time, while the
//                partial stores went through the TMA unit.  The roles are now swapped:
//                TMA carries the gather, the load/store unit the partial stores,
//                0.554 -> 0.498 ms at M3.)
//   warps 12-15  output: O -> registers -> bf16 -> 16-byte global stores, no staging:
//                the partial workspace is chunk-major inside each aligned group of 8
//                CSR positions (part_index), so the 32 rows a warp holds after one
//                TMEM load (32 consecutive columns each) are stored as 512 contiguous
//                bytes per 16-byte column chunk.  No shared memory or CTA barrier is
//                spent on the partials (a staged TMA store moved 64 KB of shared memory
//                per tile, a third of the kernel's shared-memory traffic)
// Registers are rebalanced per warpgroup with setmaxnreg: 72 for the control
// warpgroup (at 64 its scheduler / MMA code spills, which costs 6% of kernel time),
// 176 for the softmax warpgroups (a row's 128 scores stay in registers), 88 for the
// output warpgroup: 128*72 + 256*176 + 128*88 = 65536, the block's launch allocation
// (512 x 128), so every increase can be granted.
// TMEM rotation: a region serves tile t as S / P, then tile t + 1 as O, then tile t + 4 as S.
// S of tile t therefore waits only for the output warps to have read O of tile t - 3, and
// three tiles are between S and the reuse of its columns (with fixed S[2] / O[2] stages S
// of tile t waited for P V of tile t - 2: the chain S -> softmax -> P V of one tile set the
// pace of two).  P V of tile t writes over the P of tile t - 1, so it waits for that P V to
// complete (the ordering PTX guarantees between pipelined MMAs of one thread covers a shared
// accumulator, not a later MMA writing its accumulator over an earlier one's A operand, so the
// wait is explicit; it costs nothing measurable, P of tile t comes much later).  Each barrier of the S / P / O chain has four slots, one
// per region, so no waiter can fall a whole phase behind.  Measured at M3: 0.494 -> 0.479 ms
// with four Q stages (three: 0.489).
// A softmax thread owns one MMA row (TMEM lane): row maximum m (base-2 units,
// scale folded in), P = 2^(s*scale*log2e - m) written back over S as bf16 pairs,
// row sum l; (m, l) go to global as one float2 per row.
//
// Partial layout: raw bf16 (O_k = sum_j P_j V_j, not yet divided by l) of (CSR position
// p, head h) in the chunk-major groups of part_index, and float2 (m, l) at [16 p + h].
// A tile's entries are consecutive CSR positions, so its partials fill one aligned
// group of 8 positions (32 KB, contiguous) or parts of two.
//
// fp8 E4M3 inputs (per-tensor descales): S = Q K^T runs on kind::f8f6f4 (K-major, one
// 128-byte swizzle span per row, 32 elements per MMA); q and k descales are folded
// into the softmax scale.  P V runs in f16: the forward widens the whole E4M3 V tensor
// to f16 once per call (exact, widen_e4m3_kernel below), the loader loads its blocks by
// TMA as the bf16 path loads V, and P is packed as f16 (more mantissa than bf16 for
// values in [0, 1]).  The v descale is applied by the combine.  (Widening each selected
// block in shared memory with the loader warp instead cost 45% more kernel time on the
// 65536-query E4M3 workload: one warp's conversion, once per row change, was on the
// critical path.)
//
// Optional E4M3 P V (kP8, msa_fwd_opts_t.debug_flags bit 1): P rounded to E4M3 (scaled so
// that its largest value is 256) into a shared-memory tile per tile parity, V transposed per
// block to E4M3 V^T by transpose_e4m3_kernel, and P V as 4 kind::f8f6f4 MMAs with both
// operands K-major.  Measured on the 65536-query E4M3 workload: 3.84 against 3.85 ms, relative
// L2 error 9.3e-3 against 1.9e-3 with f16 P V, so f16 P V is the default.
#include <cfloat>

#include <cuda_bf16.h>

#include "msa_internal.h"
#include "ptx.cuh"

namespace msa {
namespace {

constexpr int kThreads = 512;
// setmaxnreg shares per warpgroup (control, each of the two softmax, output).  An
// increase is granted only from registers the block already holds, so the shares must
// add up to no more than the launch allocation (512 threads x 128 registers); a larger
// sum would leave setmaxnreg.inc waiting forever.
constexpr uint32_t kRegCtl = 72, kRegSoftmax = 176, kRegOut = 88;
static_assert(kThreads == 512 && 128 * (kRegCtl + 2 * kRegSoftmax + kRegOut) <= 512 * 128,
              "setmaxnreg shares exceed the launch allocation");
constexpr int kChunkTiles = 8;  // tiles per chunk of tile metadata the scheduler warp reads at once
// chunks per claim: a CTA takes kClaimChunks * 8 consecutive tiles of the work list at once,
// so it changes row (a 64 KB K + V load) about once per claim
constexpr int kClaimChunks = 2;
constexpr int kRing = 8;        // tile-info ring slots
constexpr int kQStages = 4;
// TMEM: four regions of 128 columns.  Tile t computes S (and P over it) in region t % 4
// and accumulates O in region (t + 3) % 4, the region tile t - 1's P occupied.
constexpr int kRegions = 4;
constexpr uint32_t kCtlBytes = 1024;
constexpr uint32_t kTileBytes = 128 * 128 * 2;  // a 16-bit 128 x 128 tile (two 16 KB halves)

// Shared-memory layout per input type (offsets from the 1024-aligned base).
// kP8 (E4M3 inputs only): P V on kind::f8f6f4 from an E4M3 V^T copy and an E4M3 P staged in
// shared memory, instead of f16 V and f16 P in tensor memory
template <bool kFp8, bool kP8 = false>
struct Lay {
  static constexpr uint32_t kInTile = kFp8 ? 16384 : 32768;  // Q or K tile in the input type
  static constexpr uint32_t kOffQ = 0;                       // + kInTile * stage
  static constexpr uint32_t kOffK0 = kQStages * kInTile;
  static constexpr uint32_t kOffK1 = kOffK0 + kInTile;
  // 16-bit V (bf16, or f16 widened from E4M3): one buffer for bf16 (shared memory is full),
  // two for E4M3 so that the next row's V loads while this row's P V runs
  static constexpr int kVBuf = kFp8 ? 2 : 1;
  static constexpr uint32_t kVTile = kP8 ? 16384 : kTileBytes;  // one V block (kP8: E4M3 V^T)
  static constexpr uint32_t kOffV = kOffK1 + kInTile;
  static constexpr uint32_t kOffP = kOffV + kVBuf * kVTile;  // kP8: two E4M3 P tiles (128 x 128 bytes)
  static constexpr uint32_t kOffCtl = kOffP + (kP8 ? 2 * 16384 : 0);
  static constexpr uint32_t kSmemBytes = kOffCtl + kCtlBytes + 1024;  // + alignment slack
};
static_assert(Lay<false>::kSmemBytes <= 232448 && Lay<true>::kSmemBytes <= 232448 &&
                  Lay<true, true>::kSmemBytes <= 232448, "shared memory");

// barrier slots (8 bytes each) at the start of the control area
enum {
  B_QFULL0 = 0, B_KFULL0 = B_QFULL0 + kQStages, B_KFREE0 = B_KFULL0 + 2, B_VFULL0 = B_KFREE0 + 2,
  B_VFREE0 = B_VFULL0 + 2, B_SFULL0 = B_VFREE0 + 2, B_PFULL0 = B_SFULL0 + kRegions, B_PVDONE0 = B_PFULL0 + kRegions,
  B_OFREE0 = B_PVDONE0 + kRegions, B_TFULL0 = B_OFREE0 + kRegions, B_TEMPTY0 = B_TFULL0 + kRing,
  B_QFREE0 = B_TEMPTY0 + kRing, B_COUNT = B_QFREE0 + kQStages
};
constexpr uint32_t kOffTmemSlot = 8 * B_COUNT;  // 4 bytes
constexpr uint32_t kOffRing = 512;              // kRing entries of 64 bytes
static_assert(kOffTmemSlot + 4 <= kOffRing && kOffRing + 64 * kRing <= kCtlBytes, "control area");

// One published tile: row (g * nblocks + b), first CSR position, count (0 = no more
// work), flags (bit 0: new row, bits 8-15: K/V buffer), then the query ids.
struct TileInfo {
  int row, first, count, flags;
  int q[kTileQ];
  int pad[4];
};
static_assert(sizeof(TileInfo) == 64, "ring entry");

struct KvParams {
  const uint8_t* Q;  // bf16 or E4M3 elements
  uint4* partial;
  int Hq;
  const int4* tiles;
  const int32_t* qlist;
  SchedHeader* hdr;
  float2* pstat;
  int N, Lkv, nblocks;
  int R;          // Hkv * nblocks schedule rows
  int64_t cap_e;  // CSR positions the schedule's arrays and the partial workspace hold
  float sl2;  // scale * log2(e) (* q descale * k descale for E4M3)
  int force_path;
};

__device__ __forceinline__ void flag_timeout(SchedHeader* hdr) { atomicOr(&hdr->status, kStatusTimeout); }

__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// (x0, x1) * s + c for a pair of floats held as one 64-bit register
__device__ __forceinline__ uint64_t ffma2(uint64_t x, uint64_t s, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(x), "l"(s), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
__device__ __forceinline__ void unpack2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// 16-bit P pair: f16 for the E4M3 path (its P V runs on f16 V), bf16 otherwise
template <bool kF16>
__device__ __forceinline__ uint32_t pack_p(float lo, float hi) {
  return kF16 ? pack_f16x2(lo, hi) : pack_bf16x2(lo, hi);
}

template <uint32_t N>
__device__ __forceinline__ void regs_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N)); }
template <uint32_t N>
__device__ __forceinline__ void regs_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N)); }

// One row of a tile: scores v[0..127] (raw S), keys c > lim masked when kMasked.
// Writes P = 2^(v * sl2 - m2) as bf16 pairs over columns [0, 64) of the row's S
// columns in TMEM and returns (m2, l).  A positive scale is assumed here; a
// negative one goes through softmax_row_any_scale.
template <bool kMasked, bool kF16>
__device__ __forceinline__ float2 softmax_row(uint32_t (&v)[128], int lim, float sl2, uint32_t tS) {
  float a0 = -FLT_MAX, a1 = -FLT_MAX, a2 = -FLT_MAX, a3 = -FLT_MAX;
#pragma unroll
  for (int e = 0; e < 128; e += 8) {
    float x[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) x[q] = (kMasked && e + q > lim) ? -FLT_MAX : __uint_as_float(v[e + q]);
    a0 = max3(a0, x[0], x[1]);
    a1 = max3(a1, x[2], x[3]);
    a2 = max3(a2, x[4], x[5]);
    a3 = max3(a3, x[6], x[7]);
  }
  const float m2 = fmaxf(fmaxf(a0, a1), fmaxf(a2, a3)) * sl2;
  const uint64_t sl2x2 = pack2(sl2, sl2), negm2 = pack2(-m2, -m2);
  uint64_t s0 = 0, s1 = 0;  // pairs of partial row sums
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t pk[16];
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      const int col = 32 * c + e;
      float x0, x1;
      unpack2(ffma2(pack2(__uint_as_float(v[col]), __uint_as_float(v[col + 1])), sl2x2, negm2), x0, x1);
      float p0 = ex2(x0), p1 = ex2(x1);
      if (kMasked) {
        if (col > lim) p0 = 0.f;
        if (col + 1 > lim) p1 = 0.f;
      }
      if ((e >> 1) & 1) s1 = fadd2(s1, pack2(p0, p1));
      else s0 = fadd2(s0, pack2(p0, p1));
      pk[e >> 1] = pack_p<kF16>(p0, p1);
    }
    tmem_st16(tS + c * 16, pk);
  }
  float l0, l1, l2, l3;
  unpack2(s0, l0, l1);
  unpack2(s1, l2, l3);
  return make_float2(m2, (l0 + l1) + (l2 + l3));
}

// E4M3 P for the kind::f8f6f4 P V (positive scales): P = 2^(v * sl2 - mb) with mb = m2 - 8,
// so P <= 256 (E4M3's largest value is 448) and values down to 2^-14 of the row maximum
// stay in E4M3's normal range; (mb, l) are returned, l summed from the unrounded P, and
// the combine merges them like any other base.  The row's 128 keys go to shared memory as
// one 128-byte K-major row (16-byte chunks swizzled by row % 8).
template <bool kMasked>
__device__ __forceinline__ float2 softmax_row_p8(uint32_t (&v)[128], int lim, float sl2, uint8_t* prow, int sw) {
  float a0 = -FLT_MAX, a1 = -FLT_MAX, a2 = -FLT_MAX, a3 = -FLT_MAX;
#pragma unroll
  for (int e = 0; e < 128; e += 8) {
    float x[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) x[q] = (kMasked && e + q > lim) ? -FLT_MAX : __uint_as_float(v[e + q]);
    a0 = max3(a0, x[0], x[1]);
    a1 = max3(a1, x[2], x[3]);
    a2 = max3(a2, x[4], x[5]);
    a3 = max3(a3, x[6], x[7]);
  }
  const float mb = fmaxf(fmaxf(a0, a1), fmaxf(a2, a3)) * sl2 - 8.f;
  const uint64_t sl2x2 = pack2(sl2, sl2), negm = pack2(-mb, -mb);
  uint64_t s0 = 0, s1 = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {  // keys 16 j .. 16 j + 15: one 16-byte chunk
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 16; e += 2) {
      const int col = 16 * j + e;
      float x0, x1;
      unpack2(ffma2(pack2(__uint_as_float(v[col]), __uint_as_float(v[col + 1])), sl2x2, negm), x0, x1);
      float p0 = ex2(x0), p1 = ex2(x1);
      if (kMasked) {
        if (col > lim) p0 = 0.f;
        if (col + 1 > lim) p1 = 0.f;
      }
      if ((e >> 1) & 1) s1 = fadd2(s1, pack2(p0, p1));
      else s0 = fadd2(s0, pack2(p0, p1));
      uint16_t h;
      asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(h) : "f"(p1), "f"(p0));
      if ((e >> 1) & 1) w[e >> 2] |= static_cast<uint32_t>(h) << 16;
      else w[e >> 2] = h;
    }
    *reinterpret_cast<uint4*>(prow + ((j ^ sw) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  float l0, l1, l2, l3;
  unpack2(s0, l0, l1);
  unpack2(s1, l2, l3);
  return make_float2(mb, (l0 + l1) + (l2 + l3));
}

// Any finite scale: the row extremum of v * sl2 taken directly (slower, rare).
template <bool kF16>
__device__ __forceinline__ float2 softmax_row_any_scale(uint32_t (&v)[128], int lim, float sl2, uint32_t tS) {
  float m2 = -FLT_MAX;
  for (int e = 0; e < 128; ++e)
    if (e <= lim) m2 = fmaxf(m2, __uint_as_float(v[e]) * sl2);
  float l = 0.f;
  for (int c = 0; c < 4; ++c) {
    uint32_t pk[16];
    for (int e = 0; e < 32; e += 2) {
      const int col = 32 * c + e;
      const float p0 = col <= lim ? ex2(fmaf(__uint_as_float(v[col]), sl2, -m2)) : 0.f;
      const float p1 = col + 1 <= lim ? ex2(fmaf(__uint_as_float(v[col + 1]), sl2, -m2)) : 0.f;
      l += p0 + p1;
      pk[e >> 1] = pack_p<kF16>(p0, p1);
    }
    tmem_st16(tS + c * 16, pk);
  }
  return make_float2(m2, l);
}

// kWithhold (a separate instance, test use only): the scheduler warp publishes no work,
// so every other role's bounded wait expires
template <bool kFp8, bool kF32P, bool kWithhold = false, bool kP8 = false>
__global__ void __launch_bounds__(kThreads, 1)
kv_outer_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                const __grid_constant__ CUtensorMap tmQ, const KvParams p) {
  griddep_wait();
  // (no early griddep_launch: a combine grid left pending for the whole persistent run of
  // this kernel cost 0.09 ms per M3 step; the combine is released when this grid ends)
  using L = Lay<kFp8, kP8>;
  const int path = p.force_path ? p.force_path : p.hdr->path;
  if (path != kPathKvOuter) return;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw_u & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sb = raw_u + pad;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffCtl);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffCtl + kOffTmemSlot);
  TileInfo* ring = reinterpret_cast<TileInfo*>(smem + L::kOffCtl + kOffRing);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // zero the Q stages once so rows of a partly filled tile (no TMA box for its missing
  // queries: they keep an earlier tile's finite values) never hold NaN patterns
  for (uint32_t o = tid * 16; o < kQStages * L::kInTile; o += kThreads * 16)
    *reinterpret_cast<uint4*>(smem + L::kOffQ + o) = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();

  if (tid == 0) {
    for (int s = 0; s < kQStages; ++s) {
      mbar_init(bar(B_QFULL0 + s), 1);
      mbar_init(bar(B_QFREE0 + s), 1);
    }
    for (int v = 0; v < 2; ++v) {
      mbar_init(bar(B_VFULL0 + v), 1);
      mbar_init(bar(B_VFREE0 + v), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_KFULL0 + s), 1);
      mbar_init(bar(B_KFREE0 + s), 1);
    }
    for (int r = 0; r < kRegions; ++r) {
      mbar_init(bar(B_SFULL0 + r), 1);
      mbar_init(bar(B_PFULL0 + r), 128);
      mbar_init(bar(B_PVDONE0 + r), 1);
      mbar_init(bar(B_OFREE0 + r), 128);
    }
    for (int r = 0; r < kRing; ++r) {
      mbar_init(bar(B_TFULL0 + r), 1);
      mbar_init(bar(B_TEMPTY0 + r), 2);  // released by the output warps and the K/V loader
    }
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
    regs_dec<kRegCtl>();
    if (warp == 0) {
      // (the withholding instance keeps this warp idle; the condition stays plain: folding
      // a second test into it slowed the kernel by 6%)
      if constexpr (!kWithhold) {
        // ---------------------------------------------------------- producer (whole warp)
        int* counter = &p.hdr->pad[0];
        const int T = p.hdr->ntiles;
        if (lane == 0) tma_prefetch_desc(&tmQ);
        const uint64_t pol_q = policy_evict_normal();
        const unsigned full = 0xffffffffu;
        // Metadata of a chunk, spread over the warp: lane k < 8 holds tile k's
        // (row, first, count, -) in `tile`; lane j holds the id of query (j % 8) of
        // tile j / 8 in qa and of tile j / 8 + 4 in qb.  Loaded one chunk ahead.
        struct Meta {
          int4 tile;
          int qa, qb, n;
        };
        auto load_tiles = [&](int c, Meta& m) {
          const int base = c * kChunkTiles;
          m.n = base < T ? min(kChunkTiles, T - base) : 0;
          m.tile = lane < m.n ? p.tiles[base + lane] : make_int4(0, 0, 0, 0);
        };
        auto load_ids = [&](Meta& m) {
          const int t0 = lane >> 3, j = lane & 7;
          const int f0 = __shfl_sync(full, m.tile.y, t0), n0 = __shfl_sync(full, m.tile.z, t0);
          const int f1 = __shfl_sync(full, m.tile.y, t0 + 4), n1 = __shfl_sync(full, m.tile.z, t0 + 4);
          const bool in0 = j < n0 && dbg_ok(f0 + j >= 0 && f0 + j < p.cap_e, &p.hdr->status);
          const bool in1 = j < n1 && dbg_ok(f1 + j >= 0 && f1 + j < p.cap_e, &p.hdr->status);
          m.qa = in0 ? p.qlist[f0 + j] : 0;
          m.qb = in1 ? p.qlist[f1 + j] : 0;
        };
        // lane 0 hands out chunk ids: one atomicAdd claims kClaimChunks consecutive chunks
        int claim_next = 0, claim_left = 0;
        auto claim = [&]() -> int {
          if (claim_left == 0) {
            claim_next = atomicAdd(counter, 1) * kClaimChunks;
            claim_left = kClaimChunks;
          }
          --claim_left;
          return claim_next++;
        };
        int c_cur = 0, c_next = 0, c_claim = 0;
        if (lane == 0) {
          c_cur = claim();
          c_next = claim();
          c_claim = claim();
        }
        c_cur = __shfl_sync(full, c_cur, 0);
        c_next = __shfl_sync(full, c_next, 0);
        Meta cur, nxt;
        load_tiles(c_cur, cur);
        load_ids(cur);
        load_tiles(c_next, nxt);
        // writes ring entry `it` (count 0 marks the end of the work); false on timeout
        auto publish = [&](int it, int row, int first, int count, int flags, int q) -> bool {
          const int slot = it % kRing;
          bool w = true;
          if (lane == 0) w = mbar_wait(bar(B_TEMPTY0 + slot), ((it / kRing) & 1) ^ 1);
          if (!__shfl_sync(full, w, 0)) return false;
          if (lane < kTileQ) ring[slot].q[lane] = q;
          if (lane == 0) {
            ring[slot].row = row;
            ring[slot].first = first;
            ring[slot].count = count;
            ring[slot].flags = flags;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(B_TFULL0 + slot));
          return true;
        };
        int it = 0, prev_row = -1, nk = 0;
        bool ok = true;
        while (ok) {
          if (cur.n == 0) {
            // two end markers: the softmax warpgroups read alternate entries
            for (int e = 0; e < 2 && ok; ++e) ok = publish(it + e, 0, 0, 0, 0, 0);
            break;
          }
          bool ids_next = false;
          for (int t = 0; t < cur.n; ++t, ++it) {
            if (t == 3) { load_ids(nxt); ids_next = true; }  // the next chunk's tiles have arrived by now
            int row = __shfl_sync(full, cur.tile.x, t);
            int first = __shfl_sync(full, cur.tile.y, t);
            int count = __shfl_sync(full, cur.tile.z, t);
            int qv = __shfl_sync(full, t < 4 ? cur.qa : cur.qb, ((t & 3) << 3) | (lane & 7));
            if (MSA_DEBUG) {
              // a tile record or query id out of range: the tile becomes one entry of row 0 at
              // position 0 (valid addresses; the status reports the fault)
              if (!dbg_ok(row >= 0 && row < p.R && count >= 1 && count <= kTileQ && first >= 0 &&
                              first + count <= p.cap_e, &p.hdr->status)) {
                row = 0;
                first = 0;
                count = 1;
              }
              if (lane < count && !dbg_ok(qv >= 0 && qv < p.N, &p.hdr->status)) qv = 0;
            }
            const bool new_row = row != prev_row;
            const int kb = new_row ? (nk & 1) : ((nk - 1) & 1);
            {
              // Q of this tile into stage it % 4 once S(it - 4) has read that stage: one TMA
              // box per query (its 16 heads, 4 KB bf16 / 2 KB E4M3), issued by lane j for
              // query j after lane 0 has armed the stage's barrier with the byte count
              const int qs = it % kQStages;
              bool w = true;
              if (lane == 0) {
                if (it >= kQStages) w = mbar_wait(bar(B_QFREE0 + qs), ((it / kQStages) - 1) & 1);
                if (w) mbar_expect_tx(bar(B_QFULL0 + qs), static_cast<uint32_t>(count) * (L::kInTile / kTileQ));
              }
              if (!__shfl_sync(full, w, 0)) { ok = false; break; }
              if (lane < count) {
                const uint32_t dq = sb + L::kOffQ + qs * L::kInTile + lane * (L::kInTile / kTileQ);
                const int g = row / p.nblocks;
                if constexpr (kFp8) tma_load_3d(dq, &tmQ, 0, g * kGroup, qv, bar(B_QFULL0 + qs), pol_q);
                else tma_load_5d(dq, &tmQ, 0, 0, 0, 2 * g, qv, bar(B_QFULL0 + qs), pol_q);
              }
            }
            if (!publish(it, row, first, count, (new_row ? 1 : 0) | (kb << 8), qv)) { ok = false; break; }
            if (new_row) {
              ++nk;
              prev_row = row;
            }
          }
          if (!ok) break;
          if (!ids_next) load_ids(nxt);
          cur = nxt;
          // claim the chunk after next; the claim made a chunk ago becomes the next one
          const int claimed = __shfl_sync(full, c_claim, 0);
          if (lane == 0 && claimed * kChunkTiles < T) c_claim = claim();
          load_tiles(claimed, nxt);
        }
        if (!ok && lane == 0) flag_timeout(p.hdr);
      }
    } else if (warp == 1) {
      // ---------------------------------------------------------- S = Q K^T issuer
      if (lane == 0) {
        constexpr uint32_t idesc_qk = kFp8 ? idesc_f8(128, 128, 0, 0) : idesc_f16(128, 128, 1, 1, 0, 0);
        bool ok = true;
        int seg = -1;
        for (int it = 0;; ++it) {
          const int slot = it % kRing;
          if (!(ok = mbar_wait(bar(B_TFULL0 + slot), (it / kRing) & 1))) break;
          const int count = ring[slot].count, flags = ring[slot].flags;
          if (count == 0) break;
          const int r = it & 3;  // TMEM region of this tile's S and P
          if (flags & 1) {
            // a new row: the previous row's K buffer is read no more once the S MMAs
            // issued so far are done
            if (++seg > 0) mma_commit(bar(B_KFREE0 + ((seg - 1) & 1)));
          }
          // region r last held O of tile it - 3: the output warps must have read it
          if (it >= 3 && !(ok = mbar_wait(bar(B_OFREE0 + ((it - 3) & 3)), ((it - 3) >> 2) & 1))) break;
          if ((flags & 1) && !(ok = mbar_wait(bar(B_KFULL0 + (seg & 1)), (seg >> 1) & 1))) break;
          const int qs = it % kQStages;
          if (!(ok = mbar_wait(bar(B_QFULL0 + qs), (it / kQStages) & 1))) break;
          tc_fence_after();
          const uint32_t qa = sb + L::kOffQ + qs * L::kInTile, ka = sb + ((seg & 1) ? L::kOffK1 : L::kOffK0);
          if constexpr (kFp8) {
            // E4M3: K = 128 bytes = one swizzle span, 32 elements per MMA
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_f8_ss(tmem + r * 128, smem_desc(qa + k * 32, 16, 1024, 2), smem_desc(ka + k * 32, 16, 1024, 2),
                        idesc_qk, k > 0);
          } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              // Q: [query][8-head group][D half][8 rows][128 B] (8-row groups 2048 B apart,
              // D halves 1024 B apart); K: [D half][128 rows][128 B]
              mma_f16_ss(tmem + r * 128, smem_desc(qa + (k >> 2) * 1024 + (k & 3) * 32, 16, 2048, 2),
                         smem_desc(ka + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024, 2), idesc_qk, k > 0);
            }
          }
          mma_commit(bar(B_SFULL0 + r));
          mma_commit(bar(B_QFREE0 + qs));  // the scheduler may load tile it + 3's Q into this stage
        }
        if (!ok) flag_timeout(p.hdr);
      }
    } else if (warp == 2) {
      // ---------------------------------------------------------- K/V loader (lane 0 issues,
      // the whole warp converts E4M3 V to f16)
      const unsigned full = 0xffffffffu;
      if (lane == 0) { tma_prefetch_desc(&tmK); tma_prefetch_desc(&tmV); }
      const uint64_t pol_kv = policy_evict_last();
      int nk = 0;
      bool ok = true;
      for (int it = 0; ok; ++it) {
        const int slot = it % kRing;
        int count = 0, row = 0, flags = 0;
        if (lane == 0) {
          ok = mbar_wait(bar(B_TFULL0 + slot), (it / kRing) & 1);
          if (ok) {
            count = ring[slot].count;
            row = ring[slot].row;
            flags = ring[slot].flags;
            mbar_arrive(bar(B_TEMPTY0 + slot));
          }
        }
        ok = __shfl_sync(full, ok, 0);
        count = __shfl_sync(full, count, 0);
        row = __shfl_sync(full, row, 0);
        flags = __shfl_sync(full, flags, 0);
        if (!ok || count == 0) break;
        if (!(flags & 1)) continue;
        const int g = row / p.nblocks, b = row - g * p.nblocks, kb = nk & 1;
        const int vb = nk % L::kVBuf, vuse = nk / L::kVBuf;  // V buffer of this row, its use count
        if (lane == 0) {
          // K: two buffers, buffer kb was last read by the row before the previous one
          const uint32_t dk = sb + (kb ? L::kOffK1 : L::kOffK0);
          ok = mbar_wait(bar(B_KFREE0 + kb), ((nk >> 1) & 1) ^ 1);
          if (ok) {
            mbar_expect_tx(bar(B_KFULL0 + kb), L::kInTile);
            tma_load_3d(dk, &tmK, 0, g, b * kBlock, bar(B_KFULL0 + kb), pol_kv);
            if constexpr (!kFp8) tma_load_3d(dk + 16384, &tmK, 64, g, b * kBlock, bar(B_KFULL0 + kb), pol_kv);
            // V buffer vb: free once the last P V of the row that used it before is done
            ok = mbar_wait(bar(B_VFREE0 + vb), (vuse & 1) ^ 1);
          }
          if (ok) {
            // V (bf16, or the f16 copy of E4M3 V): two 64-column boxes of 128-byte rows
            const uint32_t dv = sb + L::kOffV + vb * L::kVTile;
            mbar_expect_tx(bar(B_VFULL0 + vb), L::kVTile);
            if constexpr (kP8) {  // the block's E4M3 V^T: 128 rows (d) of 128 keys, one box
              tma_load_3d(dv, &tmV, 0, 0, row, bar(B_VFULL0 + vb), pol_kv);
            } else {
              tma_load_3d(dv, &tmV, 0, g, b * kBlock, bar(B_VFULL0 + vb), pol_kv);
              tma_load_3d(dv + 16384, &tmV, 64, g, b * kBlock, bar(B_VFULL0 + vb), pol_kv);
            }
          }
        }
        ok = __shfl_sync(full, ok, 0);
        if (!ok) break;
        ++nk;
      }
      if (!ok && lane == 0) flag_timeout(p.hdr);
    } else if (warp == 3) {
      // ---------------------------------------------------------- O = P V issuer
      if (lane == 0) {
        // P V: f16 x f16 for the E4M3 path (V converted to f16), bf16 x bf16 otherwise; V MN-major
        constexpr uint32_t idesc_pv = kFp8 ? idesc_f16(128, 128, 0, 0, 0, 1) : idesc_f16(128, 128, 1, 1, 0, 1);
        bool ok = true;
        int vseg = -1;
        for (int u = 0;; ++u) {
          const int slot = u % kRing;
          if (!(ok = mbar_wait(bar(B_TFULL0 + slot), (u / kRing) & 1))) break;
          const int count = ring[slot].count, flags = ring[slot].flags;
          if (count == 0) break;
          const int r = u & 3, ro = (u + 3) & 3;  // P in region r, O into region ro
          if (flags & 1) {
            // a new row: the previous row's V buffer is free once the P V MMAs issued so far are done
            if (++vseg > 0) mma_commit(bar(B_VFREE0 + (vseg - 1) % L::kVBuf));
            if (!(ok = mbar_wait(bar(B_VFULL0 + vseg % L::kVBuf), (vseg / L::kVBuf) & 1))) break;
          }
          if (!(ok = mbar_wait(bar(B_PFULL0 + r), (u >> 2) & 1))) break;
          // O goes over the P of tile u - 1: its P V must have completed
          if (u >= 1 && !(ok = mbar_wait(bar(B_PVDONE0 + ((u - 1) & 3)), ((u - 1) >> 2) & 1))) break;
          tc_fence_after();
          const uint32_t va = sb + L::kOffV + (vseg % L::kVBuf) * L::kVTile;
          if constexpr (kP8) {
            // E4M3 P (shared memory, buffer u % 2) x E4M3 V^T, both K-major: 32 keys per MMA
            const uint32_t pa = sb + L::kOffP + (u & 1) * 16384;
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_f8_ss(tmem + ro * 128, smem_desc(pa + k * 32, 16, 1024, 2), smem_desc(va + k * 32, 16, 1024, 2),
                        idesc_f8(128, 128, 0, 0), k > 0);
          } else {
#pragma unroll
            for (int k = 0; k < 8; ++k)
              mma_f16_ts(tmem + ro * 128, tmem + r * 128 + k * 8, smem_desc(va + k * 2048, 16384, 1024, 2),
                         idesc_pv, k > 0);
          }
          mma_commit(bar(B_PVDONE0 + r));
        }
        if (!ok) flag_timeout(p.hdr);
      }
    }
  } else if (warp < 12) {
    regs_inc<kRegSoftmax>();
    // ------------------------------------------------------------ softmax
    const int wg = (warp - 4) >> 2;  // 0 or 1: the stage (tile parity) handled
    const int row = 32 * (warp & 3) + lane;
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const bool neg = p.sl2 < 0.f;  // a negative scale turns the row maximum into a minimum
    // Each warp decides for itself (tcgen05.ld / st are warp-collective, not warpgroup-
    // collective): a bounded wait that expires in one warp ends that warp's loop, and the
    // others' waits then expire too, since the arrivals they wait for never come.
    for (int it = wg;; it += 2) {
      const int slot = it % kRing;
      bool ok = mbar_wait(bar(B_TFULL0 + slot), (it / kRing) & 1);
      if (!__all_sync(0xffffffffu, ok)) { flag_timeout(p.hdr); break; }
      const int count = ring[slot].count;
      if (count == 0) break;
      const int j = row >> 4;
      const bool valid = j < count;
      const int qi = valid ? ring[slot].q[j] : 0;
      const int first = ring[slot].first;
      const int b = ring[slot].row % p.nblocks;
      // keys c <= lim are visible; only rows whose own block is b are masked
      const int lim = valid ? (p.Lkv - p.N + qi) - b * kBlock : kBlock - 1;
      // The branch below contains warp-collective tcgen05.st: take it warp-uniformly
      // (a row with lim >= 127 is unaffected by the masked path).
      const bool masked = __any_sync(0xffffffffu, lim < kBlock - 1);

      ok = mbar_wait(bar(B_SFULL0 + (it & 3)), (it >> 2) & 1);
      if (!__all_sync(0xffffffffu, ok)) { flag_timeout(p.hdr); break; }
      tc_fence_after();
      const uint32_t tS = tmem + lane_base + (it & 3) * 128;
      uint32_t v[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32 * c]));
      tmem_ld_wait();
      float2 ml;
      if constexpr (kP8) {
        // P buffer it % 2 was last read by the P V of tile it - 2 (the host runs this instance
        // for positive scales only)
        if (it >= 2) {
          ok = mbar_wait(bar(B_PVDONE0 + ((it - 2) & 3)), ((it - 2) >> 2) & 1);
          if (!__all_sync(0xffffffffu, ok)) { flag_timeout(p.hdr); break; }
        }
        uint8_t* prow = smem + L::kOffP + (it & 1) * 16384 + (row >> 3) * 1024 + (row & 7) * 128;
        ml = masked ? softmax_row_p8<true>(v, lim, p.sl2, prow, row & 7) : softmax_row_p8<false>(v, lim, p.sl2, prow, row & 7);
        fence_proxy_async_smem();  // generic-proxy writes of P before the MMA reads them
      } else {
        if (neg) ml = softmax_row_any_scale<kFp8>(v, lim, p.sl2, tS);
        else if (masked) ml = softmax_row<true, kFp8>(v, lim, p.sl2, tS);
        else ml = softmax_row<false, kFp8>(v, lim, p.sl2, tS);
        tmem_st_wait();
      }
      tc_fence_before();
      mbar_arrive(bar(B_PFULL0 + (it & 3)));
      if (valid) p.pstat[static_cast<size_t>(first) * kGroup + row] = ml;
    }
  } else {
    regs_dec<kRegOut>();
    // ------------------------------------------------------------ output (raw O -> global)
    const uint32_t bar_id = 3;
    const int row = 32 * (warp & 3) + lane;
    const int jr = row >> 4, h = row & 15;
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const bool elected = (tid == 384);
    const uint64_t pol_st = policy_evict_first();
    constexpr int kChunks = kF32P ? 32 : 16;
    for (int it = 0;; ++it) {
      const int slot = it % kRing;
      bool ok = mbar_wait(bar(B_TFULL0 + slot), (it / kRing) & 1);
      if (!named_bar_and(bar_id, 128, ok)) { flag_timeout(p.hdr); break; }
      const int count = ring[slot].count, first = ring[slot].first;
      if (count == 0) break;
      const int s = it & 3;
      ok = mbar_wait(bar(B_PVDONE0 + s), (it >> 2) & 1);
      if (!named_bar_and(bar_id, 128, ok)) { flag_timeout(p.hdr); break; }
      if (elected) mbar_arrive(bar(B_TEMPTY0 + slot));
      tc_fence_after();
      const uint32_t tO = tmem + lane_base + ((it + 3) & 3) * 128;
      const bool store = jr < count;
      uint4* dst = p.partial + part_index(static_cast<int64_t>(first) + jr, h, 0, kChunks);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld32(tO + c * 32, v);
        tmem_ld_wait();
        if (c == 3) {
          tc_fence_before();
          mbar_arrive(bar(B_OFREE0 + s));
        }
        if (store) {
          if constexpr (kF32P) {
#pragma unroll
            for (int q = 0; q < 8; ++q)
              st_global_v4_hint(dst + (c * 8 + q) * (kPartGroup * kGroup), v[4 * q], v[4 * q + 1], v[4 * q + 2],
                                v[4 * q + 3], pol_st);
          } else {
#pragma unroll
            for (int q = 0; q < 4; ++q)
              st_global_v4_hint(dst + (c * 4 + q) * (kPartGroup * kGroup),
                                pack_bf16x2(__uint_as_float(v[q * 8 + 0]), __uint_as_float(v[q * 8 + 1])),
                                pack_bf16x2(__uint_as_float(v[q * 8 + 2]), __uint_as_float(v[q * 8 + 3])),
                                pack_bf16x2(__uint_as_float(v[q * 8 + 4]), __uint_as_float(v[q * 8 + 5])),
                                pack_bf16x2(__uint_as_float(v[q * 8 + 6]), __uint_as_float(v[q * 8 + 7])), pol_st);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// E4M3 -> f16, elementwise and exact (every E4M3 value is an f16 value): 16 source bytes
// per thread and step, read once (streaming), written as two 16-byte f16 chunks in order.
__global__ void __launch_bounds__(256) widen_e4m3_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                         int64_t n16, const SchedHeader* __restrict__ hdr,
                                                         int force_path) {
  griddep_wait();
  griddep_launch();
  if ((force_path ? force_path : hdr->path) != kPathKvOuter) return;  // only the KV-outer kernel reads the copy
  for (int64_t i = blockIdx.x * 256ll + threadIdx.x; i < n16; i += static_cast<int64_t>(gridDim.x) * 256) {
    const uint4 v = __ldcs(src + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t h[8];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h[2 * q]) : "h"(static_cast<uint16_t>(w[q] & 0xFFFFu)));
      asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h[2 * q + 1]) : "h"(static_cast<uint16_t>(w[q] >> 16)));
    }
    dst[2 * i] = make_uint4(h[0], h[1], h[2], h[3]);
    dst[2 * i + 1] = make_uint4(h[4], h[5], h[6], h[7]);
  }
}

}  // namespace

cudaError_t launch_widen_e4m3(const void* src, void* dst, int64_t n, const SchedHeader* hdr, int force_path,
                              cudaStream_t st) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t n16 = n / 16;
  int64_t grid = (n16 + 255) / 256;
  if (grid > sms * 8) grid = sms * 8;
  if (grid < 1) grid = 1;
  MSA_LAUNCH(widen_e4m3_kernel, static_cast<int>(grid), 256, 0, st, static_cast<const uint4*>(src), static_cast<uint4*>(dst),
             n16, hdr, force_path);
  return cudaGetLastError();
}

namespace {

// E4M3 V [Lkv][Hkv][128] -> V^T per (group, block): vt[(g * nblocks + b) * 128 + d][key], 128
// keys of one d in 128 contiguous bytes (16 KB per block), so that P V can read V as a
// K-major E4M3 operand.  One CTA per (group, block): the block goes through shared memory
// (rows padded to 129 bytes), 16-byte loads and stores.
__global__ void __launch_bounds__(256) transpose_e4m3_kernel(const uint8_t* __restrict__ v, uint8_t* __restrict__ vt,
                                                             int Hkv, int nblocks, const SchedHeader* __restrict__ hdr,
                                                             int force_path) {
  griddep_wait();
  griddep_launch();
  if ((force_path ? force_path : hdr->path) != kPathKvOuter) return;
  __shared__ uint8_t tile[128 * 129];
  const int gb = blockIdx.x, g = gb / nblocks, b = gb - g * nblocks;
  const int t = threadIdx.x;
#pragma unroll
  for (int i = 0; i < 4; ++i) {  // key = q / 8, 16-byte chunk q % 8 of its row
    const int q = t + 256 * i, key = q >> 3, c = q & 7;
    const uint4 w = __ldcs(reinterpret_cast<const uint4*>(v + ((static_cast<size_t>(b) * kBlock + key) * Hkv + g) * kHeadDim) + c);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 16; ++j) tile[key * 129 + 16 * c + j] = static_cast<uint8_t>(ws[j >> 2] >> (8 * (j & 3)));
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 4; ++i) {  // d = q / 8, keys 16 (q % 8) .. + 15
    const int q = t + 256 * i, d = q >> 3, k0 = 16 * (q & 7);
    uint32_t ws[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int j = 0; j < 16; ++j) ws[j >> 2] |= static_cast<uint32_t>(tile[(k0 + j) * 129 + d]) << (8 * (j & 3));
    reinterpret_cast<uint4*>(vt + (static_cast<size_t>(gb) * kHeadDim + d) * kBlock)[q & 7] =
        make_uint4(ws[0], ws[1], ws[2], ws[3]);
  }
}

}  // namespace

cudaError_t launch_transpose_e4m3(const void* v, void* vt, int Hkv, int nblocks, const SchedHeader* hdr, int force_path,
                                  cudaStream_t st) {
  MSA_LAUNCH(transpose_e4m3_kernel, Hkv * nblocks, 256, 0, st, static_cast<const uint8_t*>(v), static_cast<uint8_t*>(vt),
             Hkv, nblocks, hdr, force_path);
  return cudaGetLastError();
}

cudaError_t launch_kv_outer(const KvOuterArgs& a, cudaStream_t st) {
  if (a.force_path == kPathQOuter) return cudaSuccess;  // (the kernel would exit at once)
  const msa_schedule* s = a.s;
  const bool fp8 = a.fp8;
  const uint64_t es = fp8 ? 1 : 2;  // bytes per input element
  CUtensorMap tmK, tmV, tmQ;
  {
    // Q [N][Hq][128]: bf16 as a 5-D view (64 elements of a D half, head within 8, D half,
    // group of 8 heads, query): one box = one query's 16 heads, 4 KB, landing as
    // [8-head group][D half][8 rows][128 B]; E4M3 as (128 elements, head, query), one box
    // = 16 rows of 128 B
    const uint64_t es = a.fp8 ? 1 : 2;
    const uint64_t row = kHeadDim * es;
    if (a.fp8) {
      const uint64_t dims[3] = {kHeadDim, static_cast<uint64_t>(a.Hq), static_cast<uint64_t>(s->N)};
      const uint64_t strides[2] = {row, static_cast<uint64_t>(a.Hq) * row};
      const uint32_t box[3] = {128, 16, 1};
      if (!encode_tmap(&tmQ, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, a.Q, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    } else {
      const uint64_t dims[5] = {64, 8, 2, static_cast<uint64_t>(a.Hq) / 8, static_cast<uint64_t>(s->N)};
      const uint64_t strides[4] = {row, 128, 8 * row, static_cast<uint64_t>(a.Hq) * row};
      const uint32_t box[5] = {64, 8, 2, 2, 1};
      if (!encode_tmap(&tmQ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, a.Q, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    }
  }
  {
    // K / V [Lkv][Hkv][128]: one block of one group per load, 64 elements (bf16) or
    // 128 elements (E4M3) = 128 bytes per box row
    const CUtensorMapDataType dt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const uint64_t dims[3] = {kHeadDim, static_cast<uint64_t>(s->Hkv), static_cast<uint64_t>(a.Lkv)};
    const uint64_t strides[2] = {kHeadDim * es, static_cast<uint64_t>(s->Hkv) * kHeadDim * es};
    const uint32_t box[3] = {fp8 ? 128u : 64u, 1, kBlock};
    if (!encode_tmap(&tmK, dt, 3, a.K, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
    // V: bf16, or (E4M3 inputs) the f16 copy made by launch_widen_e4m3, 64 elements per box row
    const uint64_t vstrides[2] = {kHeadDim * 2, static_cast<uint64_t>(s->Hkv) * kHeadDim * 2};
    const uint32_t vbox[3] = {64u, 1, kBlock};
    if (a.p8) {
      // E4M3 P V: V^T [Hkv * nblocks][128 d][128 keys] (launch_transpose_e4m3), one block per box
      const uint64_t tdims[3] = {kBlock, kHeadDim, static_cast<uint64_t>(s->Hkv) * s->nblocks};
      const uint64_t tstrides[2] = {kBlock, static_cast<uint64_t>(kBlock) * kHeadDim};
      const uint32_t tbox[3] = {kBlock, kHeadDim, 1};
      if (!encode_tmap(&tmV, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, a.Vf16, tdims, tstrides, tbox, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    } else if (!encode_tmap(&tmV, fp8 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                            fp8 ? a.Vf16 : a.V, dims, vstrides, vbox, CU_TENSOR_MAP_SWIZZLE_128B)) {
      return cudaErrorInvalidValue;
    }
  }
  KvParams p;
  p.Q = static_cast<const uint8_t*>(a.Q);
  p.partial = static_cast<uint4*>(s->partial);
  p.Hq = a.Hq;
  p.tiles = s->d.tiles;
  p.qlist = s->d.qlist;
  p.hdr = s->d.hdr;
  p.pstat = s->pstat;
  p.N = s->N;
  p.Lkv = a.Lkv;
  p.nblocks = s->nblocks;
  p.R = s->R;
  p.cap_e = s->cap_entries;
  p.sl2 = a.scale * a.qk_descale * 1.4426950408889634f;
  p.force_path = a.force_path;
  static std::atomic<uint64_t> attr_done[5];
  const int inst = a.p8 ? 4 : (fp8 ? 1 : 0) | (a.f32p ? 2 : 0);
  void (*kern)(CUtensorMap, CUtensorMap, CUtensorMap, KvParams);
  switch (inst) {
    case 0: kern = kv_outer_kernel<false, false>; break;
    case 1: kern = kv_outer_kernel<true, false>; break;
    case 2: kern = kv_outer_kernel<false, true>; break;
    case 3: kern = kv_outer_kernel<true, true>; break;
    default: kern = kv_outer_kernel<true, false, false, true>; break;  // E4M3 P V
  }
  // test use: the bf16 instance whose scheduler publishes no work
  const bool withhold = (a.debug_flags & 1) != 0 && inst == 0;
  if (withhold) kern = kv_outer_kernel<false, false, true>;
  const uint32_t smem = a.p8 ? Lay<true, true>::kSmemBytes : fp8 ? Lay<true>::kSmemBytes : Lay<false>::kSmemBytes;
  if (withhold) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
  } else {
    cudaError_t e = set_smem_limit(kern, static_cast<int>(smem), attr_done[inst]);
    if (e != cudaSuccess) return e;
  }
  // the chunk counter this launch claims its work from is zero: the schedule build clears the
  // header and the combine kernel that follows every launch of this kernel clears the counter
  // again (a memset here would break the launch chain's programmatic dependency)
  // no more CTAs than work-list chunks can exist (decode sizes: a few; also makes the
  // launch cheap where the device picks the Q-outer path and this kernel exits at once)
  const int64_t max_claims = (s->cap_tiles + kChunkTiles * kClaimChunks - 1) / (kChunkTiles * kClaimChunks);
  const int grid = max_claims < a.num_ctas ? static_cast<int>(max_claims) : a.num_ctas;
  MSA_LAUNCH(kern, grid, kThreads, smem, st, tmK, tmV, tmQ, p);
  return cudaGetLastError();
}

}  // namespace msa
