// Backward of the block-sparse forward: dQ, dK, dV over the cached block lists.
//
// "Flash-MSA: accelerating million-token training with sparse attention", order of
// operations: the forward keeps the block indices it attended and its log-sum-exp,
// and the backward computes the main-attention gradients over the same blocks.  With
// P = exp(scale * Q K^T - LSE) restricted to the visible keys of the selected blocks
// and D = rowsum(dO * O) (equal to sum_j P_j dP_j):
//   dP = dO V^T,  dS = P * (dP - D),  dV = P^T dO,  dK = scale * dS^T Q,  dQ = scale * dS K.
//
// The backward reuses the forward's reverse index ("Sparse Attention", Chapter 5):
// row r = (group g, block b) lists the queries that selected b.  It is KV-stationary:
// one CTA holds K_b and V_b and walks the queries of a unit (at most kUnitEntries
// consecutive entries of one row) in tiles of 8 queries x 16 heads = 128 MMA rows,
// accumulating dK_b and dV_b in TMEM (M = the block's 128 keys) and writing each
// entry's dQ contribution dS K_b (bf16, 16 rows per entry) to the partial slab.
// Kernels:
//   bwd_prep_kernel     D[i, h] = dO[i, h, :] . O[i, h, :]
//   bwd_units_kernel    units (row, first entry, count) and their per-row offsets
//   bwd_kv_kernel       the tcgen05 kernel above; fp32 dK/dV per unit
//   bwd_reduce_kernel   dK = scale * sum over a row's units, dV = sum; bf16; zero for
//                       blocks nobody selected
//   bwd_dq_kernel       dQ[i, g heads] = scale * sum of the entry partials of (i, g)
// Every reduction runs in a fixed order, so results do not depend on scheduling.
//
// bwd_kv_kernel, one CTA of 512 threads per SM, persistent (units claimed with an
// atomicAdd).  It works on the transposed products so that the block's keys sit on the
// TMEM lanes: S^T = K_b Q^T and dP^T = V_b dO^T (M = keys, N = the tile's 128 rows);
// P^T = exp2(S^T * scale * log2 e - LSE * log2 e) is written back to TMEM as bf16 and
// feeds dV += P^T dO as the A operand read from TMEM; dS^T = P^T (dP^T - D) goes to
// shared memory, one 128-byte row per key, which serves dK += dS^T Q (read K-major) and
// dQ = dS K_b (read MN-major, M = rows); dQ lands in the columns dP^T held.  TMEM (512
// columns): [0, 128) S^T -> P^T (bf16 pairs), [128, 256) dP^T -> dQ, [256, 384) dV,
// [384, 512) dK.  Shared memory, bf16 128 x 128 tiles with the
// 128-byte swizzle: K_b, V_b (TMA) and dS as two 64-column halves, so one tile is K-major
// for a matrix and MN-major for its transpose (dS serves dQ as A = dS, M = rows, and dK as
// A = dS^T, M = keys); Q and dO in two stages, one TMA box of 4 KB per query laid out as
// [8-row group][D half][8 rows] (K-major with 2 KB between row groups, MN-major with the
// D halves 1 KB apart).  Warp roles:
//   warp 0      producer: claims units, loads K_b / V_b and gathers Q / dO of each tile
//               into the stage the tile uses, publishes tiles in a 4-slot ring
//   warp 1      TMEM allocation and MMA issue (one thread)
//   warps 4-11  two warpgroups, one per half of the tile's rows: thread = key (TMEM
//               lane); P^T, dS^T for its 64 rows, dS to shared memory
//   warps 12-15 evacuation: dQ rows of each tile (bf16 partial rows) and, at the end
//               of a unit, its dK / dV (fp32, thread = key)
// The MMAs of tile t + 1 start once dQ of tile t has left TMEM; the gathers run two
// tiles ahead of the MMAs.
#include <cuda_bf16.h>

#include "msa_internal.h"
#include "ptx.cuh"

namespace msa {
namespace {

constexpr int kThreads = 512;
// setmaxnreg shares (control, each compute warpgroup, evacuation): their sum over the
// four warpgroups must stay within the launch allocation (512 threads x 128 registers)
constexpr uint32_t kRegCtl = 96, kRegCompute = 168, kRegEvac = 80;
static_assert(kThreads == 512 && 128 * (kRegCtl + 2 * kRegCompute + kRegEvac) <= 512 * 128,
              "setmaxnreg shares exceed the launch allocation");
constexpr int kRing = 4;
constexpr uint32_t kTile = 32768;  // bf16 128 x 128
// control area at the (16-byte aligned) start of shared memory, tiles after it at the
// next 1024-byte boundary
constexpr uint32_t kCtlBytes = 2048;
constexpr uint32_t kOffRing = 512, kOffLD = 1024;  // ring: kRing x 64 B; per compute warpgroup 512 B of (LSE, D)
constexpr uint32_t kOffK = 0, kOffV = kTile, kOffQ0 = 2 * kTile, kOffDO0 = 4 * kTile, kOffDS = 6 * kTile;
constexpr uint32_t kTilesBytes = 7 * kTile;
constexpr uint32_t kSmemBytes = kCtlBytes + 1024 + kTilesBytes;
static_assert(kSmemBytes <= 232448, "shared memory");
enum {
  B_TFULL0 = 0, B_TEMPTY0 = kRing, B_QFULL0 = 2 * kRing, B_QFREE0 = 2 * kRing + 2, B_KVFULL = 2 * kRing + 4,
  B_KVFREE, B_SFULL, B_DPFULL, B_PREADY, B_DSREADY, B_DVDONE, B_MMA2, B_DQFREE, B_DSFREE, B_DKVFREE, B_COUNT
};
static_assert(8 * B_COUNT + 4 <= kOffRing, "control area");

// One published tile: its first CSR position, entry count (0 = no more work), schedule
// row, flags (bit 0 first tile of its unit, bit 1 last), unit id, query ids.
struct BTile {
  int e0, cnt, row, flags, uid, pad[3];
  int q[kTileQ];
};
static_assert(sizeof(BTile) == 64, "ring entry");

struct BwdParams {
  const float* LSE2;  // [N * Hq]: LSE * log2 e
  const float* Dv;    // [N * Hq]: D = dO . O
  const int4* units;
  const int32_t* qlist;
  int32_t* counter;
  const int32_t* nunits;
  float* dkv;              // [units][2][128][128]: dK then dV
  SchedHeader* hdr;
  int N, Lkv, Hq, nblocks;
  int R;          // schedule rows (Hkv * nblocks)
  int64_t cap_e;  // CSR positions the schedule holds
  float sl2;  // scale * log2(e)
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void lds4(uint32_t addr, float& a, float& b, float& c, float& d) {
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(a), "=f"(b), "=f"(c), "=f"(d) : "r"(addr) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
template <uint32_t N>
__device__ __forceinline__ void regs_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N)); }
template <uint32_t N>
__device__ __forceinline__ void regs_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N)); }

__global__ void __launch_bounds__(kThreads, 1)
bwd_kv_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
              const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
              const __grid_constant__ CUtensorMap tmP128, const __grid_constant__ CUtensorMap tmP16, const BwdParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint8_t* ctl = smem_raw;
  const uint32_t raw_u = smem_u32(smem_raw);
  const uint32_t sb = (raw_u + kCtlBytes + 1023u) & ~1023u;  // tiles, 1024-byte aligned
  uint8_t* smem = smem_raw + (sb - raw_u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(ctl);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctl + 8 * B_COUNT);
  BTile* ring = reinterpret_cast<BTile*>(ctl + kOffRing);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // stale rows of a partly filled tile are weighted 0; zero the Q / dO stages once so
  // that they never hold NaN bit patterns
  for (uint32_t o = tid * 16; o < 4 * kTile; o += kThreads * 16)
    *reinterpret_cast<uint4*>(smem + kOffQ0 + o) = make_uint4(0, 0, 0, 0);
  if (tid < 64) reinterpret_cast<uint4*>(ctl + kOffLD)[tid] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (tid == 0) {
    for (int r = 0; r < kRing; ++r) {
      mbar_init(bar(B_TFULL0 + r), 1);
      mbar_init(bar(B_TEMPTY0 + r), 4);  // MMA thread, two compute warpgroups, evacuation
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_QFULL0 + s), 1);
      mbar_init(bar(B_QFREE0 + s), 1);
    }
    mbar_init(bar(B_KVFULL), 1);
    mbar_init(bar(B_KVFREE), 1);
    mbar_init(bar(B_SFULL), 1);
    mbar_init(bar(B_DPFULL), 1);
    mbar_init(bar(B_PREADY), 2);
    mbar_init(bar(B_DSREADY), 2);
    mbar_init(bar(B_DVDONE), 1);
    mbar_init(bar(B_DSFREE), 1);
    mbar_init(bar(B_MMA2), 1);
    mbar_init(bar(B_DQFREE), 1);
    mbar_init(bar(B_DKVFREE), 1);
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
    if (warp == 0 && lane == 0) {
      // ------------------------------------------------------------ producer
      tma_prefetch_desc(&tmK); tma_prefetch_desc(&tmV); tma_prefetch_desc(&tmQ); tma_prefetch_desc(&tmDO);
      const uint64_t pol_kv = policy_evict_last(), pol_q = policy_evict_normal();
      const int nunits = *p.nunits;
      int it = 0, nu = 0;
      bool ok = true;
      // waits for ring slot `it`; false on timeout
      auto slot_free = [&](int t) {
        return t < kRing || mbar_wait(bar(B_TEMPTY0 + t % kRing), ((t / kRing) & 1) ^ 1);
      };
      while (ok) {
        const int u = atomicAdd(p.counter, 1);
        if (u >= nunits) {
          if ((ok = slot_free(it))) {
            ring[it % kRing].cnt = 0;
            mbar_arrive(bar(B_TFULL0 + it % kRing));
          }
          break;
        }
        int4 un = p.units[u];
        // (bounds-checked build: a unit record out of range becomes one entry of row 0)
        if (!dbg_ok(un.x >= 0 && un.x < p.R && un.y >= 0 && un.z >= 1 && un.y + un.z <= p.cap_e, &p.hdr->status))
          un = make_int4(0, 0, 1, un.w);
        const int g = un.x / p.nblocks, b = un.x - g * p.nblocks;
        const int ntile = (un.z + kTileQ - 1) / kTileQ;
        for (int t = 0; t < ntile && ok; ++t, ++it) {
          const int slot = it % kRing, s = it & 1;
          if (!(ok = slot_free(it))) break;
          if (it >= 2 && !(ok = mbar_wait(bar(B_QFREE0 + s), ((it - 2) >> 1) & 1))) break;
          const int e0 = un.y + t * kTileQ, cnt = min(kTileQ, un.z - t * kTileQ);
          BTile& tl = ring[slot];
          tl.e0 = e0;
          tl.cnt = cnt;
          tl.row = un.x;
          tl.flags = (t == 0 ? 1 : 0) | (t == ntile - 1 ? 2 : 0);
          tl.uid = u;
          const uint32_t bq = bar(B_QFULL0 + s);
          mbar_expect_tx(bq, static_cast<uint32_t>(cnt) * 8192u);
          const uint32_t dq = sb + kOffQ0 + s * kTile, ddo = sb + kOffDO0 + s * kTile;
          for (int j = 0; j < cnt; ++j) {
            // one 4 KB box per query and tensor: its 16 heads as two 8-row groups, each
            // with both D halves ([group][D half][8 rows][128 B])
            int q = __ldg(p.qlist + e0 + j);
            if (!dbg_ok(q >= 0 && q < p.N, &p.hdr->status)) q = 0;
            tl.q[j] = q;
            tma_load_5d(dq + j * 4096, &tmQ, 0, 0, 0, 2 * g, q, bq, pol_q);
            tma_load_5d(ddo + j * 4096, &tmDO, 0, 0, 0, 2 * g, q, bq, pol_q);
          }
          if (t == 0) {
            // K_b, V_b: their buffers are free once the previous unit's MMAs are done
            if (nu > 0 && !(ok = mbar_wait(bar(B_KVFREE), (nu - 1) & 1))) break;
            mbar_expect_tx(bar(B_KVFULL), 2 * kTile);
            tma_load_3d(sb + kOffK, &tmK, 0, g, b * kBlock, bar(B_KVFULL), pol_kv);
            tma_load_3d(sb + kOffK + 16384, &tmK, 64, g, b * kBlock, bar(B_KVFULL), pol_kv);
            tma_load_3d(sb + kOffV, &tmV, 0, g, b * kBlock, bar(B_KVFULL), pol_kv);
            tma_load_3d(sb + kOffV + 16384, &tmV, 64, g, b * kBlock, bar(B_KVFULL), pol_kv);
          }
          mbar_arrive(bar(B_TFULL0 + slot));
        }
        ++nu;
      }
      if (!ok) atomicOr(&p.hdr->status, kStatusTimeout);
    } else if (warp == 1 && lane == 0) {
      // ------------------------------------------------------------ MMA issue
      constexpr uint32_t idesc_kk = idesc_f16(128, 128, 1, 1, 0, 0);  // A, B K-major
      constexpr uint32_t idesc_ts = idesc_f16(128, 128, 1, 1, 0, 1);  // A from TMEM, B MN-major
      constexpr uint32_t idesc_tt = idesc_f16(128, 128, 1, 1, 1, 1);  // A, B MN-major
      bool ok = true;
      int nu = 0;
      for (int it = 0;; ++it) {
        const int slot = it % kRing, s = it & 1;
        if (!(ok = mbar_wait(bar(B_TFULL0 + slot), (it / kRing) & 1))) break;
        const int cnt = ring[slot].cnt, flags = ring[slot].flags;
        if (cnt == 0) break;
        mbar_arrive(bar(B_TEMPTY0 + slot));
        if ((flags & 1) && !(ok = mbar_wait(bar(B_KVFULL), nu & 1))) break;
        if (!(ok = mbar_wait(bar(B_QFULL0 + s), (it >> 1) & 1))) break;
        // S^T lands in TMEM [0, 128): P^T of the previous tile there has been read by its dV
        if (it > 0 && !(ok = mbar_wait(bar(B_DVDONE), (it - 1) & 1))) break;
        tc_fence_after();
        const uint32_t qa = sb + kOffQ0 + s * kTile, oa = sb + kOffDO0 + s * kTile;
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_f16_ss(tmem, smem_desc(sb + kOffK + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024, 2),
                     smem_desc(qa + (k >> 2) * 1024 + (k & 3) * 32, 16, 2048, 2), idesc_kk, k > 0);
        mma_commit(bar(B_SFULL));
        // dP^T lands in TMEM [128, 256): dQ of the previous tile has been read out
        if (it > 0 && !(ok = mbar_wait(bar(B_DQFREE), (it - 1) & 1))) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_f16_ss(tmem + 128, smem_desc(sb + kOffV + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024, 2),
                     smem_desc(oa + (k >> 2) * 1024 + (k & 3) * 32, 16, 2048, 2), idesc_kk, k > 0);
        mma_commit(bar(B_DPFULL));
        if (!(ok = mbar_wait(bar(B_PREADY), it & 1))) break;
        // the first tile of a unit starts dK / dV afresh: the previous unit's must be out
        if ((flags & 1) && nu > 0 && !(ok = mbar_wait(bar(B_DKVFREE), (nu - 1) & 1))) break;
        tc_fence_after();
        const uint32_t acc0 = (flags & 1) ? 0u : 1u;
        // dV += P^T dO: P^T rows 0-63 at TMEM columns 0-31, rows 64-127 at 64-95 (16 rows per MMA)
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t col = (k < 4 ? 0 : 64) + 8 * (k & 3);
          mma_f16_ts(tmem + 256, tmem + col, smem_desc(oa + k * 4096, 1024, 2048, 2), idesc_ts, k > 0 ? 1u : acc0);
        }
        mma_commit(bar(B_DVDONE));
        // dK += dS^T Q: the dS tile read K-major is dS^T (M = keys, K = rows); formed while dV runs
        if (!(ok = mbar_wait(bar(B_DSREADY), it & 1))) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_f16_ss(tmem + 384, smem_desc(sb + kOffDS + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024, 2),
                     smem_desc(qa + k * 4096, 1024, 2048, 2), idesc_ts, k > 0 ? 1u : acc0);
        mma_commit(bar(B_QFREE0 + s));  // Q / dO of this stage are read no more
        // dQ = dS K_b into TMEM [128, 256): A = dS (M = rows) MN-major, B = K_b MN-major
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_f16_ss(tmem + 128, smem_desc(sb + kOffDS + k * 2048, 16384, 1024, 2),
                     smem_desc(sb + kOffK + k * 2048, 16384, 1024, 2), idesc_tt, k > 0);
        mma_commit(bar(B_MMA2));
        if (flags & 2) {
          mma_commit(bar(B_KVFREE));
          ++nu;
        }
      }
      if (!ok) atomicOr(&p.hdr->status, kStatusTimeout);
    }
  } else if (warp < 12) {
    regs_inc<kRegCompute>();
    // -------------------------------------------------------------- P^T, dS^T
    const int wg = (warp - 4) >> 2;  // rows [64 wg, 64 wg + 64) of each tile
    const uint32_t bar_id = 1 + wg;
    const int kk = 32 * (warp & 3) + lane;  // key of the block = TMEM lane
    const uint32_t tl = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
    const int gtid = tid - 128 - 128 * wg;
    // LSE * log2 e [4 queries][16 heads], then D [4][16], of this half's queries
    const uint32_t ld = smem_u32(ctl + kOffLD + 512 * wg);
    for (int it = 0;; ++it) {
      const int slot = it % kRing;
      bool ok = mbar_wait(bar(B_TFULL0 + slot), (it / kRing) & 1);
      if (!named_bar_and(bar_id, 128, ok)) { atomicOr(&p.hdr->status, kStatusTimeout); break; }
      const BTile& t = ring[slot];
      const int cnt = t.cnt;
      if (cnt == 0) break;
      const int g = t.row / p.nblocks, b = t.row - g * p.nblocks;
      if (gtid < 32) {
        // 64 contiguous bytes per query and array: query jj = gtid / 8, array (gtid / 4) % 2, chunk gtid % 4
        const int jj = gtid >> 3, arr = (gtid >> 2) & 1, j = 4 * wg + jj;
        if (j < cnt) {
          const float* src = (arr ? p.Dv : p.LSE2) + static_cast<size_t>(t.q[j]) * p.Hq + g * kGroup + (gtid & 3) * 4;
          cp_async16(ld + arr * 256 + jj * 64 + (gtid & 3) * 16, src);
        }
      }
      int lim[4];  // keys kk <= lim[jj] are visible to query 4 wg + jj; -1 for rows past cnt
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int j = 4 * wg + jj;
        lim[jj] = j < cnt ? p.Lkv - p.N + t.q[j] - b * kBlock : -1;
      }
      named_bar_sync(bar_id, 128);  // everyone has read the ring entry
      if (gtid == 0) mbar_arrive(bar(B_TEMPTY0 + slot));
      cp_async_wait_all();
      ok = mbar_wait(bar(B_SFULL), it & 1);
      if (!named_bar_and(bar_id, 128, ok)) { atomicOr(&p.hdr->status, kStatusTimeout); break; }
      tc_fence_after();
      // P^T first (it needs S^T only; dP^T is still being computed), to TMEM for dV
      float pv[64];
      {
        uint32_t sv[64];
        tmem_ld32(tl + 64 * wg, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
        tmem_ld32(tl + 64 * wg + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
        tmem_ld_wait();
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const bool vis = kk <= lim[jj];
          float l2[16];
#pragma unroll
          for (int q = 0; q < 4; ++q) lds4(ld + jj * 64 + q * 16, l2[4 * q], l2[4 * q + 1], l2[4 * q + 2], l2[4 * q + 3]);
          uint32_t pp[8];
#pragma unroll
          for (int h = 0; h < 16; h += 2) {
            const float p0 = vis ? ex2(fmaf(__uint_as_float(sv[16 * jj + h]), p.sl2, -l2[h])) : 0.f;
            const float p1 = vis ? ex2(fmaf(__uint_as_float(sv[16 * jj + h + 1]), p.sl2, -l2[h + 1])) : 0.f;
            pv[16 * jj + h] = p0;
            pv[16 * jj + h + 1] = p1;
            pp[h >> 1] = pack_bf16x2(p0, p1);
          }
          tmem_st8(tl + 64 * wg + 8 * jj, pp);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      named_bar_sync(bar_id, 128);
      if (gtid == 0) mbar_arrive(bar(B_PREADY));
      ok = mbar_wait(bar(B_DPFULL), it & 1);
      // dS goes to the tile the previous tile's dQ was staged in: its store must have read it
      if (it > 0) ok = mbar_wait(bar(B_DSFREE), (it - 1) & 1) && ok;
      if (!named_bar_and(bar_id, 128, ok)) { atomicOr(&p.hdr->status, kStatusTimeout); break; }
      tc_fence_after();
#pragma unroll
      for (int hv = 0; hv < 2; ++hv) {
        uint32_t dv[32];  // dP^T of rows 32 hv .. 32 hv + 31 of this half
        tmem_ld32(tl + 128 + 64 * wg + 32 * hv, dv);
        tmem_ld_wait();
#pragma unroll
        for (int j2 = 0; j2 < 2; ++j2) {
          const int jj = 2 * hv + j2;
          const bool vis = kk <= lim[jj];
          float dd0[16];
#pragma unroll
          for (int q = 0; q < 4; ++q)
            lds4(ld + 256 + jj * 64 + q * 16, dd0[4 * q], dd0[4 * q + 1], dd0[4 * q + 2], dd0[4 * q + 3]);
          uint32_t dd[8];
#pragma unroll
          for (int h = 0; h < 16; h += 2)
            dd[h >> 1] = vis ? pack_bf16x2(pv[16 * jj + h] * (__uint_as_float(dv[16 * j2 + h]) - dd0[h]),
                                           pv[16 * jj + h + 1] * (__uint_as_float(dv[16 * j2 + h + 1]) - dd0[h + 1]))
                             : 0u;
          // dS [rows][keys] for dQ (and, read K-major, dS^T for dK): row kk of this half's tile holds the 64 rows' values of key kk
          uint8_t* dsrow = smem + kOffDS + wg * 16384 + kk * 128;
          *reinterpret_cast<uint4*>(dsrow + (((2 * jj) ^ (kk & 7)) << 4)) = make_uint4(dd[0], dd[1], dd[2], dd[3]);
          *reinterpret_cast<uint4*>(dsrow + (((2 * jj + 1) ^ (kk & 7)) << 4)) = make_uint4(dd[4], dd[5], dd[6], dd[7]);
        }
      }
      tc_fence_before();
      fence_proxy_async_smem();
      named_bar_sync(bar_id, 128);
      if (gtid == 0) mbar_arrive(bar(B_DSREADY));
    }
  } else {
    regs_dec<kRegEvac>();
    // -------------------------------------------------------------- evacuation
    const uint32_t bar_id = 3;
    const int rr = 32 * (warp & 3) + lane;  // TMEM lane: tile row for dQ, key for dK / dV
    const uint32_t tl = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
    const bool elected = tid == 384;
    const uint64_t pol_st = policy_evict_normal();
    if (elected) { tma_prefetch_desc(&tmP128); tma_prefetch_desc(&tmP16); }
    int nu = 0;
    for (int it = 0;; ++it) {
      const int slot = it % kRing;
      bool ok = mbar_wait(bar(B_TFULL0 + slot), (it / kRing) & 1);
      if (!named_bar_and(bar_id, 128, ok)) { atomicOr(&p.hdr->status, kStatusTimeout); break; }
      const int cnt = ring[slot].cnt, e0 = ring[slot].e0, flags = ring[slot].flags, uid = ring[slot].uid;
      if (cnt == 0) break;
      ok = mbar_wait(bar(B_MMA2), it & 1);
      if (!named_bar_and(bar_id, 128, ok)) { atomicOr(&p.hdr->status, kStatusTimeout); break; }
      if (elected) mbar_arrive(bar(B_TEMPTY0 + slot));
      tc_fence_after();
      // dQ (TMEM lane = tile row) -> bf16 -> the dS tile (dQ, its last reader, is done), in
      // the 128-byte-swizzled layout of the partial rows' tensor map -> TMA store
#pragma unroll
      for (int qt = 0; qt < 4; ++qt) {
        uint32_t v[32];
        tmem_ld32(tl + 128 + 32 * qt, v);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int ch = 4 * qt + c;  // 8-column chunk 0..15
          const uint32_t off = (ch >> 3) * 16384 + rr * 128 + (((ch & 7) ^ (rr & 7)) << 4);
          *reinterpret_cast<uint4*>(smem + kOffDS + off) =
              make_uint4(pack_bf16x2(__uint_as_float(v[8 * c + 0]), __uint_as_float(v[8 * c + 1])),
                         pack_bf16x2(__uint_as_float(v[8 * c + 2]), __uint_as_float(v[8 * c + 3])),
                         pack_bf16x2(__uint_as_float(v[8 * c + 4]), __uint_as_float(v[8 * c + 5])),
                         pack_bf16x2(__uint_as_float(v[8 * c + 6]), __uint_as_float(v[8 * c + 7])));
        }
      }
      tc_fence_before();
      fence_proxy_async_smem();
      named_bar_sync(bar_id, 128);
      if (elected) {
        mbar_arrive(bar(B_DQFREE));  // dQ is out of TMEM: the next tile's dP^T may overwrite it
        const uint32_t src = sb + kOffDS;
        if (cnt == kTileQ) {
          tma_store_2d(&tmP128, 0, e0 * kGroup, src, pol_st);
          tma_store_2d(&tmP128, 64, e0 * kGroup, src + 16384, pol_st);
        } else {
          for (int q = 0; q < cnt; ++q) {
            tma_store_2d(&tmP16, 0, (e0 + q) * kGroup, src + q * 2048, pol_st);
            tma_store_2d(&tmP16, 64, (e0 + q) * kGroup, src + 16384 + q * 2048, pol_st);
          }
        }
        bulk_commit();
        bulk_wait_read0();
        mbar_arrive(bar(B_DSFREE));  // the staging has been read: the next dS may be written
      }
      if (flags & 2) {
        // the unit's dK (columns 384..) and dV (256..), thread = key -> fp32 partials
        float* dk = p.dkv + static_cast<size_t>(uid) * 2 * kBlock * kHeadDim;
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t v[64];
            const uint32_t ta = tl + (m == 0 ? 384 : 256) + 64 * half;
            tmem_ld32(ta, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
            tmem_ld32(ta + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
            tmem_ld_wait();
            float4* d4 = reinterpret_cast<float4*>(dk + (static_cast<size_t>(m) * kBlock + rr) * kHeadDim + 64 * half);
#pragma unroll
            for (int q = 0; q < 16; ++q)
              d4[q] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                  __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
          }
        tc_fence_before();
        named_bar_sync(bar_id, 128);
        if (elected) mbar_arrive(bar(B_DKVFREE));
        ++nu;
      }
    }
    if (elected) bulk_wait_all0();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// LSE[i, h] * log2 e and D[i, h] = dO[i, h, :] . O[i, h, :] in fp32: 16 threads per row
// (8 elements each), two rows per warp; the loop bound is warp-uniform so every lane
// joins the shuffles.
__global__ void __launch_bounds__(256) bwd_prep_kernel(const uint4* __restrict__ O, const uint4* __restrict__ dO,
                                                       const float* __restrict__ LSE, float* __restrict__ LSE2,
                                                       float* __restrict__ Dv, int64_t rows) {
  const int sub = threadIdx.x & 15;
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t r0 = warp0 * 2; r0 < rows; r0 += nwarps * 2) {
    const int64_t r = r0 + ((threadIdx.x >> 4) & 1);
    float s = 0.f;
    if (r < rows) {
      const uint4 a = __ldg(O + r * 16 + sub), c = __ldg(dO + r * 16 + sub);
      const uint32_t x[4] = {a.x, a.y, a.z, a.w}, y[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        s = fmaf(__uint_as_float(x[q] << 16), __uint_as_float(y[q] << 16), s);
        s = fmaf(__uint_as_float(x[q] & 0xFFFF0000u), __uint_as_float(y[q] & 0xFFFF0000u), s);
      }
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (sub == 0 && r < rows) {
      LSE2[r] = __ldg(LSE + r) * 1.4426950408889634f;
      Dv[r] = s;
    }
  }
}

// Units of at most kUnitEntries consecutive entries per row, listed row by row; unit_off[r]
// is the first unit of row r (exclusive prefix), unit_off[R] the total.  One CTA.
__global__ void __launch_bounds__(1024) bwd_units_kernel(const int32_t* __restrict__ counts,
                                                         const int32_t* __restrict__ offsets, int R, int4* units,
                                                         int32_t* unit_off) {
  __shared__ int32_t warp_sums[32];
  __shared__ int32_t carry;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  for (int base = 0; base < R; base += 1024) {
    const int r = base + threadIdx.x;
    const int nu = r < R ? (counts[r] + kUnitEntries - 1) / kUnitEntries : 0;
    int x = nu;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[w] = x;
    __syncthreads();
    if (w == 0) {
      int s = warp_sums[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, s, o);
        if (lane >= o) s += y;
      }
      warp_sums[lane] = s;
    }
    __syncthreads();
    const int excl = carry + (w > 0 ? warp_sums[w - 1] : 0) + x - nu;
    if (r < R) {
      unit_off[r] = excl;
      const int c = counts[r], f = offsets[r];
      for (int u = 0; u < nu; ++u)
        units[excl + u] = make_int4(r, f + u * kUnitEntries, min(kUnitEntries, c - u * kUnitEntries), 0);
    }
    __syncthreads();
    if (threadIdx.x == 1023) carry = excl + nu;
    __syncthreads();
  }
  if (threadIdx.x == 0) unit_off[R] = carry;
}

// dK, dV rows of one (row, 8 keys) per CTA: thread = (key, 4 columns); sums the row's units
// in order.  Blocks with no unit get zeros.
__global__ void __launch_bounds__(256) bwd_reduce_kernel(const float4* __restrict__ dkv,
                                                         const int32_t* __restrict__ unit_off, int R, int nblocks,
                                                         int Hkv, float scale, __nv_bfloat16* dK, __nv_bfloat16* dV) {
  const int key8 = blockIdx.x & 15, r = blockIdx.x >> 4;
  if (r >= R) return;
  const int g = r / nblocks, b = r - g * nblocks;
  const int kk = key8 * 8 + (threadIdx.x >> 5), c4 = threadIdx.x & 31;
  const int u0 = unit_off[r], u1 = unit_off[r + 1];
  float4 ak = make_float4(0.f, 0.f, 0.f, 0.f), av = ak;
  for (int u = u0; u < u1; ++u) {
    const float4* base = dkv + static_cast<size_t>(u) * 2 * kBlock * 32;
    const float4 x = __ldg(base + kk * 32 + c4), y = __ldg(base + (kBlock + kk) * 32 + c4);
    ak.x += x.x; ak.y += x.y; ak.z += x.z; ak.w += x.w;
    av.x += y.x; av.y += y.y; av.z += y.z; av.w += y.w;
  }
  const size_t o = ((static_cast<size_t>(b) * kBlock + kk) * Hkv + g) * kHeadDim + c4 * 4;
  uint2 wk, wv;
  wk.x = pack_bf16x2(ak.x * scale, ak.y * scale);
  wk.y = pack_bf16x2(ak.z * scale, ak.w * scale);
  wv.x = pack_bf16x2(av.x, av.y);
  wv.y = pack_bf16x2(av.z, av.w);
  *reinterpret_cast<uint2*>(dK + o) = wk;
  *reinterpret_cast<uint2*>(dV + o) = wv;
}

// dQ[i, g heads] = scale * sum over the (i, g) entries of their partial rows, in list order.
// Thread (head h, 8 columns c) of a 256-thread CTA per (i, g) unit.
__global__ void __launch_bounds__(256) bwd_dq_kernel(const int32_t* __restrict__ cmap, const uint4* __restrict__ part,
                                                     int N, int Hkv, int topK, int Hq, float scale,
                                                     __nv_bfloat16* __restrict__ dQ) {
  const int h = threadIdx.x >> 4, c = threadIdx.x & 15;
  const int64_t nunit = static_cast<int64_t>(N) * Hkv;
  for (int64_t u = blockIdx.x; u < nunit; u += gridDim.x) {
    const int32_t* cm = cmap + u * topK;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int k = 0; k < topK; ++k) {
      const int pos = __ldg(cm + k);
      if (pos < 0) continue;
      const uint4 v = __ldg(part + (static_cast<int64_t>(pos) * kGroup + h) * 16 + c);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc[2 * q] += __uint_as_float(w[q] << 16);
        acc[2 * q + 1] += __uint_as_float(w[q] & 0xFFFF0000u);
      }
    }
    const int64_t i = u / Hkv, g = u % Hkv;
    uint4 out;
    out.x = pack_bf16x2(acc[0] * scale, acc[1] * scale);
    out.y = pack_bf16x2(acc[2] * scale, acc[3] * scale);
    out.z = pack_bf16x2(acc[4] * scale, acc[5] * scale);
    out.w = pack_bf16x2(acc[6] * scale, acc[7] * scale);
    reinterpret_cast<uint4*>(dQ)[(i * Hq + g * kGroup + h) * 16 + c] = out;
  }
}

}  // namespace

size_t bwd_workspace_bytes(const msa_schedule* s) {
  const int64_t units = bwd_unit_capacity(s);
  size_t b = 0;
  b += 2 * ((static_cast<size_t>(s->N) * s->Hkv * kGroup * sizeof(float) + 255) / 256 * 256);  // LSE log2 e, D
  b += (static_cast<size_t>(units) * sizeof(int4) + 255) / 256 * 256;                     // units
  b += (static_cast<size_t>(s->R + 1) * sizeof(int32_t) + 255) / 256 * 256;               // unit_off
  b += 256;                                                                                // claim counter
  b += static_cast<size_t>(units) * 2 * kBlock * kHeadDim * sizeof(float);                // dK/dV partials
  return b;
}

int64_t bwd_unit_capacity(const msa_schedule* s) {
  const int64_t nonempty = s->R < s->cap_entries ? s->R : s->cap_entries;
  return nonempty + (s->cap_entries + kUnitEntries - 1) / kUnitEntries;
}

cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t st) {
  const msa_schedule* s = a.s;
  char* ws = static_cast<char*>(a.workspace);
  const int64_t cap_units = bwd_unit_capacity(s);
  auto take = [&](size_t bytes) {
    char* p = ws;
    ws += (bytes + 255) / 256 * 256;
    return p;
  };
  const int64_t qrows = static_cast<int64_t>(s->N) * a.Hq;
  float* LSE2 = reinterpret_cast<float*>(take(static_cast<size_t>(qrows) * sizeof(float)));
  float* Dv = reinterpret_cast<float*>(take(static_cast<size_t>(qrows) * sizeof(float)));
  int4* units = reinterpret_cast<int4*>(take(static_cast<size_t>(cap_units) * sizeof(int4)));
  int32_t* unit_off = reinterpret_cast<int32_t*>(take(static_cast<size_t>(s->R + 1) * sizeof(int32_t)));
  int32_t* counter = reinterpret_cast<int32_t*>(take(256));
  float* dkv = reinterpret_cast<float*>(ws);

  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaError_t e;
  {
    int64_t grid = (qrows * 16 + 255) / 256;
    if (grid > static_cast<int64_t>(sms) * 32) grid = static_cast<int64_t>(sms) * 32;
    bwd_prep_kernel<<<static_cast<int>(grid), 256, 0, st>>>(static_cast<const uint4*>(a.O),
                                                            static_cast<const uint4*>(a.dO), a.LSE, LSE2, Dv,
                                                            qrows);
    if ((e = cudaGetLastError())) return e;
  }
  bwd_units_kernel<<<1, 1024, 0, st>>>(s->d.counts, s->d.offsets, s->R, units, unit_off);
  if ((e = cudaGetLastError())) return e;
  if ((e = cudaMemsetAsync(counter, 0, sizeof(int32_t), st))) return e;

  CUtensorMap tmK, tmV, tmQ, tmDO, tmP128, tmP16;
  {
    // dQ partial rows [E * 16][128] bf16: a full tile's 128 rows, or 16 rows per entry
    const uint64_t dims[2] = {kHeadDim, static_cast<uint64_t>(s->cap_entries) * kGroup};
    const uint64_t strides[1] = {kHeadDim * 2};
    const uint32_t box128[2] = {64, 128}, box16[2] = {64, 16};
    if (!encode_tmap(&tmP128, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, s->partial, dims, strides, box128,
                     CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
    if (!encode_tmap(&tmP16, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, s->partial, dims, strides, box16,
                     CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  {
    // Q, dO [N][Hq][128] viewed as (64 elements of a D half, head within 8, D half, group of
    // 8 heads, query): one box = the 16 heads of one query's GQA group, 4 KB, landing as
    // [8-head group][D half][8 heads][128 B]
    const uint64_t row = kHeadDim * 2;
    const uint64_t dims[5] = {64, 8, 2, static_cast<uint64_t>(a.Hq) / 8, static_cast<uint64_t>(s->N)};
    const uint64_t strides[4] = {row, 128, 8 * row, static_cast<uint64_t>(a.Hq) * row};
    const uint32_t box[5] = {64, 8, 2, 2, 1};
    if (!encode_tmap(&tmQ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, a.Q, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
    if (!encode_tmap(&tmDO, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, a.dO, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[3] = {kHeadDim, static_cast<uint64_t>(s->Hkv), static_cast<uint64_t>(a.Lkv)};
    const uint64_t strides[2] = {kHeadDim * 2, static_cast<uint64_t>(s->Hkv) * kHeadDim * 2};
    const uint32_t box[3] = {64u, 1, kBlock};
    if (!encode_tmap(&tmK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.K, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
    if (!encode_tmap(&tmV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.V, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  BwdParams p;
  p.LSE2 = LSE2;
  p.Dv = Dv;
  p.units = units;
  p.qlist = s->d.qlist;
  p.counter = counter;
  p.nunits = unit_off + s->R;
  p.dkv = dkv;
  p.hdr = s->d.hdr;
  p.N = s->N;
  p.Lkv = a.Lkv;
  p.Hq = a.Hq;
  p.nblocks = s->nblocks;
  p.R = s->R;
  p.cap_e = s->cap_entries;
  p.sl2 = a.scale * 1.4426950408889634f;
  static std::atomic<uint64_t> attr_done{0};
  if ((e = set_smem_limit(bwd_kv_kernel, kSmemBytes, attr_done))) return e;
  if (a.ev[0] && (e = cudaEventRecord(a.ev[0], st))) return e;
  bwd_kv_kernel<<<a.num_ctas, kThreads, kSmemBytes, st>>>(tmK, tmV, tmQ, tmDO, tmP128, tmP16, p);
  if ((e = cudaGetLastError())) return e;
  if (a.ev[1] && (e = cudaEventRecord(a.ev[1], st))) return e;
  bwd_reduce_kernel<<<s->R * 16, 256, 0, st>>>(reinterpret_cast<const float4*>(dkv), unit_off, s->R, s->nblocks,
                                                s->Hkv, a.scale, static_cast<__nv_bfloat16*>(a.dK),
                                                static_cast<__nv_bfloat16*>(a.dV));
  if ((e = cudaGetLastError())) return e;
  {
    const int64_t nunit = static_cast<int64_t>(s->N) * s->Hkv;
    int64_t grid = static_cast<int64_t>(sms) * 16;
    if (grid > nunit) grid = nunit;
    bwd_dq_kernel<<<static_cast<int>(grid), 256, 0, st>>>(s->d.cmap, static_cast<const uint4*>(s->partial), s->N,
                                                          s->Hkv, s->topK, a.Hq, a.scale,
                                                          static_cast<__nv_bfloat16*>(a.dQ));
    if ((e = cudaGetLastError())) return e;
  }
  if (a.ev[2] && (e = cudaEventRecord(a.ev[2], st))) return e;
  return cudaSuccess;
}

}  // namespace msa
