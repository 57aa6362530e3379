// KV-outer (KV-stationary) attention kernel, bf16, tcgen05 + TMA, persistent.
//
// "Kernel optimization for MiniMax M3 on NVIDIA Blackwell" (kernel stages): a CTA
// owns one KV block at a time and attends every query that chose it; because each
// tile sees a single block there is exactly one softmax step and no rescale of a
// running output; partial outputs are written tile-ordered and contiguous, and the
// combine kernel gathers them.  "Sparse Attention", Chapter 5: the KV-centric kernel
// writes, per query and head, a partial output and a log-sum-exp.
//
// Work unit (tile): up to 8 consecutive CSR entries of one (group g, block b) row,
// i.e. 8 queries x 16 heads = 128 MMA rows (the head-packed "box" of one query is
// 16 rows).  Tiles come from the schedule's work list, window by window; inside a
// window, CTA c takes the c-th contiguous slice.
//
// Warp roles (384 threads, one CTA per SM):
//   warp 0      producer: TMA of the Q boxes of each tile (two 64-column halves per
//               query) and of K_b / V_b whenever the row changes
//   warp 1      MMA issuer: S[s] = Q K^T (tcgen05, smem x smem), then
//               O[s] = P V with P read from TMEM (it overwrites S[s] in place)
//   warp 2      TMEM allocation (512 columns: S[0], S[1], O[0], O[1])
//   warps 4-7   group 0: softmax + epilogue of even tiles (stage 0)
//   warps 8-11  group 1: softmax + epilogue of odd tiles  (stage 1)
// Each thread of a group owns one MMA row (TMEM lane) through softmax and epilogue,
// so 1/l never leaves its register.  The epilogue normalises, rounds to bf16,
// writes a 128-byte-swizzled staging tile and one elected thread stores it with TMA
// at partial rows [16*first, 16*(first+count)).
//
// Partial layout: bf16 [E*16, 128] (row = 16*CSR position + head-in-group) and
// base-2 log-sum-exp fp32 [E*16].
#include <cfloat>

#include "msa_internal.h"
#include "ptx.cuh"

namespace msa {
namespace {

constexpr int kThreads = 384;
constexpr uint32_t kQBytes = 128 * 128 * 2;  // one Q tile (two 16 KB halves)
constexpr uint32_t kKVBytes = 128 * 128 * 2;
constexpr uint32_t kOffQ0 = 0, kOffQ1 = 32768, kOffK = 65536, kOffV = 98304, kOffSt0 = 131072,
                   kOffSt1 = 163840, kOffCtl = 196608;
constexpr uint32_t kSmemBytes = kOffCtl + 256 + 1024;  // + alignment slack

// barrier slots (8 bytes each) in the control area
enum {
  B_QFULL0 = 0, B_QFULL1, B_QFREE0, B_QFREE1, B_KFULL, B_KFREE, B_VFULL, B_VFREE,
  B_SFULL0, B_SFULL1, B_PFULL0, B_PFULL1, B_PVDONE0, B_PVDONE1, B_COUNT
};

struct KvParams {
  const int4* tiles;
  const int32_t* window_tiles;
  const int32_t* qlist;
  SchedHeader* hdr;
  float* plse;
  int nW, N, Lkv, nblocks;
  float sl2;  // scale * log2(e)
  int force_path;
};

// This CTA's tiles, window by window: in window w (tiles [a, b)) it takes
// [a + n*c/P, a + n*(c+1)/P).
struct TileIter {
  const int32_t* wt;
  int nW, cta, P, w;
  int64_t t, tend;
  __device__ void init(const int32_t* wt_, int nW_, int cta_, int P_) {
    wt = wt_; nW = nW_; cta = cta_; P = P_; w = -1; t = tend = 0;
  }
  __device__ bool next(int* ti) {
    while (t >= tend) {
      if (++w >= nW) return false;
      const int64_t a = wt[w], n = wt[w + 1] - a;
      t = a + n * cta / P;
      tend = a + n * (cta + 1) / P;
    }
    *ti = static_cast<int>(t++);
    return true;
  }
};

__device__ __forceinline__ void flag_timeout(SchedHeader* hdr) { atomicOr(&hdr->status, kStatusTimeout); }

__global__ void __launch_bounds__(kThreads, 1)
kv_outer_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmP128,
                const __grid_constant__ CUtensorMap tmP16, const KvParams p) {
  const int path = p.force_path ? p.force_path : p.hdr->path;
  if (path != kPathKvOuter) return;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw_u & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sb = raw_u + pad;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffCtl);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffCtl + 8 * B_COUNT);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // zero the Q stages once so rows of a partly filled tile never hold NaN patterns
  for (uint32_t o = tid * 16; o < 2 * kQBytes; o += kThreads * 16)
    *reinterpret_cast<uint4*>(smem + kOffQ0 + o) = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();

  if (tid == 0) {
    mbar_init(bar(B_QFULL0), 1); mbar_init(bar(B_QFULL1), 1);
    mbar_init(bar(B_QFREE0), 1); mbar_init(bar(B_QFREE1), 1);
    mbar_init(bar(B_KFULL), 1);  mbar_init(bar(B_KFREE), 1);
    mbar_init(bar(B_VFULL), 1);  mbar_init(bar(B_VFREE), 1);
    mbar_init(bar(B_SFULL0), 1); mbar_init(bar(B_SFULL1), 1);
    mbar_init(bar(B_PFULL0), 128); mbar_init(bar(B_PFULL1), 128);
    mbar_init(bar(B_PVDONE0), 1); mbar_init(bar(B_PVDONE1), 1);
    mbar_fence_init();
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  TileIter iter;
  iter.init(p.window_tiles, p.nW, blockIdx.x, gridDim.x);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ); tma_prefetch_desc(&tmK); tma_prefetch_desc(&tmV);
      const uint64_t pol_q = policy_evict_normal(), pol_kv = policy_evict_last();
      int ti, it = 0, prev_row = -1, nk = 0;
      while (iter.next(&ti)) {
        const int4 tl = p.tiles[ti];
        const int s = it & 1;
        const int g = tl.x / p.nblocks, b = tl.x - g * p.nblocks;
        if (!mbar_wait(bar(B_QFREE0 + s), ((it >> 1) & 1) ^ 1)) { flag_timeout(p.hdr); break; }
        mbar_expect_tx(bar(B_QFULL0 + s), static_cast<uint32_t>(tl.z) * 4096u);
        const uint32_t dq = sb + (s ? kOffQ1 : kOffQ0);
        for (int j = 0; j < tl.z; ++j) {
          const int q = p.qlist[tl.y + j];
          tma_load_3d(dq + j * 2048, &tmQ, 0, g * kGroup, q, bar(B_QFULL0 + s), pol_q);
          tma_load_3d(dq + 16384 + j * 2048, &tmQ, 64, g * kGroup, q, bar(B_QFULL0 + s), pol_q);
        }
        if (tl.x != prev_row) {
          if (!mbar_wait(bar(B_KFREE), (nk & 1) ^ 1)) { flag_timeout(p.hdr); break; }
          mbar_expect_tx(bar(B_KFULL), kKVBytes);
          tma_load_3d(sb + kOffK, &tmK, 0, g, b * kBlock, bar(B_KFULL), pol_kv);
          tma_load_3d(sb + kOffK + 16384, &tmK, 64, g, b * kBlock, bar(B_KFULL), pol_kv);
          if (!mbar_wait(bar(B_VFREE), (nk & 1) ^ 1)) { flag_timeout(p.hdr); break; }
          mbar_expect_tx(bar(B_VFULL), kKVBytes);
          tma_load_3d(sb + kOffV, &tmV, 0, g, b * kBlock, bar(B_VFULL), pol_kv);
          tma_load_3d(sb + kOffV + 16384, &tmV, 64, g, b * kBlock, bar(B_VFULL), pol_kv);
          ++nk;
          prev_row = tl.x;
        }
        ++it;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_f16(128, 128, 1, 1, 0, 0);
      constexpr uint32_t idesc_pv = idesc_f16(128, 128, 1, 1, 0, 1);
      int ti, ti2;
      bool have = iter.next(&ti);
      int4 tl = have ? p.tiles[ti] : make_int4(0, 0, 0, 0);
      int it = 0, prev_row = -1, nk = 0, nv = 0;
      bool pv_pending = false, pv_new_row = false, pv_last = false;
      bool ok = true;
      while (ok && (have || pv_pending)) {
        bool new_row = false, last = false, have2 = false;
        int4 tl2 = make_int4(0, 0, 0, 0);
        if (have) {
          have2 = iter.next(&ti2);
          if (have2) tl2 = p.tiles[ti2];
          const int s = it & 1;
          // S[s] / P[s] is reused: PV of tile it-2 must have consumed P
          if (it >= 2 && !mbar_wait(bar(B_PVDONE0 + s), ((it - 2) >> 1) & 1)) { ok = false; break; }
          new_row = tl.x != prev_row;
          last = !have2 || tl2.x != tl.x;
          if (new_row) {
            if (!mbar_wait(bar(B_KFULL), nk & 1)) { ok = false; break; }
            ++nk;
          }
          if (!mbar_wait(bar(B_QFULL0 + s), (it >> 1) & 1)) { ok = false; break; }
          tc_fence_after();
          const uint32_t qa = sb + (s ? kOffQ1 : kOffQ0), ka = sb + kOffK;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
            mma_f16_ss(tmem + s * 128, smem_desc(qa + off, 16, 1024, 2), smem_desc(ka + off, 16, 1024, 2), idesc_qk,
                       k > 0);
          }
          mma_commit(bar(B_SFULL0 + s));
          mma_commit(bar(B_QFREE0 + s));
          if (last) mma_commit(bar(B_KFREE));
        }
        if (pv_pending) {
          const int u = it - 1, s = u & 1;
          if (pv_new_row) {
            if (!mbar_wait(bar(B_VFULL), nv & 1)) { ok = false; break; }
            ++nv;
          }
          if (!mbar_wait(bar(B_PFULL0 + s), (u >> 1) & 1)) { ok = false; break; }
          tc_fence_after();
          const uint32_t va = sb + kOffV;
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma_f16_ts(tmem + 256 + s * 128, tmem + s * 128 + k * 8, smem_desc(va + k * 2048, 16384, 1024, 2),
                       idesc_pv, k > 0);
          mma_commit(bar(B_PVDONE0 + s));
          if (pv_last) mma_commit(bar(B_VFREE));
        }
        pv_pending = have;
        pv_new_row = new_row;
        pv_last = last;
        if (have) prev_row = tl.x;
        have = have2;
        tl = tl2;
        ti = ti2;
        ++it;
      }
      if (!ok) flag_timeout(p.hdr);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax + epilogue
    const int wg = (warp - 4) >> 2;  // 0 or 1: stage handled
    const uint32_t bar_id = 1 + wg;
    const int row = 32 * (warp & 3) + lane;
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const uint32_t tS = tmem + lane_base + wg * 128;
    const uint32_t tO = tmem + lane_base + 256 + wg * 128;
    const bool elected = (tid == 128 + wg * 128);
    const uint32_t st_off = wg ? kOffSt1 : kOffSt0;
    uint8_t* stage = smem + st_off;
    const uint64_t pol_st = policy_evict_first();
    if (elected) { tma_prefetch_desc(&tmP128); tma_prefetch_desc(&tmP16); }
    int ti, it = 0;
    bool stored_before = false;
    while (iter.next(&ti)) {
      if ((it & 1) != wg) { ++it; continue; }
      const int4 tl = p.tiles[ti];
      const int j = row >> 4;
      const bool valid = j < tl.z;
      const int qi = valid ? p.qlist[tl.y + j] : 0;
      const int b = tl.x % p.nblocks;
      const int lim = (p.Lkv - p.N + qi) - b * kBlock;  // keys c <= lim visible

      bool ok = mbar_wait(bar(B_SFULL0 + wg), (it >> 1) & 1);
      if (!named_bar_and(bar_id, 128, ok)) { flag_timeout(p.hdr); break; }
      tc_fence_after();

      // pass 1: row maximum of s * scale * log2(e) over visible keys
      float m2 = -FLT_MAX;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld32(tS + c * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e)
          if (c * 32 + e <= lim) m2 = fmaxf(m2, __uint_as_float(v[e]) * p.sl2);
      }
      // pass 2: P = 2^(s*sl2 - m2), row sum, P as bf16 pairs over the S columns
      float l = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32], pk[16];
        tmem_ld32(tS + c * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float p0 = (c * 32 + e <= lim) ? ex2(fmaf(__uint_as_float(v[e]), p.sl2, -m2)) : 0.f;
          const float p1 = (c * 32 + e + 1 <= lim) ? ex2(fmaf(__uint_as_float(v[e + 1]), p.sl2, -m2)) : 0.f;
          l += p0 + p1;
          pk[e >> 1] = pack_bf16x2(p0, p1);
        }
        tmem_st16(tS + c * 16, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(B_PFULL0 + wg));
      if (valid) p.plse[static_cast<size_t>(tl.y) * kGroup + row] = m2 + lg2(l);
      const float linv = 1.f / l;

      // epilogue: wait for O = P V, normalise, bf16, swizzled staging, TMA store
      ok = mbar_wait(bar(B_PVDONE0 + wg), (it >> 1) & 1);
      if (elected && stored_before) bulk_wait_read0();
      if (!named_bar_and(bar_id, 128, ok)) { flag_timeout(p.hdr); break; }
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld32(tO + c * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int ch = c * 4 + q;
          uint4 w;
          w.x = pack_bf16x2(__uint_as_float(v[q * 8 + 0]) * linv, __uint_as_float(v[q * 8 + 1]) * linv);
          w.y = pack_bf16x2(__uint_as_float(v[q * 8 + 2]) * linv, __uint_as_float(v[q * 8 + 3]) * linv);
          w.z = pack_bf16x2(__uint_as_float(v[q * 8 + 4]) * linv, __uint_as_float(v[q * 8 + 5]) * linv);
          w.w = pack_bf16x2(__uint_as_float(v[q * 8 + 6]) * linv, __uint_as_float(v[q * 8 + 7]) * linv);
          const uint32_t off = (ch >> 3) * 16384 + row * 128 + (((ch & 7) ^ (row & 7)) << 4);
          *reinterpret_cast<uint4*>(stage + off) = w;
        }
      }
      tc_fence_before();
      fence_proxy_async_smem();
      named_bar_sync(bar_id, 128);
      if (elected) {
        const uint32_t src = sb + st_off;
        if (tl.z == kTileQ) {
          tma_store_2d(&tmP128, 0, tl.y * kGroup, src, pol_st);
          tma_store_2d(&tmP128, 64, tl.y * kGroup, src + 16384, pol_st);
        } else {
          for (int q = 0; q < tl.z; ++q) {
            tma_store_2d(&tmP16, 0, (tl.y + q) * kGroup, src + q * 2048, pol_st);
            tma_store_2d(&tmP16, 64, (tl.y + q) * kGroup, src + 16384 + q * 2048, pol_st);
          }
        }
        bulk_commit();
      }
      stored_before = true;
      ++it;
    }
    if (elected) bulk_wait_all0();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t launch_kv_outer(const KvOuterArgs& a, cudaStream_t st) {
  const msa_schedule* s = a.s;
  CUtensorMap tmQ, tmK, tmV, tmP128, tmP16;
  {
    const uint64_t dims[3] = {kHeadDim, static_cast<uint64_t>(a.Hq), static_cast<uint64_t>(s->N)};
    const uint64_t strides[2] = {kHeadDim * 2, static_cast<uint64_t>(a.Hq) * kHeadDim * 2};
    const uint32_t box[3] = {64, kGroup, 1};
    if (!encode_tmap(&tmQ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.Q, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[3] = {kHeadDim, static_cast<uint64_t>(s->Hkv), static_cast<uint64_t>(a.Lkv)};
    const uint64_t strides[2] = {kHeadDim * 2, static_cast<uint64_t>(s->Hkv) * kHeadDim * 2};
    const uint32_t box[3] = {64, 1, kBlock};
    if (!encode_tmap(&tmK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.K, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
    if (!encode_tmap(&tmV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.V, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  {
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
  KvParams p;
  p.tiles = s->d.tiles;
  p.window_tiles = s->d.window_tiles;
  p.qlist = s->d.qlist;
  p.hdr = s->d.hdr;
  p.plse = s->plse;
  p.nW = s->nW;
  p.N = s->N;
  p.Lkv = a.Lkv;
  p.nblocks = s->nblocks;
  p.sl2 = a.scale * 1.4426950408889634f;
  p.force_path = a.force_path;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kv_outer_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  kv_outer_kernel<<<a.num_ctas, kThreads, kSmemBytes, st>>>(tmQ, tmK, tmV, tmP128, tmP16, p);
  return cudaGetLastError();
}

}  // namespace msa
