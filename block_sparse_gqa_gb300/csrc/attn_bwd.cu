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
// bwd_kv_kernel, one CTA of 256 threads per SM (persistent; units claimed with an
// atomicAdd).  Shared memory (bf16 128 x 128 tiles, two 64-column halves with the
// 128-byte swizzle): K_b, V_b (TMA), Q and dO of the tile (cp.async gathers), P and
// dS (written by the threads).  The same physical tile layout is K-major for a matrix
// and MN-major for its transpose, so P and dS serve both as P^T / dS^T (M = keys) and
// as dS (M = rows); K_b is read K-major for S and MN-major for dQ.  TMEM (512
// columns): S [0, 128) (later dQ), dP [128, 256), dV [256, 384), dK [384, 512).
// Per tile: gather -> S, dP MMAs -> P, dS -> dV, dK, dQ MMAs -> dQ rows to global.
// Thread (warp w, lane) owns MMA row / TMEM lane 32 (w % 4) + lane and the column
// half w / 4.
#include <cuda_bf16.h>

#include "msa_internal.h"
#include "ptx.cuh"

namespace msa {
namespace {

constexpr int kThreads = 256;
constexpr uint32_t kTile = 32768;  // bf16 128 x 128
constexpr uint32_t kOffK = 0, kOffV = kTile, kOffQ = 2 * kTile, kOffDO = 3 * kTile, kOffP = 4 * kTile,
                   kOffDS = 5 * kTile, kOffCtl = 6 * kTile;
constexpr uint32_t kSmemBytes = kOffCtl + 1024 + 1024;  // + control + alignment slack
enum { B_KV = 0, B_MMA1 = 1, B_MMA2 = 2 };

struct BwdParams {
  const uint8_t* Q;
  const uint8_t* dO;
  const float* LSE;
  const float* Dv;
  const int4* units;
  const int32_t* qlist;
  int32_t* counter;
  const int32_t* nunits;
  __nv_bfloat16* dq_part;  // [E * 16, 128]
  float* dkv;              // [units][2][128][128]: dK then dV
  SchedHeader* hdr;
  int N, Lkv, Hq, nblocks;
  float sl2;  // scale * log2(e)
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__global__ void __launch_bounds__(kThreads, 1)
bwd_kv_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, const BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw_u & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sb = raw_u + pad;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffCtl);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffCtl + 64);
  int4* unit_slot = reinterpret_cast<int4*>(smem + kOffCtl + 128);
  int* flag_slot = reinterpret_cast<int*>(smem + kOffCtl + 192);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rr = 32 * (warp & 3) + lane;  // MMA row / TMEM lane
  const int hc = warp >> 2;               // column half
  const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;

  // rows of a partly filled tile keep earlier (finite) data; zero everything once so
  // that 0-weighted rows never meet NaN bit patterns in the MMAs
  for (uint32_t o = tid * 16; o < 6 * kTile; o += kThreads * 16)
    *reinterpret_cast<uint4*>(smem + o) = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (tid == 0) {
    mbar_init(bar(B_KV), 1);
    mbar_init(bar(B_MMA1), 1);
    mbar_init(bar(B_MMA2), 1);
    mbar_fence_init();
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint64_t pol_kv = policy_evict_last();
  constexpr uint32_t idesc_kk = idesc_f16(128, 128, 1, 1, 0, 0);  // A, B K-major
  constexpr uint32_t idesc_tt = idesc_f16(128, 128, 1, 1, 1, 1);  // A, B MN-major
  constexpr uint32_t idesc_kt = idesc_f16(128, 128, 1, 1, 0, 1);  // A K-major, B MN-major
  const int nunits = *p.nunits;
  uint32_t kv_ph = 0, m1_ph = 0, m2_ph = 0;
  bool ok = true;

  for (;;) {
    if (tid == 0) {
      const int u = atomicAdd(p.counter, 1);
      *unit_slot = u < nunits ? p.units[u] : make_int4(-1, 0, 0, 0);
      flag_slot[0] = u;
    }
    __syncthreads();
    const int4 un = *unit_slot;
    const int uid = flag_slot[0];
    if (un.x < 0) break;
    const int g = un.x / p.nblocks, b = un.x - g * p.nblocks;
    if (tid == 0) {
      mbar_expect_tx(bar(B_KV), 2 * kTile);
      tma_load_3d(sb + kOffK, &tmK, 0, g, b * kBlock, bar(B_KV), pol_kv);
      tma_load_3d(sb + kOffK + 16384, &tmK, 64, g, b * kBlock, bar(B_KV), pol_kv);
      tma_load_3d(sb + kOffV, &tmV, 0, g, b * kBlock, bar(B_KV), pol_kv);
      tma_load_3d(sb + kOffV + 16384, &tmV, 64, g, b * kBlock, bar(B_KV), pol_kv);
    }
    const int ntile = (un.z + kTileQ - 1) / kTileQ;
    for (int t = 0; t < ntile && ok; ++t) {
      const int e0 = un.y + t * kTileQ;
      const int cnt = min(kTileQ, un.z - t * kTileQ);
      // gather Q and dO rows of the tile: chunk c (8 elements) of query j, head h
      for (int idx = tid; idx < cnt * 256; idx += kThreads) {
        const int j = idx >> 8, h = (idx >> 4) & 15, c = idx & 15;
        const int r = j * 16 + h;
        const size_t src = ((static_cast<size_t>(__ldg(p.qlist + e0 + j)) * p.Hq + g * kGroup + h) * kHeadDim + c * 8) * 2;
        const uint32_t dst = (c >> 3) * 16384 + r * 128 + (((c & 7) ^ (r & 7)) << 4);
        cp_async16(sb + kOffQ + dst, p.Q + src);
        cp_async16(sb + kOffDO + dst, p.dO + src);
      }
      const int j = rr >> 4, h = rr & 15;
      const bool valid = j < cnt;
      float lse2 = 0.f, dv = 0.f;
      int lim = -1;  // keys c <= lim of the block are visible to this row
      if (valid) {
        const int qi = __ldg(p.qlist + e0 + j);
        const size_t o = static_cast<size_t>(qi) * p.Hq + g * kGroup + h;
        lse2 = __ldg(p.LSE + o) * 1.4426950408889634f;
        dv = __ldg(p.Dv + o);
        lim = min(p.Lkv - p.N + qi - b * kBlock, kBlock - 1);
      }
      cp_async_wait_all();
      fence_proxy_async_smem();
      __syncthreads();
      if (tid == 0) {
        if (t == 0) {
          ok = mbar_wait(bar(B_KV), kv_ph);
          kv_ph ^= 1;
        }
        if (ok) {
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
            mma_f16_ss(tmem, smem_desc(sb + kOffQ + off, 16, 1024, 2), smem_desc(sb + kOffK + off, 16, 1024, 2),
                       idesc_kk, k > 0);
          }
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
            mma_f16_ss(tmem + 128, smem_desc(sb + kOffDO + off, 16, 1024, 2),
                       smem_desc(sb + kOffV + off, 16, 1024, 2), idesc_kk, k > 0);
          }
          mma_commit(bar(B_MMA1));
        }
        flag_slot[1] = ok;
      }
      __syncthreads();
      ok = flag_slot[1] != 0;
      if (!ok) break;
      ok = __syncthreads_and(mbar_wait(bar(B_MMA1), m1_ph));
      m1_ph ^= 1;
      if (!ok) break;
      tc_fence_after();
      {
        // P = 2^(S * scale * log2 e - LSE * log2 e) on visible keys, dS = P (dP - D)
        uint32_t s[64], d[64];
        const uint32_t tS = tmem + lane_base + 64 * hc;
        tmem_ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
        tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
        tmem_ld32(tS + 128, *reinterpret_cast<uint32_t(*)[32]>(&d[0]));
        tmem_ld32(tS + 160, *reinterpret_cast<uint32_t(*)[32]>(&d[32]));
        tmem_ld_wait();
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          uint32_t pw[4], dw[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int c0 = ch * 8 + 2 * q, key0 = 64 * hc + c0;
            const float p0 = key0 <= lim ? ex2(fmaf(__uint_as_float(s[c0]), p.sl2, -lse2)) : 0.f;
            const float p1 = key0 + 1 <= lim ? ex2(fmaf(__uint_as_float(s[c0 + 1]), p.sl2, -lse2)) : 0.f;
            pw[q] = pack_bf16x2(p0, p1);
            dw[q] = pack_bf16x2(p0 * (__uint_as_float(d[c0]) - dv), p1 * (__uint_as_float(d[c0 + 1]) - dv));
          }
          const uint32_t off = hc * 16384 + rr * 128 + ((ch ^ (rr & 7)) << 4);
          *reinterpret_cast<uint4*>(smem + kOffP + off) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
          *reinterpret_cast<uint4*>(smem + kOffDS + off) = make_uint4(dw[0], dw[1], dw[2], dw[3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();
      if (tid == 0) {
        tc_fence_after();
        // dV += P^T dO and dK += dS^T Q: A = P^T / dS^T (M = keys, K = rows), B = dO / Q
        // (K = rows, N = d), both MN-major; 16 rows per MMA = 2 KB of the tile
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_f16_ss(tmem + 256, smem_desc(sb + kOffP + k * 2048, 16384, 1024, 2),
                     smem_desc(sb + kOffDO + k * 2048, 16384, 1024, 2), idesc_tt, (t > 0 || k > 0) ? 1u : 0u);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_f16_ss(tmem + 384, smem_desc(sb + kOffDS + k * 2048, 16384, 1024, 2),
                     smem_desc(sb + kOffQ + k * 2048, 16384, 1024, 2), idesc_tt, (t > 0 || k > 0) ? 1u : 0u);
        // dQ part = dS K_b: A = dS (M = rows, K = keys) K-major, B = K_b (K = keys, N = d) MN-major
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
          mma_f16_ss(tmem, smem_desc(sb + kOffDS + off, 16, 1024, 2), smem_desc(sb + kOffK + k * 2048, 16384, 1024, 2),
                     idesc_kt, k > 0);
        }
        mma_commit(bar(B_MMA2));
      }
      ok = __syncthreads_and(mbar_wait(bar(B_MMA2), m2_ph));
      m2_ph ^= 1;
      if (!ok) break;
      tc_fence_after();
      {
        uint32_t v[64];
        const uint32_t tQ = tmem + lane_base + 64 * hc;
        tmem_ld32(tQ, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
        tmem_ld32(tQ + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
        tmem_ld_wait();
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(p.dq_part + ((static_cast<size_t>(e0 + j) * kGroup + h) * kHeadDim + 64 * hc));
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(v[8 * ch + 0]), __uint_as_float(v[8 * ch + 1]));
            w.y = pack_bf16x2(__uint_as_float(v[8 * ch + 2]), __uint_as_float(v[8 * ch + 3]));
            w.z = pack_bf16x2(__uint_as_float(v[8 * ch + 4]), __uint_as_float(v[8 * ch + 5]));
            w.w = pack_bf16x2(__uint_as_float(v[8 * ch + 6]), __uint_as_float(v[8 * ch + 7]));
            dst[ch] = w;
          }
        }
      }
      tc_fence_before();
      __syncthreads();
    }
    if (!ok) break;
    // the unit's dK, dV (TMEM lane = key of the block) -> fp32 partials of the unit
    tc_fence_after();
    float* dk = p.dkv + static_cast<size_t>(uid) * 2 * kBlock * kHeadDim;
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      uint32_t v[64];
      const uint32_t tA = tmem + lane_base + (m == 0 ? 384 : 256) + 64 * hc;
      tmem_ld32(tA, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
      tmem_ld32(tA + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
      tmem_ld_wait();
      float4* dst = reinterpret_cast<float4*>(dk + (static_cast<size_t>(m) * kBlock + rr) * kHeadDim + 64 * hc);
#pragma unroll
      for (int q = 0; q < 16; ++q)
        dst[q] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]), __uint_as_float(v[4 * q + 2]),
                             __uint_as_float(v[4 * q + 3]));
    }
    tc_fence_before();
    __syncthreads();
  }
  if (!ok && tid == 0) atomicOr(&p.hdr->status, kStatusTimeout);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

// D[i, h] = dO[i, h, :] . O[i, h, :] in fp32: 16 threads per row (8 elements each), two
// rows per warp; the loop bound is warp-uniform so every lane joins the shuffles.
__global__ void __launch_bounds__(256) bwd_prep_kernel(const uint4* __restrict__ O, const uint4* __restrict__ dO,
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
    if (sub == 0 && r < rows) Dv[r] = s;
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
  b += (static_cast<size_t>(s->N) * s->Hkv * kGroup * sizeof(float) + 255) / 256 * 256;  // D
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
                                                            static_cast<const uint4*>(a.dO), Dv, qrows);
    if ((e = cudaGetLastError())) return e;
  }
  bwd_units_kernel<<<1, 1024, 0, st>>>(s->d.counts, s->d.offsets, s->R, units, unit_off);
  if ((e = cudaGetLastError())) return e;
  if ((e = cudaMemsetAsync(counter, 0, sizeof(int32_t), st))) return e;

  CUtensorMap tmK, tmV;
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
  p.Q = static_cast<const uint8_t*>(a.Q);
  p.dO = static_cast<const uint8_t*>(a.dO);
  p.LSE = a.LSE;
  p.Dv = Dv;
  p.units = units;
  p.qlist = s->d.qlist;
  p.counter = counter;
  p.nunits = unit_off + s->R;
  p.dq_part = static_cast<__nv_bfloat16*>(s->partial);
  p.dkv = dkv;
  p.hdr = s->d.hdr;
  p.N = s->N;
  p.Lkv = a.Lkv;
  p.Hq = a.Hq;
  p.nblocks = s->nblocks;
  p.sl2 = a.scale * 1.4426950408889634f;
  static bool attr_set = false;
  if (!attr_set) {
    if ((e = cudaFuncSetAttribute(bwd_kv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes))) return e;
    attr_set = true;
  }
  bwd_kv_kernel<<<a.num_ctas, kThreads, kSmemBytes, st>>>(tmK, tmV, p);
  if ((e = cudaGetLastError())) return e;
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
  }
  return cudaGetLastError();
}

}  // namespace msa
