// Combine: merge each query's partial outputs by their softmax statistics.
//
// "Sparse Attention" (dinara-dl), Chapter 5, "Partial outputs and Combine": every
// selected block of a query yields a partial output and its softmax statistics;
// combine turns them into relative weights and merges the partials (not a plain
// average).  "Kernel optimization for MiniMax M3", load/store section: the
// attention kernel stores partials tile-ordered and raw (normalisation deferred to
// combine); combine gathers them through the map (query, kv_head, top-i) ->
// partial row.  It is bandwidth-bound and tolerant of gather latency.
//
// Partial k of (query i, group g, head h) belongs to CSR position p = cmap[i, g, k] of
// the bf16 (or, on request, fp32) partial workspace, in the chunk-major layout of
// part_index (aligned groups of 8 positions, 16-byte column chunks outermost), with its
// statistics at pstat[16 p + h]: O_k = sum_j 2^(x_j - m_k) V_j over the block's visible keys
// (x = score * scale * log2 e), with statistics (m_k, l_k = sum_j 2^(x_j - m_k)).
// For E4M3 inputs the V descale multiplies the merged output (the partials hold P V
// of the stored E4M3 values).
// With M = max_k m_k and w_k = 2^(m_k - M):
//   O = sum_k w_k O_k / sum_k w_k l_k,   LSE = ln 2 * (M + log2 sum_k w_k l_k).
//
// One CTA of 256 threads per (i, g) unit at a time: thread (h, c) = (tid % 16, tid / 16)
// owns head h and output columns [8c, 8c + 8); a warp reads two 256-byte runs of each
// partial (column chunks c, c + 1 of the 16 heads).  The
// statistics and partial loads of 8 slots are issued together once the combine map is
// known; the first 8 map entries of a CTA's next unit are loaded while it merges the
// current one, so a unit of up to 8 slots costs one round trip.  Partials and statistics
// are read once: streaming loads (evict-first).  64 registers per thread keep 4 CTAs (32
// warps) resident per SM so that enough loads are in flight to cover HBM latency; the
// grid is 64 CTAs per SM (16 waves), which shortens the tail of the last wave (16, 32,
// 64, 128 per SM measured: 0.335, 0.332, 0.331, 0.333 ms at M3).
#include <cuda_bf16.h>

#include "msa_internal.h"
#include "ptx.cuh"

namespace msa {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ void acc8(float (&a)[8], const uint4& v, float w) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    a[2 * q] = fmaf(w, __uint_as_float(u[q] << 16), a[2 * q]);
    a[2 * q + 1] = fmaf(w, __uint_as_float(u[q] & 0xFFFF0000u), a[2 * q + 1]);
  }
}

// 8 consecutive columns of one partial row: bf16 (one 16-byte load) or fp32 (two)
template <bool kF32>
struct Part8;
template <>
struct Part8<false> {
  uint4 a;
};
template <>
struct Part8<true> {
  uint4 a, b;
};
template <bool kF32>
__device__ __forceinline__ void acc_part8(float (&a)[8], const Part8<kF32>& v, float w) {
  if constexpr (kF32) {
    const uint32_t u[8] = {v.a.x, v.a.y, v.a.z, v.a.w, v.b.x, v.b.y, v.b.z, v.b.w};
#pragma unroll
    for (int q = 0; q < 8; ++q) a[q] = fmaf(w, __uint_as_float(u[q]), a[q]);
  } else {
    acc8(a, v.a, w);
  }
}

template <bool kF32>
__global__ void __launch_bounds__(kThreads, kF32 ? 3 : 4)
combine_kernel(const int32_t* __restrict__ cmap, const uint4* __restrict__ partial,
               const float2* __restrict__ pstat, int N, int Hkv, int topK, int Hq,
               __nv_bfloat16* __restrict__ O, float* __restrict__ LSE, float v_descale,
               SchedHeader* __restrict__ hdr, int force_path, int64_t cap_e) {
  griddep_wait();
  // (no early griddep_launch here: the Q-outer kernel after this one would then be scheduled
  // beside running combine CTAs, and its ~210 KB of shared memory takes the L1 this kernel's
  // gathers rely on -- 0.83 -> 0.92 ms per M3 step)
  // the KV-outer launch before this one is complete: its chunk counter starts the next launch at zero
  if (blockIdx.x == 0 && threadIdx.x == 0) hdr->pad[0] = 0;
  constexpr int kKChunk = kF32 ? 4 : 8;  // partial loads in flight per thread
  const int path = force_path ? force_path : hdr->path;
  if (path != kPathKvOuter) return;
  const int h = threadIdx.x & 15, c = threadIdx.x >> 4;
  const int64_t units = static_cast<int64_t>(N) * Hkv;
  int pre[kKChunk];  // the first map entries of this CTA's next unit
  {
    const int64_t u0 = blockIdx.x;
#pragma unroll
    for (int k = 0; k < kKChunk; ++k) pre[k] = (u0 < units && k < topK) ? __ldg(cmap + u0 * topK + k) : -1;
  }
  for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
    const int32_t* cm = cmap + u * topK;
    int first[kKChunk];
#pragma unroll
    for (int k = 0; k < kKChunk; ++k) first[k] = pre[k];
    {
      const int64_t un = u + gridDim.x;
#pragma unroll
      for (int k = 0; k < kKChunk; ++k) pre[k] = (un < units && k < topK) ? __ldg(cmap + un * topK + k) : -1;
    }
    float M = -INFINITY, L = 0.f;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int k0 = 0; k0 < topK; k0 += kKChunk) {
      int pos[kKChunk];
#pragma unroll
      for (int k = 0; k < kKChunk; ++k) pos[k] = k0 == 0 ? first[k] : (k0 + k < topK) ? __ldg(cm + k0 + k) : -1;
#pragma unroll
      for (int k = 0; k < kKChunk; ++k)  // (bounds-checked build: a map entry out of range is dropped)
        if (!dbg_ok(pos[k] >= -1 && pos[k] < cap_e, &hdr->status)) pos[k] = -1;
      float2 st[kKChunk];
      Part8<kF32> v[kKChunk];
#pragma unroll
      for (int k = 0; k < kKChunk; ++k) {
        const int64_t r = static_cast<int64_t>(pos[k]) * kGroup + h;
        st[k] = pos[k] >= 0 ? __ldcs(pstat + r) : make_float2(-INFINITY, 0.f);
        if constexpr (kF32) {
          const int64_t x = part_index(pos[k], h, 2 * c, 32);
          v[k].a = pos[k] >= 0 ? __ldcs(partial + x) : make_uint4(0, 0, 0, 0);
          v[k].b = pos[k] >= 0 ? __ldcs(partial + x + kPartGroup * kGroup) : make_uint4(0, 0, 0, 0);
        } else {
          v[k].a = pos[k] >= 0 ? __ldcs(partial + part_index(pos[k], h, c, 16)) : make_uint4(0, 0, 0, 0);
        }
      }
      float Mc = M;
#pragma unroll
      for (int k = 0; k < kKChunk; ++k) Mc = fmaxf(Mc, st[k].x);
      if (Mc == -INFINITY) continue;  // no partial so far
      const float r = ex2(M - Mc);     // rescale what earlier chunks accumulated (0 when M = -inf)
      L *= r;
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] *= r;
#pragma unroll
      for (int k = 0; k < kKChunk; ++k) {
        const float w = pos[k] >= 0 ? ex2(st[k].x - Mc) : 0.f;
        L = fmaf(w, st[k].y, L);
        acc_part8<kF32>(acc, v[k], w);
      }
      M = Mc;
    }
    const int64_t i = u / Hkv, g = u % Hkv;
    const int64_t orow = i * Hq + g * kGroup + h;
    uint4 out;
    float lse;
    if (L > 0.f) {
      const float inv = v_descale / L;
      out.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
      out.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
      out.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
      out.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
      lse = (M + lg2(L)) * 0.6931471805599453f;
    } else {
      out = make_uint4(0, 0, 0, 0);
      lse = -INFINITY;
    }
    reinterpret_cast<uint4*>(O)[orow * 16 + c] = out;
    if (LSE && c == 0) LSE[orow] = lse;
  }
}

}  // namespace

cudaError_t launch_combine(const msa_schedule* s, int Hq, void* O, float* LSE, float v_descale, int force_path,
                           bool f32p, cudaStream_t st) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t units = static_cast<int64_t>(s->N) * s->Hkv;
  int64_t grid = sms * 64;
  if (grid > units) grid = units;
  if (f32p)
    MSA_LAUNCH(combine_kernel<true>, static_cast<int>(grid), kThreads, 0, st, 
        s->d.cmap, static_cast<const uint4*>(s->partial), s->pstat, s->N, s->Hkv, s->topK, Hq,
        static_cast<__nv_bfloat16*>(O), LSE, v_descale, s->d.hdr, force_path, s->cap_entries);
  else
    MSA_LAUNCH(combine_kernel<false>, static_cast<int>(grid), kThreads, 0, st, 
        s->d.cmap, static_cast<const uint4*>(s->partial), s->pstat, s->N, s->Hkv, s->topK, Hq,
        static_cast<__nv_bfloat16*>(O), LSE, v_descale, s->d.hdr, force_path, s->cap_entries);
  return cudaGetLastError();
}

}  // namespace msa
