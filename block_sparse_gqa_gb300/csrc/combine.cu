// Combine: merge each query's partial outputs by log-sum-exp weighting.
//
// "Sparse Attention" (dinara-dl), Chapter 5, "Partial outputs and Combine": every
// selected block of a query yields a partial output and an LSE; combine turns the
// LSEs into relative weights and merges the partials (not a plain average).
// "Kernel optimization for MiniMax M3", load/store section: the attention kernel
// stores partials tile-ordered; combine gathers them through the map
// (query, kv_head, top-i) -> partial row.  It is bandwidth-bound and tolerant of
// gather latency.
//
// Partial k of (query i, group g, head h) is row 16 * cmap[i, g, k] + h of the
// bf16 [E*16, 128] slab, already normalised by its own softmax sum, with base-2
// log-sum-exp lse2_k.  With M = max_k lse2_k and w_k = 2^(lse2_k - M):
//   O = sum_k w_k O_k / sum_k w_k,   LSE = ln 2 * (M + log2 sum_k w_k).
//
// One CTA of 256 threads per (i, g) unit: thread (h, c) owns head h and output
// columns [8c, 8c + 8) and gathers 16-byte pieces of each partial row, so a warp
// reads 512 contiguous bytes per partial.
#include <cuda_bf16.h>

#include "msa_internal.h"
#include "ptx.cuh"

namespace msa {
namespace {

constexpr int kThreads = 256;
constexpr int kKChunk = 16;

__device__ __forceinline__ void acc8(float (&a)[8], const uint4& v, float w) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    a[2 * q] = fmaf(w, __uint_as_float(u[q] << 16), a[2 * q]);
    a[2 * q + 1] = fmaf(w, __uint_as_float(u[q] & 0xFFFF0000u), a[2 * q + 1]);
  }
}

__global__ void __launch_bounds__(kThreads)
combine_kernel(const int32_t* __restrict__ cmap, const uint4* __restrict__ partial, const float* __restrict__ plse,
               int N, int Hkv, int topK, int Hq, __nv_bfloat16* __restrict__ O, float* __restrict__ LSE,
               const SchedHeader* __restrict__ hdr, int force_path) {
  const int path = force_path ? force_path : hdr->path;
  if (path != kPathKvOuter) return;
  const int h = threadIdx.x >> 4, c = threadIdx.x & 15;
  const int64_t units = static_cast<int64_t>(N) * Hkv;
  for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
    const int32_t* cm = cmap + u * topK;
    // weights: max and sum of 2^(lse2 - M) over the valid partials
    float M = -INFINITY;
    for (int k = 0; k < topK; ++k) {
      const int pk = __ldg(cm + k);
      if (pk >= 0) M = fmaxf(M, __ldg(plse + static_cast<int64_t>(pk) * kGroup + h));
    }
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float S = 0.f;
    for (int k0 = 0; k0 < topK; k0 += kKChunk) {
      int pos[kKChunk];
      float w[kKChunk];
      uint4 v[kKChunk];
#pragma unroll
      for (int k = 0; k < kKChunk; ++k) {
        pos[k] = (k0 + k < topK) ? __ldg(cm + k0 + k) : -1;
        w[k] = pos[k] >= 0 ? ex2(__ldg(plse + static_cast<int64_t>(pos[k]) * kGroup + h) - M) : 0.f;
      }
#pragma unroll
      for (int k = 0; k < kKChunk; ++k)
        v[k] = pos[k] >= 0 ? __ldg(partial + (static_cast<int64_t>(pos[k]) * kGroup + h) * 16 + c)
                           : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int k = 0; k < kKChunk; ++k) {
        S += w[k];
        acc8(acc, v[k], w[k]);
      }
    }
    const int64_t i = u / Hkv, g = u % Hkv;
    const int64_t orow = i * Hq + g * kGroup + h;
    uint4 out;
    float lse;
    if (S > 0.f) {
      const float inv = 1.f / S;
      out.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
      out.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
      out.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
      out.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
      lse = (M + lg2(S)) * 0.6931471805599453f;
    } else {
      out = make_uint4(0, 0, 0, 0);
      lse = -INFINITY;
    }
    reinterpret_cast<uint4*>(O)[orow * 16 + c] = out;
    if (LSE && c == 0) LSE[orow] = lse;
  }
}

}  // namespace

cudaError_t launch_combine(const msa_schedule* s, int Hq, void* O, float* LSE, int force_path, cudaStream_t st) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t units = static_cast<int64_t>(s->N) * s->Hkv;
  int64_t grid = sms * 8;
  if (grid > units) grid = units;
  combine_kernel<<<static_cast<int>(grid), kThreads, 0, st>>>(
      s->d.cmap, static_cast<const uint4*>(s->partial), s->plse, s->N, s->Hkv, s->topK, Hq,
      static_cast<__nv_bfloat16*>(O), LSE, s->d.hdr, force_path);
  return cudaGetLastError();
}

}  // namespace msa
