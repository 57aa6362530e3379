// Block selector R1: the step before the attention, producing its block lists.
//
// "Sparse Attention" (dinara-dl), Chapter 4, "R1: One Representative": for a tile of
// 128 consecutive queries and a GQA group, each query head of the group is summarised
// by the mean of its 128 query vectors and each KV block by the mean of its 128 key
// vectors; the block's score is the largest, over the group's heads, of the dot
// product of the two means; the tile keeps its topK best blocks, shared by all of its
// queries.  The blocks holding the tile's own queries are always kept (first, by id),
// blocks after the tile's last query are never candidates, ties go to the smaller
// block id, and short candidate sets are padded with -1.
//
// Kernels (fp32 arithmetic on bf16 inputs):
//   pool_keys     one CTA per (block, group): 16 row groups x 16 column chunks of
//                 16-byte loads, partial sums added in shared memory      -> kbar
//   pool_queries  one CTA per (tile, group): 4 query quarters x 256 column chunks of
//                 16-byte loads, partial sums added in shared memory      -> qbar
//   select        one CTA per (tile, group): the 16 query means in shared memory; a
//                 warp per candidate block computes the 16 dot products (lane = 4
//                 columns) and their maximum; then topK rounds of a CTA-wide arg-max;
//                 the list is written for every query of the tile.
// All three read their inputs once: the selector is bound by HBM reads of Q and K.
//
// Block selector R4 (same chapter, "R4: Four Representatives"): the tile and the block
// are each cut into four consecutive 32-token quarters, each summarised by its mean; the
// block's score is the largest of the 16 quarter-pair dot products over the group's
// heads.  A quarter of a short last tile that holds no query has no representative.
//   pool_keys4    one CTA per (block, group): quarter x 4 row groups x 16 chunks
//                 -> krepT [group][128 columns][4 nblocks]
//   pool_queries4 one CTA per (tile, group): thread = (quarter, head, 8 columns)
//                 -> qrepT [tile][group][128 columns][64 = head x 4 + quarter]
//   select4       the scores are a 64 x 4 nblocks x 128 product per (tile, group) with a
//                 maximum over each block's 64 x 4 entries: chunks of 16 candidate blocks,
//                 both operands transposed in shared memory, each thread accumulating 8
//                 query x 2 key representatives with packed fp32 FMAs; then the R1 top-K.
#include <cuda_bf16.h>

#include "msa_internal.h"

namespace msa {
namespace {

constexpr int kSelThreads = 256;

// 8 bf16 (one 16-byte word) added into a[0..7]
__device__ __forceinline__ void add8(float (&a)[8], const uint4& v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    a[2 * q] += __uint_as_float(w[q] << 16);
    a[2 * q + 1] += __uint_as_float(w[q] & 0xFFFF0000u);
  }
}

// One CTA of 256 threads per (block, group): thread = (key row group r = tid / 16,
// 16-byte column chunk c = tid % 16) sums keys r, r + 16, ... with 16-byte loads; the
// 16 row-group partials are added in shared memory.
__global__ void __launch_bounds__(256) k_pool_keys(const __nv_bfloat16* __restrict__ K, int Hkv, int nblocks,
                                                   float* __restrict__ kbar) {
  __shared__ float part[16][kHeadDim];
  const int b = blockIdx.x, g = blockIdx.y, tid = threadIdx.x, r = tid >> 4, c = tid & 15;
  const int64_t row = static_cast<int64_t>(Hkv) * kHeadDim / 8;  // uint4 per key
  const uint4* src = reinterpret_cast<const uint4*>(K + (static_cast<int64_t>(b) * kBlock * Hkv + g) * kHeadDim) + c;
  float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
  for (int j = r; j < kBlock; j += 16) add8(a, __ldg(src + j * row));
#pragma unroll
  for (int e = 0; e < 8; ++e) part[r][c * 8 + e] = a[e];
  __syncthreads();
  if (tid < kHeadDim) {
    float s = 0.f;
#pragma unroll
    for (int q = 0; q < 16; ++q) s += part[q][tid];
    kbar[(static_cast<int64_t>(g) * nblocks + b) * kHeadDim + tid] = s * (1.f / kBlock);
  }
}

// One CTA of 1024 threads per (tile, group): thread = (query quarter qq = tid / 256,
// 16-byte chunk c = tid % 256 of the group's 16 x 128 row block) sums queries
// i0 + qq, i0 + qq + 4, ...; the four partials are added in shared memory.
__global__ void __launch_bounds__(1024) k_pool_queries(const __nv_bfloat16* __restrict__ Q, int N, int Hq,
                                                       float* __restrict__ qbar) {
  __shared__ float part[3][kGroup * kHeadDim];
  const int t = blockIdx.x, g = blockIdx.y, tid = threadIdx.x, qq = tid >> 8, c = tid & 255;
  const int i0 = t * kBlock, i1 = min(i0 + kBlock, N);
  const int64_t row = static_cast<int64_t>(Hq) * kHeadDim / 8;  // uint4 per query row
  const uint4* src = reinterpret_cast<const uint4*>(Q + (static_cast<int64_t>(i0) * Hq + g * kGroup) * kHeadDim) + c;
  float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
  for (int i = qq; i < i1 - i0; i += 4) add8(a, __ldg(src + i * row));
  if (qq > 0) {
#pragma unroll
    for (int e = 0; e < 8; ++e) part[qq - 1][c * 8 + e] = a[e];
  }
  __syncthreads();
  if (qq == 0) {
    const float inv = 1.f / static_cast<float>(i1 - i0);
    float* dst = qbar + (static_cast<int64_t>(t) * Hq + g * kGroup) * kHeadDim + c * 8;
#pragma unroll
    for (int e = 0; e < 8; ++e) dst[e] = (a[e] + part[0][c * 8 + e] + part[1][c * 8 + e] + part[2][c * 8 + e]) * inv;
  }
}

// 16 per-lane values (one per head) reduced over the warp with 16 shuffles; lane l ends
// with the sum for head (l >> 1) % 16.
__device__ __forceinline__ float warp_sum16(const float (&v)[16], int lane) {
  float a[8], b[4], c[2];
  bool up = lane & 16;
#pragma unroll
  for (int j = 0; j < 8; ++j) a[j] = (up ? v[j + 8] : v[j]) + __shfl_xor_sync(0xffffffffu, up ? v[j] : v[j + 8], 16);
  up = lane & 8;
#pragma unroll
  for (int j = 0; j < 4; ++j) b[j] = (up ? a[j + 4] : a[j]) + __shfl_xor_sync(0xffffffffu, up ? a[j] : a[j + 4], 8);
  up = lane & 4;
#pragma unroll
  for (int j = 0; j < 2; ++j) c[j] = (up ? b[j + 2] : b[j]) + __shfl_xor_sync(0xffffffffu, up ? b[j] : b[j + 2], 4);
  up = lane & 2;
  const float d = (up ? c[1] : c[0]) + __shfl_xor_sync(0xffffffffu, up ? c[0] : c[1], 2);
  return d + __shfl_xor_sync(0xffffffffu, d, 1);
}

// (score, id) order of the list: higher score first, then smaller id
__device__ __forceinline__ bool better(float sa, int ba, float sb, int bb) {
  return sa > sb || (sa == sb && ba >= 0 && (bb < 0 || ba < bb));
}

// topK rounds of a CTA-wide arg-max over the scores sc[nblocks] (a chosen block is
// struck out), then the list is written for every query of the tile.
__device__ void topk_and_write(float* sc, int nblocks, int topK, int N, int Hkv, int g, int i0, int i1,
                               int32_t* __restrict__ indices) {
  __shared__ float red_s[kSelThreads / 32];
  __shared__ int red_b[kSelThreads / 32];
  __shared__ int list[64];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int k = 0; k < topK; ++k) {
    float bs = -INFINITY;
    int bb = -1;
    for (int b = tid; b < nblocks; b += kSelThreads) {
      const float s = sc[b];
      if (s != -INFINITY && better(s, b, bs, bb)) { bs = s; bb = b; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float os = __shfl_xor_sync(0xffffffffu, bs, o);
      const int ob = __shfl_xor_sync(0xffffffffu, bb, o);
      if (ob >= 0 && better(os, ob, bs, bb)) { bs = os; bb = ob; }
    }
    if (lane == 0) { red_s[warp] = bs; red_b[warp] = bb; }
    __syncthreads();
    if (tid == 0) {
      for (int w = 1; w < kSelThreads / 32; ++w)
        if (red_b[w] >= 0 && better(red_s[w], red_b[w], bs, bb)) { bs = red_s[w]; bb = red_b[w]; }
      list[k] = bb;
      if (bb >= 0) sc[bb] = -INFINITY;
    }
    __syncthreads();
  }
  for (int e = tid; e < (i1 - i0) * topK; e += kSelThreads) {
    const int i = i0 + e / topK, k = e % topK;
    indices[(static_cast<int64_t>(i) * Hkv + g) * topK + k] = list[k];
  }
}

__global__ void __launch_bounds__(kSelThreads) k_select(const float* __restrict__ qbar, const float* __restrict__ kbar,
                                                        int N, int Lkv, int Hq, int Hkv, int nblocks, int topK,
                                                        int32_t* __restrict__ indices) {
  extern __shared__ float sm[];
  float* qs = sm;                        // [16][128]
  float* sc = sm + kGroup * kHeadDim;    // [nblocks]
  const int t = blockIdx.x, g = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int i0 = t * kBlock, i1 = min(i0 + kBlock, N);
  const int lb_first = (Lkv - N + i0) / kBlock, lb_last = (Lkv - N + i1 - 1) / kBlock;

  const float* qsrc = qbar + (static_cast<int64_t>(t) * Hq + g * kGroup) * kHeadDim;
  for (int e = tid; e < kGroup * kHeadDim; e += kSelThreads) qs[e] = qsrc[e];
  __syncthreads();
  // scores: one warp per candidate block, lane = columns 4 lane .. 4 lane + 3
  for (int b = warp; b < nblocks; b += kSelThreads / 32) {
    float s;
    if (b > lb_last) {
      s = -INFINITY;
    } else if (b >= lb_first) {
      s = INFINITY;
    } else {
      const float4 k4 = reinterpret_cast<const float4*>(kbar + (static_cast<int64_t>(g) * nblocks + b) * kHeadDim)[lane];
      float part[kGroup];
#pragma unroll
      for (int h = 0; h < kGroup; ++h) {
        const float4 q4 = reinterpret_cast<const float4*>(qs + h * kHeadDim)[lane];
        part[h] = fmaf(q4.x, k4.x, fmaf(q4.y, k4.y, fmaf(q4.z, k4.z, q4.w * k4.w)));
      }
      float m = warp_sum16(part, lane);  // dot product of head (lane >> 1)
#pragma unroll
      for (int o = 2; o < 32; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      s = m;
    }
    if (lane == 0) sc[b] = s;
  }
  __syncthreads();
  topk_and_write(sc, nblocks, topK, N, Hkv, g, i0, i1, indices);
}


// R4 key representatives: one CTA of 256 threads per (block, group); thread = (quarter
// s = tid / 64, row group r = (tid / 16) % 4, 16-byte chunk c = tid % 16) sums keys
// 32 s + r, 32 s + r + 4, ... of the block; the row groups are added in shared memory.
__global__ void __launch_bounds__(256) k_pool_keys4(const __nv_bfloat16* __restrict__ K, int Hkv, int nblocks,
                                                    float* __restrict__ krep) {
  __shared__ float part[4][4][kHeadDim];
  const int b = blockIdx.x, g = blockIdx.y, tid = threadIdx.x, sq = tid >> 6, r = (tid >> 4) & 3, c = tid & 15;
  const int64_t row = static_cast<int64_t>(Hkv) * kHeadDim / 8;  // uint4 per key
  const uint4* src =
      reinterpret_cast<const uint4*>(K + ((static_cast<int64_t>(b) * kBlock + 32 * sq) * Hkv + g) * kHeadDim) + c;
  float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int j = r; j < 32; j += 4) add8(a, __ldg(src + j * row));
#pragma unroll
  for (int e = 0; e < 8; ++e) part[sq][r][c * 8 + e] = a[e];
  __syncthreads();
  for (int o = tid; o < 4 * kHeadDim; o += 256) {
    const int q = o & 3, d = o >> 2;
    const float v = (part[q][0][d] + part[q][1][d]) + (part[q][2][d] + part[q][3][d]);
    krep[(static_cast<int64_t>(g) * kHeadDim + d) * (4 * static_cast<int64_t>(nblocks)) + 4 * b + q] = v * (1.f / 32.f);
  }
}

// R4 query representatives: one CTA of 1024 threads per (tile, group); thread = (quarter
// s = tid / 256, head h = (tid / 16) % 16, 8 columns c = tid % 16) sums the quarter's
// queries (0 queries -> 0, never read).
__global__ void __launch_bounds__(1024) k_pool_queries4(const __nv_bfloat16* __restrict__ Q, int N, int Hq,
                                                        float* __restrict__ qrep) {
  const int t = blockIdx.x, g = blockIdx.y, tid = threadIdx.x, sq = tid >> 8, h = (tid >> 4) & 15, c = tid & 15;
  const int a0 = t * kBlock + 32 * sq, a1 = min(a0 + 32, N);
  const int64_t row = static_cast<int64_t>(Hq) * kHeadDim / 8;
  const uint4* src = reinterpret_cast<const uint4*>(Q + (static_cast<int64_t>(a0) * Hq + g * kGroup + h) * kHeadDim) + c;
  float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int i = 0; i < a1 - a0; ++i) add8(a, __ldg(src + i * row));
  const float inv = a1 > a0 ? 1.f / static_cast<float>(a1 - a0) : 0.f;
  const int Hkv = Hq / kGroup;
  float* dst = qrep + ((static_cast<int64_t>(t) * Hkv + g) * kHeadDim + c * 8) * 64 + h * 4 + sq;
#pragma unroll
  for (int e = 0; e < 8; ++e) dst[e * 64] = a[e] * inv;
}

// (x0, x1) * (s, s) + (c0, c1) on a pair of floats held as one 64-bit register
__device__ __forceinline__ uint64_t ffma2s(float s, uint64_t x, uint64_t c) {
  uint64_t ss, d;
  asm("mov.b64 %0, {%1, %1};" : "=l"(ss) : "f"(s));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(x), "l"(ss), "l"(c));
  return d;
}

// qrepT [tile][group][128][64], krepT [group][128][4 nblocks]; one CTA per (tile, group).
// Thread (warp w, lane l) of a chunk of 16 candidate blocks (64 key representatives)
// accumulates query representatives 8 w .. 8 w + 7 against key representatives 2 l, 2 l + 1.
__global__ void __launch_bounds__(kSelThreads) k_select4(const float* __restrict__ qrep, const float* __restrict__ krep,
                                                         int N, int Lkv, int Hq, int Hkv, int nblocks, int topK,
                                                         int32_t* __restrict__ indices) {
  extern __shared__ float sm[];
  float* qs = sm;                       // [128][64]
  float* ks = sm + kHeadDim * 64;       // [128][64]
  float* red = ks + kHeadDim * 64;      // [8 warps][64]
  float* sc = red + 8 * 64;             // [nblocks]
  const int t = blockIdx.x, g = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int i0 = t * kBlock, i1 = min(i0 + kBlock, N);
  const int nq = (i1 - i0 + 31) / 32;  // quarters holding queries
  const int lb_first = (Lkv - N + i0) / kBlock, lb_last = (Lkv - N + i1 - 1) / kBlock;
  const int64_t kcols = 4 * static_cast<int64_t>(nblocks);

  const float4* qsrc = reinterpret_cast<const float4*>(qrep + (static_cast<int64_t>(t) * Hkv + g) * kHeadDim * 64);
  for (int e = tid; e < kHeadDim * 16; e += kSelThreads) reinterpret_cast<float4*>(qs)[e] = qsrc[e];
  // candidates scored: blocks before the tile's first own block
  for (int b0 = 0; b0 < lb_first; b0 += 16) {
    __syncthreads();  // the previous chunk's key representatives have been read
    const float* kc = krep + static_cast<int64_t>(g) * kHeadDim * kcols + 4 * b0;
    for (int e = tid; e < kHeadDim * 16; e += kSelThreads) {
      const int d = e >> 4, c4 = (e & 15) * 4;  // 4 representatives (one block) per float4
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (b0 + (c4 >> 2) < nblocks) v = *reinterpret_cast<const float4*>(kc + d * kcols + c4);
      reinterpret_cast<float4*>(ks + d * 64)[e & 15] = v;
    }
    __syncthreads();
    uint64_t acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0;
#pragma unroll 4
    for (int d = 0; d < kHeadDim; ++d) {
      const float4 qa = reinterpret_cast<const float4*>(qs + d * 64 + 8 * warp)[0];
      const float4 qb = reinterpret_cast<const float4*>(qs + d * 64 + 8 * warp)[1];
      const uint64_t k2 = reinterpret_cast<const uint64_t*>(ks + d * 64)[lane];
      acc[0] = ffma2s(qa.x, k2, acc[0]);
      acc[1] = ffma2s(qa.y, k2, acc[1]);
      acc[2] = ffma2s(qa.z, k2, acc[2]);
      acc[3] = ffma2s(qa.w, k2, acc[3]);
      acc[4] = ffma2s(qb.x, k2, acc[4]);
      acc[5] = ffma2s(qb.y, k2, acc[5]);
      acc[6] = ffma2s(qb.z, k2, acc[6]);
      acc[7] = ffma2s(qb.w, k2, acc[7]);
    }
    // maximum over this warp's query representatives (quarter = index % 4 must hold queries)
    float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (((8 * warp + i) & 3) >= nq) continue;
      float x0, x1;
      asm("mov.b64 {%0, %1}, %2;" : "=f"(x0), "=f"(x1) : "l"(acc[i]));
      m0 = fmaxf(m0, x0);
      m1 = fmaxf(m1, x1);
    }
    red[warp * 64 + 2 * lane] = m0;
    red[warp * 64 + 2 * lane + 1] = m1;
    __syncthreads();
    if (tid < 16 && b0 + tid < lb_first) {
      float m = -INFINITY;
#pragma unroll
      for (int w = 0; w < 8; ++w)
#pragma unroll
        for (int r = 0; r < 4; ++r) m = fmaxf(m, red[w * 64 + 4 * tid + r]);
      sc[b0 + tid] = m;
    }
  }
  for (int b = lb_first + tid; b < nblocks; b += kSelThreads) sc[b] = b > lb_last ? -INFINITY : INFINITY;
  __syncthreads();
  topk_and_write(sc, nblocks, topK, N, Hkv, g, i0, i1, indices);
}

}  // namespace

// Enough for either selector: R4 keeps four representatives per tile / block, R1 one.
size_t select_workspace_bytes(int N, int Hq, int Hkv, int nblocks) {
  const size_t ntiles = (static_cast<size_t>(N) + kBlock - 1) / kBlock;
  const size_t q = ntiles * Hq * 4 * kHeadDim * sizeof(float);
  return ((q + 255) / 256) * 256 + static_cast<size_t>(Hkv) * nblocks * 4 * kHeadDim * sizeof(float);
}

uint32_t select_smem_bytes(int nblocks, int reps) {
  if (reps == 4) return static_cast<uint32_t>((2 * kHeadDim * 64 + 8 * 64 + nblocks) * sizeof(float));
  return static_cast<uint32_t>((kGroup * kHeadDim + nblocks) * sizeof(float));
}

cudaError_t launch_select_r1(const void* Q, const void* K, int N, int Lkv, int Hq, int Hkv, int topK, int32_t* indices,
                             void* workspace, cudaStream_t st) {
  const int nblocks = Lkv / kBlock;
  const int ntiles = (N + kBlock - 1) / kBlock;
  const size_t q = static_cast<size_t>(ntiles) * Hq * kHeadDim * sizeof(float);
  float* qbar = static_cast<float*>(workspace);
  float* kbar = reinterpret_cast<float*>(static_cast<char*>(workspace) + ((q + 255) / 256) * 256);
  const uint32_t smem = select_smem_bytes(nblocks, 1);
  if (smem > 48 * 1024) {  // (a per-device attribute, set on every call: the selector is not on the timed path)
    cudaError_t e = cudaFuncSetAttribute(k_select, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
  }
  k_pool_keys<<<dim3(nblocks, Hkv), 256, 0, st>>>(static_cast<const __nv_bfloat16*>(K), Hkv, nblocks, kbar);
  k_pool_queries<<<dim3(ntiles, Hkv), 1024, 0, st>>>(static_cast<const __nv_bfloat16*>(Q), N, Hq, qbar);
  k_select<<<dim3(ntiles, Hkv), kSelThreads, smem, st>>>(qbar, kbar, N, Lkv, Hq, Hkv, nblocks, topK, indices);
  return cudaGetLastError();
}

cudaError_t launch_select_r4(const void* Q, const void* K, int N, int Lkv, int Hq, int Hkv, int topK, int32_t* indices,
                             void* workspace, cudaStream_t st) {
  const int nblocks = Lkv / kBlock;
  const int ntiles = (N + kBlock - 1) / kBlock;
  const size_t q = static_cast<size_t>(ntiles) * Hq * 4 * kHeadDim * sizeof(float);
  float* qrep = static_cast<float*>(workspace);
  float* krep = reinterpret_cast<float*>(static_cast<char*>(workspace) + ((q + 255) / 256) * 256);
  const uint32_t smem = select_smem_bytes(nblocks, 4);
  if (smem > 48 * 1024) {  // (a per-device attribute, set on every call: the selector is not on the timed path)
    cudaError_t e = cudaFuncSetAttribute(k_select4, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
  }
  k_pool_keys4<<<dim3(nblocks, Hkv), 256, 0, st>>>(static_cast<const __nv_bfloat16*>(K), Hkv, nblocks, krep);
  k_pool_queries4<<<dim3(ntiles, Hkv), 1024, 0, st>>>(static_cast<const __nv_bfloat16*>(Q), N, Hq, qrep);
  k_select4<<<dim3(ntiles, Hkv), kSelThreads, smem, st>>>(qrep, krep, N, Lkv, Hq, Hkv, nblocks, topK, indices);
  return cudaGetLastError();
}

}  // namespace msa
