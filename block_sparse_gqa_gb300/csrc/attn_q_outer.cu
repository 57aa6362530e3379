// Q-outer (query-stationary) attention, bf16: the low-reuse fallback.
//
// "Kernel optimization for MiniMax M3 on NVIDIA Blackwell", Q-outer vs KV-outer
// section: when nsb / N >= 2.85 (few queries share a block) each query walks its
// own selected blocks; no partial outputs and no combine are needed.
//
// Unit = (query i, group g): the 16 heads of the group form one m16 MMA tile.  A CTA
// of 4 warps takes a unit; warp w covers keys [32w, 32w + 32) of every selected
// block, streaming its K/V slices through a two-stage cp.async buffer and keeping an
// online softmax (running max, running sum, rescaled accumulator) across blocks.
// The four warps merge their (max, sum, output) at the end of the unit and write O
// and LSE directly.  Tensor work uses warp-level mma.sync m16n8k16 (bf16 in, fp32
// accumulate): this path moves ~64 KB of K/V per selected block per unit and is
// bound by memory, not by the tensor pipe.
#include <cuda_bf16.h>

#include "msa_internal.h"
#include "ptx.cuh"

namespace msa {
namespace {

constexpr int kWarps = 4, kThreads = 128;
constexpr int kStride = 136;                            // bf16 per padded smem row (272 B): conflict-free
constexpr int kSliceElems = 32 * kStride;               // one 32-key slice
constexpr int kWarpElems = 2 /*stages*/ * 2 /*K,V*/ * kSliceElems;
constexpr uint32_t kSmemBytes = kWarps * kWarpElems * 2 + 1024;

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                              uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait0() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

struct QoParams {
  const __nv_bfloat16* Q;
  const __nv_bfloat16* K;
  const __nv_bfloat16* V;
  const int32_t* blist;
  const SchedHeader* hdr;
  __nv_bfloat16* O;
  float* LSE;
  int N, Lkv, Hq, Hkv, topK;
  float sl2;
  int force_path;
};

__global__ void __launch_bounds__(kThreads, 1) q_outer_kernel(const QoParams p) {
  const int path = p.force_path ? p.force_path : p.hdr->path;
  if (path != kPathQOuter) return;
  extern __shared__ uint8_t smem_raw[];
  __nv_bfloat16* smem = reinterpret_cast<__nv_bfloat16*>(smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023));
  __shared__ float s_ml[kWarps][kGroup][2];
  __shared__ int s_blocks[64];
  __shared__ int s_nb;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3;
  __nv_bfloat16* wbuf = smem + warp * kWarpElems;  // [stage][K|V][32][kStride]
  const uint32_t wbuf_u = smem_u32(wbuf);
  const int64_t units = static_cast<int64_t>(p.N) * p.Hkv;

  for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
    const int i = static_cast<int>(u / p.Hkv), g = static_cast<int>(u % p.Hkv);
    const int pos = p.Lkv - p.N + i;
    if (tid == 0) {
      int nb = 0;
      for (int k = 0; k < p.topK && nb < 64; ++k) {
        const int b = p.blist[u * p.topK + k];
        if (b >= 0) s_blocks[nb++] = b;
      }
      s_nb = nb;
    }
    __syncthreads();
    const int nb = s_nb;

    // Q fragments of the 16 heads (A operand, row-major 16 x 128)
    uint32_t qa[8][4];
    {
      const uint32_t* q0 = reinterpret_cast<const uint32_t*>(p.Q + (static_cast<int64_t>(i) * p.Hq + g * kGroup + gid) * kHeadDim);
      const uint32_t* q8 = q0 + 8 * kHeadDim / 2;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        qa[kk][0] = __ldg(q0 + kk * 8 + tig);
        qa[kk][1] = __ldg(q8 + kk * 8 + tig);
        qa[kk][2] = __ldg(q0 + kk * 8 + 4 + tig);
        qa[kk][3] = __ldg(q8 + kk * 8 + 4 + tig);
      }
    }
    float o[16][4];
#pragma unroll
    for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};

    auto prefetch = [&](int t) {
      const int b = s_blocks[t];
      const int st = t & 1;
      for (int idx = lane; idx < 32 * 16; idx += 32) {
        const int r = idx >> 4, c = idx & 15;
        const int64_t key = static_cast<int64_t>(b) * kBlock + warp * 32 + r;
        const int64_t goff = (key * p.Hkv + g) * kHeadDim + c * 8;
        const uint32_t soff = ((st * 2) * kSliceElems + r * kStride + c * 8) * 2;
        cp_async16(wbuf_u + soff, p.K + goff);
        cp_async16(wbuf_u + soff + kSliceElems * 2, p.V + goff);
      }
    };
    if (nb > 0) prefetch(0);
    cp_async_commit();
    for (int t = 0; t < nb; ++t) {
      if (t + 1 < nb) prefetch(t + 1);
      cp_async_commit();
      cp_async_wait1();
      __syncwarp();
      const int st = t & 1, b = s_blocks[t];
      const __nv_bfloat16* sK = wbuf + (st * 2) * kSliceElems;
      const uint32_t sV_u = wbuf_u + ((st * 2 + 1) * kSliceElems) * 2;
      // S = Q K^T over this warp's 32 keys (4 n-tiles of 8 keys)
      float s[4][4];
#pragma unroll
      for (int n = 0; n < 4; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
        for (int n = 0; n < 4; ++n) {
          const uint32_t* kr = reinterpret_cast<const uint32_t*>(sK + (n * 8 + gid) * kStride + kk * 16);
          mma_bf16_16816(s[n], qa[kk], kr[tig], kr[4 + tig]);
        }
      }
      // scale to base-2 units, mask keys beyond the query's position, online softmax
      const int key0 = b * kBlock + warp * 32;
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int n = 0; n < 4; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = key0 + n * 8 + 2 * tig + (e & 1);
          s[n][e] = key <= pos ? s[n][e] * p.sl2 : -INFINITY;
          mx[e >> 1] = fmaxf(mx[e >> 1], s[n][e]);
        }
      float alpha[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
        const float mnew = fmaxf(mrow[r], mx[r]);
        alpha[r] = (mnew == -INFINITY) ? 1.f : ex2(mrow[r] - mnew);
        mrow[r] = mnew;
        lrow[r] *= alpha[r];
      }
#pragma unroll
      for (int n = 0; n < 4; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float v = s[n][e] == -INFINITY ? 0.f : ex2(s[n][e] - mrow[e >> 1]);
          s[n][e] = v;
          lrow[e >> 1] += v;
        }
#pragma unroll
      for (int n = 0; n < 16; ++n) {
        o[n][0] *= alpha[0]; o[n][1] *= alpha[0];
        o[n][2] *= alpha[1]; o[n][3] *= alpha[1];
      }
      // O += P V: two k-steps of 16 keys
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        uint32_t pa[4];
        pa[0] = pack_bf16x2(s[2 * kk][0], s[2 * kk][1]);
        pa[1] = pack_bf16x2(s[2 * kk][2], s[2 * kk][3]);
        pa[2] = pack_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
        pa[3] = pack_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
        const int mat = lane >> 3, rr = lane & 7;
        const int krow = kk * 16 + (mat & 1) * 8 + rr;
#pragma unroll
        for (int n = 0; n < 16; n += 2) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_trans(sV_u + (krow * kStride + (n + (mat >> 1)) * 8) * 2, b0, b1, b2, b3);
          mma_bf16_16816(o[n], pa, b0, b1);
          mma_bf16_16816(o[n + 1], pa, b2, b3);
        }
      }
      __syncwarp();
    }
    cp_async_wait0();
    // row sums over the four lanes that share a row
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      lrow[r] += __shfl_xor_sync(0xffffffffu, lrow[r], 1);
      lrow[r] += __shfl_xor_sync(0xffffffffu, lrow[r], 2);
    }
    __syncthreads();  // every warp is done with its buffers
    if (tig == 0) {
      s_ml[warp][gid][0] = mrow[0]; s_ml[warp][gid][1] = lrow[0];
      s_ml[warp][gid + 8][0] = mrow[1]; s_ml[warp][gid + 8][1] = lrow[1];
    }
    __syncthreads();
    float* red = reinterpret_cast<float*>(wbuf);  // this warp's scaled output, fp32 [16][128]
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int row = gid + 8 * r;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) M = fmaxf(M, s_ml[w][row][0]);
      float L = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w)
        if (s_ml[w][row][0] != -INFINITY) L += s_ml[w][row][1] * ex2(s_ml[w][row][0] - M);
      const float fac = (L > 0.f && mrow[r] != -INFINITY) ? ex2(mrow[r] - M) / L : 0.f;
#pragma unroll
      for (int n = 0; n < 16; ++n) {
        red[row * 128 + n * 8 + 2 * tig] = o[n][2 * r] * fac;
        red[row * 128 + n * 8 + 2 * tig + 1] = o[n][2 * r + 1] * fac;
      }
      if (warp == 0 && tig == 0 && p.LSE)
        p.LSE[static_cast<int64_t>(i) * p.Hq + g * kGroup + row] =
            L > 0.f ? (M + lg2(L)) * 0.6931471805599453f : -INFINITY;
    }
    __syncthreads();
    // sum the four warps' scaled outputs: thread handles 16 consecutive outputs
    {
      const int idx0 = tid * 16;
      const int row = idx0 >> 7, col = idx0 & 127;
      float acc[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) acc[e] = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float* rw = reinterpret_cast<const float*>(smem + w * kWarpElems) + row * 128 + col;
#pragma unroll
        for (int e = 0; e < 16; ++e) acc[e] += rw[e];
      }
      uint4 out[2];
      out[0].x = pack_bf16x2(acc[0], acc[1]);   out[0].y = pack_bf16x2(acc[2], acc[3]);
      out[0].z = pack_bf16x2(acc[4], acc[5]);   out[0].w = pack_bf16x2(acc[6], acc[7]);
      out[1].x = pack_bf16x2(acc[8], acc[9]);   out[1].y = pack_bf16x2(acc[10], acc[11]);
      out[1].z = pack_bf16x2(acc[12], acc[13]); out[1].w = pack_bf16x2(acc[14], acc[15]);
      uint4* dst = reinterpret_cast<uint4*>(p.O + (static_cast<int64_t>(i) * p.Hq + g * kGroup + row) * kHeadDim + col);
      dst[0] = out[0];
      dst[1] = out[1];
    }
    __syncthreads();  // buffers and s_blocks are reused by the next unit
  }
}

}  // namespace

cudaError_t launch_q_outer(const msa_schedule* s, const void* Q, const void* K, const void* V, int Hq, float scale,
                           void* O, float* LSE, int force_path, cudaStream_t st) {
  if (s->topK > 64) return cudaErrorInvalidValue;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(q_outer_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  QoParams p;
  p.Q = static_cast<const __nv_bfloat16*>(Q);
  p.K = static_cast<const __nv_bfloat16*>(K);
  p.V = static_cast<const __nv_bfloat16*>(V);
  p.blist = s->d.blist;
  p.hdr = s->d.hdr;
  p.O = static_cast<__nv_bfloat16*>(O);
  p.LSE = LSE;
  p.N = s->N;
  p.Lkv = s->nblocks * kBlock;
  p.Hq = Hq;
  p.Hkv = s->Hkv;
  p.topK = s->topK;
  p.sl2 = scale * 1.4426950408889634f;
  p.force_path = force_path;
  const int64_t units = static_cast<int64_t>(s->N) * s->Hkv;
  int64_t grid = sms;
  if (grid > units) grid = units;
  q_outer_kernel<<<static_cast<int>(grid), kThreads, kSmemBytes, st>>>(p);
  return cudaGetLastError();
}

}  // namespace msa
