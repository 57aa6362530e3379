// Forward main branch for block lists shared by tiles of consecutive queries, bf16,
// tcgen05 + TMA: no index inversion, no partial outputs, no combine.
//
// "Sparse Attention" (dinara-dl), Chapter 4: the selectors pick 16 KV blocks for each
// 128-query tile and GQA group, so every query of a tile attends the same blocks;
// Chapter 3 ("Q-tile" organisation): a tile of queries stays on chip while its blocks
// stream past, with one online softmax across the blocks.  Per query the result is the
// plain definition: softmax over the union of the list's blocks, keys after the query
// masked (the list is shared, the causal limit is per query).
//
// Unit = 8 consecutive queries x the 16 heads of one group = 128 MMA rows (the same
// head-packed layout as the KV-outer tile).  A CTA holds two units of one list (16
// consecutive queries) so each K/V block loaded serves both; it walks the list's
// blocks (deduplicated, ids after the pair's last query dropped) with
//   S = Q K^T  (tcgen05, both operands K-major, 128-byte swizzle) into S[u]
//   online softmax per row (thread = row): running reference maximum m_ref and sum l;
//   the O accumulator is rescaled only when a block raises the row maximum by more
//   than 8 (base 2): P = 2^(x - m_ref) stays <= 256, exact in fp32 accumulation
//   O[u] += P V   (P bf16 from TMEM over S[u], V MN-major)
// and at the end writes O = O / l (bf16) and LSE directly.
//
// Persistent CTAs of 384 threads, pairs taken round-robin:
//   warp 0      TMA: Q of both units (two 16 KB boxes each) and K_b, V_b through two
//               64 KB stages
//   warp 1      TMEM (512 columns: S[A], S[B], O[A], O[B]) and MMA issue; per unit the
//               chain is S -> softmax -> P V -> next S (S and P share columns), and the
//               two units interleave: O[A] += P V (block n), S[A] (n + 1), O[B] += P V
//               (n), S[B] (n + 1), so one unit's softmax overlaps the other's MMAs
//   warps 4-7   softmax and output of unit A; warps 8-11 of unit B
#include <cfloat>

#include <cuda.h>
#include <cuda_bf16.h>

#include "msa_internal.h"
#include "ptx.cuh"

namespace msa {
namespace {

constexpr int kThreads = 384;
constexpr uint32_t kTile = 32768;  // 128 x 128 bf16, two 16 KB halves
constexpr uint32_t kOffQ = 0;      // Q[A], Q[B]
constexpr uint32_t kOffKV = 2 * kTile;  // stage s: K at + s * 2 * kTile, V at + kTile
constexpr uint32_t kOffCtl = kOffKV + 4 * kTile;
constexpr uint32_t kSmemBytes = kOffCtl + 512 + 1024;
constexpr float kRescale = 8.f;  // lazy rescale threshold (base-2 units)
constexpr uint32_t kRegCtl = 120, kRegSm = 192;
static_assert(128 * (kRegCtl + 2 * kRegSm) <= kThreads * 168, "setmaxnreg shares exceed the launch allocation");

enum {
  B_QFULL = 0, B_QFREE = 1, B_KVFULL0 = 2, B_KVFREE0 = 4, B_SFULL0 = 6, B_PFULL0 = 8, B_PVDONE0 = 10,
  B_OFREE0 = 12, B_COUNT = 14
};

struct TlParams {
  const int32_t* lists;  // [ntiles, Hkv, topK]
  __nv_bfloat16* O;
  float* LSE;
  int32_t* status;  // may be null
  int N, Lkv, Hq, Hkv, topK, tile, nblocks;
  float sl2;  // scale * log2(e)
};

__device__ __forceinline__ void set_status(const TlParams& p, int bit) {
  if (p.status) atomicOr(p.status, bit);
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Blocks of pair `pr` (queries [16 j, 16 j + 16) of group g), in list order: valid ids
// (0 <= b < nblocks), first occurrence only, b <= the own block of the pair's last
// query.  Warp-collective; the k-th id is held by lane k % 32 in ids[k / 32].
struct PairBlocks {
  int ids[2];
  int n;
};
__device__ __forceinline__ PairBlocks pair_blocks(const TlParams& p, int j, int g, int lane, bool* bad) {
  const int i_last = min(16 * j + 15, p.N - 1);
  const int lb_max = (p.Lkv - p.N + i_last) / kBlock;
  const int32_t* lst = p.lists + (static_cast<int64_t>(16 * j / p.tile) * p.Hkv + g) * p.topK;
  PairBlocks r;
  r.ids[0] = r.ids[1] = -1;
  r.n = 0;
  const int b0 = lane < p.topK ? lst[lane] : -1;
  const int b1 = lane + 32 < p.topK ? lst[lane + 32] : -1;
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const int b = c ? b1 : b0;
    const int k = 32 * c + lane;
    bool ok = k < p.topK && b >= 0 && b < p.nblocks && b <= lb_max;
    if (k < p.topK && (b < -1 || b >= p.nblocks)) *bad = true;
    // a duplicate of an earlier slot is dropped
    for (int k2 = 0; k2 < 64; ++k2) {
      const int v = __shfl_sync(0xffffffffu, k2 < 32 ? b0 : b1, k2 & 31);
      if (k2 < k && v == b) ok = false;
    }
    const unsigned m = __ballot_sync(0xffffffffu, ok);
    for (int src = 0; src < 32; ++src) {
      const int v = __shfl_sync(0xffffffffu, b, src);
      if ((m >> src) & 1u) {
        const int dst = r.n + __popc(m & ((1u << src) - 1u));
        if ((dst & 31) == lane) {
          if (dst < 32) r.ids[0] = v;
          else r.ids[1] = v;
        }
      }
    }
    r.n += __popc(m);
  }
  return r;
}
__device__ __forceinline__ int block_at(const PairBlocks& pb, int k) {
  const int lo = __shfl_sync(0xffffffffu, pb.ids[0], k & 31);
  const int hi = __shfl_sync(0xffffffffu, pb.ids[1], k & 31);
  return k < 32 ? lo : hi;
}

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

// Maximum of the row's visible raw scores (keys c <= lim when kMasked), or of their
// negations when the scale is negative.
template <bool kMasked>
__device__ __forceinline__ float row_max(const uint32_t (&v)[128], int lim, bool neg) {
  // eight independent chains of 3-input maxima (short dependency chains)
  float a[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) a[q] = -FLT_MAX;
#pragma unroll
  for (int e = 0; e < 128; e += 16) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      float x0 = __uint_as_float(v[e + 2 * q]), x1 = __uint_as_float(v[e + 2 * q + 1]);
      if (neg) { x0 = -x0; x1 = -x1; }
      if (kMasked && e + 2 * q > lim) x0 = -FLT_MAX;
      if (kMasked && e + 2 * q + 1 > lim) x1 = -FLT_MAX;
      a[q] = max3(a[q], x0, x1);
    }
  }
  return fmaxf(fmaxf(max3(a[0], a[1], a[2]), max3(a[3], a[4], a[5])), fmaxf(a[6], a[7]));
}

// P = 2^(s * sl2 - m_ref) written over S as bf16 pairs (keys c > lim get 0 when
// kMasked); returns the row sum of P.
template <bool kMasked>
__device__ __forceinline__ float row_exp(const uint32_t (&v)[128], int lim, float sl2, float m_ref, uint32_t tS) {
  const uint64_t sl2x2 = pack2(sl2, sl2), negm2 = pack2(-m_ref, -m_ref);
  uint64_t sa[4] = {0, 0, 0, 0};  // four independent packed sums
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    uint32_t pk[8];
#pragma unroll
    for (int e = 0; e < 16; e += 2) {
      const int col = 16 * c + e;
      float x0, x1;
      unpack2(ffma2(pack2(__uint_as_float(v[col]), __uint_as_float(v[col + 1])), sl2x2, negm2), x0, x1);
      float p0 = ex2(x0), p1 = ex2(x1);
      if (kMasked) {
        if (col > lim) p0 = 0.f;
        if (col + 1 > lim) p1 = 0.f;
      }
      sa[(e >> 1) & 3] = fadd2(sa[(e >> 1) & 3], pack2(p0, p1));
      pk[e >> 1] = pack_bf16x2(p0, p1);
    }
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(tS + c * 8), "r"(pk[0]),
        "r"(pk[1]), "r"(pk[2]), "r"(pk[3]), "r"(pk[4]), "r"(pk[5]), "r"(pk[6]), "r"(pk[7])
        : "memory");
  }
  float l[8];
#pragma unroll
  for (int q = 0; q < 4; ++q) unpack2(sa[q], l[2 * q], l[2 * q + 1]);
  return ((l[0] + l[1]) + (l[2] + l[3])) + ((l[4] + l[5]) + (l[6] + l[7]));
}

template <uint32_t N>
__device__ __forceinline__ void regs_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N)); }
template <uint32_t N>
__device__ __forceinline__ void regs_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N)); }

__global__ void __launch_bounds__(kThreads, 1)
tiles_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
             const __grid_constant__ CUtensorMap tmV, const TlParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw_u & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sb = raw_u + pad;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffCtl);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffCtl + 8 * B_COUNT);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int npairs = (p.N + 15) / 16 * p.Hkv;

  if (tid == 0) {
    mbar_init(bar(B_QFULL), 1);
    mbar_init(bar(B_QFREE), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_KVFULL0 + s), 1);
      mbar_init(bar(B_KVFREE0 + s), 1);
      mbar_init(bar(B_SFULL0 + s), 1);
      mbar_init(bar(B_PFULL0 + s), 128);
      mbar_init(bar(B_PVDONE0 + s), 1);
      mbar_init(bar(B_OFREE0 + s), 128);
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
    bool bad = false;
    if (warp == 0) {
      // ---------------------------------------------------------- TMA producer
      if (lane == 0) { tma_prefetch_desc(&tmQ); tma_prefetch_desc(&tmK); tma_prefetch_desc(&tmV); }
      const uint64_t pol = policy_evict_last();
      bool ok = true;
      int n = 0, np = 0;
      for (int pr = blockIdx.x; pr < npairs && ok; pr += gridDim.x, ++np) {
        const int j = pr / p.Hkv, g = pr % p.Hkv;
        const PairBlocks pb = pair_blocks(p, j, g, lane, &bad);
        if (lane == 0) {
          // the Q buffers were last read by the S MMAs of the previous pair
          if (np > 0) ok = mbar_wait(bar(B_QFREE), (np - 1) & 1);
          if (ok) {
            mbar_expect_tx(bar(B_QFULL), 2 * kTile);
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int q0 = 16 * j + 8 * u;  // rows past N are filled with zeros
              tma_load_3d(sb + kOffQ + u * kTile, &tmQ, 0, g * kGroup, q0, bar(B_QFULL), pol);
              tma_load_3d(sb + kOffQ + u * kTile + 16384, &tmQ, 64, g * kGroup, q0, bar(B_QFULL), pol);
            }
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        for (int k = 0; k < pb.n && ok; ++k, ++n) {
          const int b = block_at(pb, k);
          if (lane == 0) {
            const int s = n & 1;
            if (n >= 2) ok = mbar_wait(bar(B_KVFREE0 + s), ((n >> 1) - 1) & 1);
            if (ok) {
              const uint32_t d = sb + kOffKV + s * 2 * kTile;
              mbar_expect_tx(bar(B_KVFULL0 + s), 2 * kTile);
              tma_load_3d(d, &tmK, 0, g, b * kBlock, bar(B_KVFULL0 + s), pol);
              tma_load_3d(d + 16384, &tmK, 64, g, b * kBlock, bar(B_KVFULL0 + s), pol);
              tma_load_3d(d + kTile, &tmV, 0, g, b * kBlock, bar(B_KVFULL0 + s), pol);
              tma_load_3d(d + kTile + 16384, &tmV, 64, g, b * kBlock, bar(B_KVFULL0 + s), pol);
            }
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
        }
      }
      if (!ok && lane == 0) set_status(p, kStatusTimeout);
      if (__any_sync(0xffffffffu, bad) && lane == 0) set_status(p, kStatusBadIndex);  // any lane saw one
    } else if (warp == 1) {
      // ---------------------------------------------------------- MMA issue
      constexpr uint32_t idesc_qk = idesc_f16(128, 128, 1, 1, 0, 0);
      constexpr uint32_t idesc_pv = idesc_f16(128, 128, 1, 1, 0, 1);
      bool ok = true;
      int n = 0, np = 0;
      for (int pr = blockIdx.x; pr < npairs && ok; pr += gridDim.x, ++np) {
        const int j = pr / p.Hkv, g = pr % p.Hkv;
        const PairBlocks pb = pair_blocks(p, j, g, lane, &bad);
        if (lane == 0 && pb.n > 0) {
          ok = mbar_wait(bar(B_QFULL), np & 1);
          // S[u] for block n: S[u] holds P of block n - 1 until that P V is done
          auto issue_s = [&](int u, int nn) -> bool {
            const int s = nn & 1;
            if (nn > 0 && !mbar_wait(bar(B_PVDONE0 + u), (nn - 1) & 1)) return false;
            tc_fence_after();
            const uint32_t qa = sb + kOffQ + u * kTile, ka = sb + kOffKV + s * 2 * kTile;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
              mma_f16_ss(tmem + u * 128, smem_desc(qa + off, 16, 1024, 2), smem_desc(ka + off, 16, 1024, 2),
                         idesc_qk, kk > 0);
            }
            mma_commit(bar(B_SFULL0 + u));
            return true;
          };
          // O[u] += P V for block nn (the first block of a pair overwrites O[u], which the
          // output warps of the previous pair must have read)
          auto issue_pv = [&](int u, int nn, bool first) -> bool {
            if (!mbar_wait(bar(B_PFULL0 + u), nn & 1)) return false;
            if (first && np > 0 && !mbar_wait(bar(B_OFREE0 + u), (np - 1) & 1)) return false;
            tc_fence_after();
            const uint32_t va = sb + kOffKV + (nn & 1) * 2 * kTile + kTile;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_f16_ts(tmem + 256 + u * 128, tmem + u * 128 + kk * 8, smem_desc(va + kk * 2048, 16384, 1024, 2),
                         idesc_pv, (!first || kk > 0) ? 1u : 0u);
            mma_commit(bar(B_PVDONE0 + u));
            return true;
          };
          // per unit the chain S -> softmax -> P V -> next S; the two units interleave:
          // P V(A, n), S(A, n + 1), P V(B, n), S(B, n + 1)
          const int n0 = n;
          ok = ok && mbar_wait(bar(B_KVFULL0 + (n0 & 1)), (n0 >> 1) & 1);
          ok = ok && issue_s(0, n0) && issue_s(1, n0);
          if (ok && pb.n == 1) mma_commit(bar(B_QFREE));
          for (int k = 0; k < pb.n && ok; ++k, ++n) {
            const bool more = k + 1 < pb.n;
            if (!(ok = issue_pv(0, n, k == 0))) break;
            if (more && !(ok = mbar_wait(bar(B_KVFULL0 + ((n + 1) & 1)), ((n + 1) >> 1) & 1))) break;
            if (more && !(ok = issue_s(0, n + 1))) break;
            if (!(ok = issue_pv(1, n, k == 0))) break;
            mma_commit(bar(B_KVFREE0 + (n & 1)));  // block n's K and V are read no more
            if (more && !(ok = issue_s(1, n + 1))) break;
            if (k + 2 == pb.n) mma_commit(bar(B_QFREE));  // the pair's last S MMAs are issued
          }
        } else if (lane == 0 && pb.n == 0) {
          // no blocks: nothing reads Q, the output warps write zeros
          ok = mbar_wait(bar(B_QFULL), np & 1);
          if (ok) mma_commit(bar(B_QFREE));
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
      if (!ok && lane == 0) set_status(p, kStatusTimeout);
    }
  } else {
    regs_inc<kRegSm>();
    // ------------------------------------------------------------ softmax + output (unit u)
    const int u = (warp - 4) >> 2;  // 0 (warps 4-7) or 1 (warps 8-11)
    const uint32_t bar_id = 1 + u;
    const int row = 32 * (warp & 3) + lane;
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const uint32_t tS = tmem + lane_base + u * 128, tO = tmem + lane_base + 256 + u * 128;
    const bool neg = p.sl2 < 0.f;
    bool ok = true, bad = false;
    int n = 0, np = 0;
    for (int pr = blockIdx.x; pr < npairs; pr += gridDim.x, ++np) {
      const int j = pr / p.Hkv, g = pr % p.Hkv;
      const PairBlocks pb = pair_blocks(p, j, g, lane, &bad);
      const int i = 16 * j + 8 * u + (row >> 4), h = row & 15;  // this row's query and head
      const int pos = p.Lkv - p.N + i;
      float m_ref = -INFINITY, l = 0.f;
      for (int k = 0; k < pb.n; ++k, ++n) {
        const int b = block_at(pb, k);
        ok = mbar_wait(bar(B_SFULL0 + u), n & 1);
        if (!named_bar_and(bar_id, 128, ok)) { ok = false; break; }
        tc_fence_after();
        uint32_t v[128];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32 * c]));
        tmem_ld_wait();
        const int lim = pos - b * kBlock;  // keys c <= lim are visible
        const bool masked = __any_sync(0xffffffffu, lim < kBlock - 1);
        // block maximum of x = s * sl2 over the visible keys (a negative scale turns the
        // maximum of s into its minimum)
        const float mm = masked ? row_max<true>(v, lim, neg) : row_max<false>(v, lim, neg);
        const float bm = (lim < 0) ? -INFINITY : (neg ? -mm : mm) * p.sl2;
        // raise the reference maximum (and rescale O and l) when the block exceeds it by
        // more than the threshold; tcgen05.ld/st are warp-collective, so a warp rescales
        // together (factor 1 for its rows that need none)
        const bool need = bm > m_ref + kRescale;
        if (__any_sync(0xffffffffu, need)) {
          const float alpha = need ? ex2(m_ref - bm) : 1.f;  // m_ref = -inf -> 0
          if (k > 0) {
            // O[u] holds the sum through the previous block: its P V completed before
            // this block's S MMA was issued (the MMA thread waits for it)
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              uint32_t o[16];
              tmem_ld16(tO + c * 16, o);
              tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
              tmem_st16(tO + c * 16, o);
            }
          }
          l *= alpha;
          if (need) m_ref = bm;
        }
        // P = 2^(x - m_ref) (bf16 pairs written over S), l += sum.  A row whose reference
        // is still -inf has seen no visible key and has none here (lim < 0): masked path.
        l += masked ? row_exp<true>(v, m_ref == -INFINITY ? -1 : lim, p.sl2, m_ref, tS)
                    : row_exp<false>(v, lim, p.sl2, m_ref, tS);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(B_PFULL0 + u));
      }
      if (!ok) break;
      // output: O / l (bf16) and LSE of this row
      if (pb.n > 0) {
        ok = mbar_wait(bar(B_PVDONE0 + u), (n - 1) & 1);
        if (!named_bar_and(bar_id, 128, ok)) { ok = false; break; }
        tc_fence_after();
      }
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint4* dst = reinterpret_cast<uint4*>(p.O + (static_cast<int64_t>(i) * p.Hq + g * kGroup + h) * kHeadDim);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        if (pb.n > 0) {
          tmem_ld32(tO + c * 32, o);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = 0u;
        }
        if (i < p.N) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            dst[c * 4 + q] = make_uint4(pack_bf16x2(__uint_as_float(o[8 * q]) * inv, __uint_as_float(o[8 * q + 1]) * inv),
                                        pack_bf16x2(__uint_as_float(o[8 * q + 2]) * inv, __uint_as_float(o[8 * q + 3]) * inv),
                                        pack_bf16x2(__uint_as_float(o[8 * q + 4]) * inv, __uint_as_float(o[8 * q + 5]) * inv),
                                        pack_bf16x2(__uint_as_float(o[8 * q + 6]) * inv, __uint_as_float(o[8 * q + 7]) * inv));
        }
      }
      tc_fence_before();
      mbar_arrive(bar(B_OFREE0 + u));
      if (p.LSE && i < p.N)
        p.LSE[static_cast<int64_t>(i) * p.Hq + g * kGroup + h] =
            l > 0.f ? (m_ref + lg2(l)) * 0.6931471805599453f : -INFINITY;
    }
    if (!ok && (tid & 127) == 0) set_status(p, kStatusTimeout);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t launch_tiles(const void* Q, const void* K, const void* V, int N, int Lkv, int Hq, int Hkv,
                         const int32_t* lists, int tile, int topK, float scale, void* O, float* LSE, int32_t* status,
                         int num_ctas, cudaStream_t st) {
  CUtensorMap tmQ, tmK, tmV;
  {
    // Q [N][Hq][128]: box = 64 columns of the 16 heads of 8 consecutive queries
    const uint64_t dims[3] = {kHeadDim, static_cast<uint64_t>(Hq), static_cast<uint64_t>(N)};
    const uint64_t strides[2] = {kHeadDim * 2, static_cast<uint64_t>(Hq) * kHeadDim * 2};
    const uint32_t box[3] = {64, kGroup, 8};
    if (!encode_tmap(&tmQ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, Q, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[3] = {kHeadDim, static_cast<uint64_t>(Hkv), static_cast<uint64_t>(Lkv)};
    const uint64_t strides[2] = {kHeadDim * 2, static_cast<uint64_t>(Hkv) * kHeadDim * 2};
    const uint32_t box[3] = {64, 1, kBlock};
    if (!encode_tmap(&tmK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, K, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
    if (!encode_tmap(&tmV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, V, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  static std::atomic<uint64_t> attr_done{0};
  {
    cudaError_t e = set_smem_limit(tiles_kernel, static_cast<int>(kSmemBytes), attr_done);
    if (e != cudaSuccess) return e;
  }
  TlParams p;
  p.lists = lists;
  p.O = static_cast<__nv_bfloat16*>(O);
  p.LSE = LSE;
  p.status = status;
  p.N = N;
  p.Lkv = Lkv;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.topK = topK;
  p.tile = tile;
  p.nblocks = Lkv / kBlock;
  p.sl2 = scale * 1.4426950408889634f;
  const int npairs = (N + 15) / 16 * Hkv;
  int grid = num_ctas < npairs ? num_ctas : npairs;
  tiles_kernel<<<grid, kThreads, kSmemBytes, st>>>(tmQ, tmK, tmV, p);
  return cudaGetLastError();
}

}  // namespace msa
