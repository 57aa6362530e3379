// Q-outer (query-stationary) attention, bf16 or fp8 E4M3, tcgen05 + TMA: the low-reuse
// fallback.
//
// "Kernel optimization for MiniMax M3 on NVIDIA Blackwell", Q-outer vs KV-outer
// section: at low reuse (few queries share a block; the dispatch rule is dispatch_path in
// msa_internal.h) each query walks its own selected blocks; no partial outputs and no
// combine are needed.
//
// Unit = (query i, group g): the 16 heads of the group against each selected block
// of the (deduplicated, causally filtered) list, with an online softmax across the
// blocks.  The MMAs run transposed so that tcgen05 sees M = 128 (keys, then D) and
// N = 16 (the heads):
//   S^T[key][h] = K_b[key][:] . Q[h][:]     (A = K_b, K-major; B = Q, K-major)
//   O^T[d][h]  += V_b[:][d] . P^T[:][h]     (A = V_b read MN-major; B = P^T, K-major)
// S^T and the block's O^T live in tensor memory (lane = key or d, column = head).
//
// Persistent CTAs of 192 threads, units taken round-robin in group-major order (all units
// of group 0, then group 1, ...): at any moment the CTAs read one group's blocks, whose
// repeated ones (a fraction of 163 MB on the low-reuse workload) the L2 can hold; in
// query-major order the four groups' 654 MB competed for it.  Warp roles:
//   warp 0       TMA producer: Q of each unit (two 2 KB boxes, double-buffered) and
//                K_b, V_b of every selected block through a ring of six 32 KB slots
//                (K freed after its S MMA, V after its P V MMA),
//                one 32 KB box per tensor through a tensor-map view that keeps both
//                halves of each 256-byte row in one request burst
//   warp 1       TMEM allocation (64 columns: S[0], S[1], O) and MMA issue: S^T of
//                item x + 1 is issued before P V of item x (one issuing thread: a second
//                one lets S run ahead and queue in front of the P V the softmax warps
//                wait for, which measured slower)
//   warps 2-5    one warpgroup, thread = key (for S) and = d (for O): per block the
//                per-head max and sum over the 128 keys (warp shuffles + shared
//                memory), P^T (bf16) into shared memory in the MMA's B layout, and the
//                running output o[h] (its column d) rescaled by 2^(m_old - m_new)
// The causal limit only matters in the query's own block (keys > pos(i) get p = 0).
//
// E4M3 inputs (per-tensor descales): S^T on kind::f8f6f4 (K-major, 32 elements per MMA),
// q and k descales folded into the softmax scale; V arrives as E4M3 and the softmax warps
// widen it (exact) into one of two f16 buffers in the bf16 V layout at the start of the
// block, while S is computed; P^T is written as f16 and P V runs on f16; the v descale
// scales the output.  (A whole-tensor f16 copy of V, as the KV-outer path uses, would
// double the V bytes of a low-reuse call.)
//
// Few units (decode-size N): each unit's list is split into S contiguous chunks of its
// valid blocks, and a work item is (unit, chunk), so that up to S times more SMs work.
// An item ends with its unnormalised output o (fp32 [16 heads][128]) and (m, l) per
// head in a workspace; the warpgroup that finishes a unit's last item (a counter per
// unit, incremented after a GPU-scope fence) merges the S partials in chunk order:
// O = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s, LSE = ln 2 (M + log2 of the
// denominator).  The merge order is fixed, so results do not depend on timing.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "msa_internal.h"
#include "ptx.cuh"

namespace msa {
namespace {

constexpr int kThreads = 192;
constexpr int kSlots = 6;                // K/V ring: K of item x in slot 2x % 6, V in slot (2x + 1) % 6
constexpr uint32_t kTmemCols = 64;
constexpr uint32_t kVhBytes = 32768;     // one 128 x 128 block of 16-bit V

// Shared-memory layout per input type.  E4M3: 16 KB ring slots (one E4M3 block) and two
// f16 V blocks, into which the softmax warps widen each block's V for the P V MMA.
template <bool kFp8>
struct QoLay {
  static constexpr uint32_t kSlot = kFp8 ? 16384 : 32768;  // one 128 x 128 K or V block as loaded
  static constexpr uint32_t kOffKV = 0;
  static constexpr uint32_t kOffVh = kSlots * kSlot;
  static constexpr uint32_t kOffQ = kOffVh + (kFp8 ? 2 * kVhBytes : 0);  // 2 x 4 KB
  static constexpr uint32_t kOffP = kOffQ + 8192;                        // 4 KB
  static constexpr uint32_t kOffRed = kOffP + 4096;  // [max, sum][2 blocks][16 heads][4 warps] floats
  static constexpr uint32_t kOffCtl = kOffRed + 1024;
  static constexpr uint32_t kSmemBytes = kOffCtl + 256 + 1024;
};
static_assert(QoLay<false>::kSmemBytes <= 232448 && QoLay<true>::kSmemBytes <= 232448, "shared memory");

enum {
  B_FULL0 = 0, B_EMPTY0 = 6, B_QFULL0 = 12, B_QEMPTY0 = 14, B_SFULL0 = 16, B_SFREE0 = 18, B_PREADY = 20,
  B_PVDONE = 21, B_COUNT = 22
};
static_assert(8 * B_COUNT + 4 <= 256, "control area");

struct QoParams {
  const int32_t* blist;
  const int32_t* counts;  // CSR row counts: how many queries chose each (group, block)
  const SchedHeader* hdr;
  SchedHeader* hdr_w;
  __nv_bfloat16* O;
  float* LSE;
  int N, Lkv, Hq, Hkv, topK, nblocks;
  float sl2;  // scale * log2(e) (E4M3: * q descale * k descale)
  float v_descale;  // E4M3: the output's factor (1 for bf16)
  int force_path;
  int splits;       // chunks per unit (1: no splitting)
  float* qs_o;      // [items][16][128] partial outputs (splits > 1)
  float2* qs_ml;    // [items][16] (m, l)
  int32_t* qs_cnt;  // [units] finished chunks, zero at launch
};

// Chunk sp of the unit's nb valid blocks (list order): [lo, hi)
__device__ __forceinline__ void chunk_range(int nb, int sp, int S, int& lo, int& hi) {
  lo = nb * sp / S;
  hi = nb * (sp + 1) / S;
}

__device__ __forceinline__ void flag_timeout(SchedHeader* hdr) { atomicOr(&hdr->status, kStatusTimeout); }

// Valid block ids of unit u's list (topK <= 64), in list order: returns their count;
// the k-th id is held by lane k % 32 in ids[k / 32] (read it with block_at).
struct UnitIds {
  int ids[2];
};
__device__ __forceinline__ int unit_blocks(const QoParams& p, int64_t u, int lane, UnitIds& out) {
  const int32_t* lst = p.blist + u * p.topK;
  int cnt = 0;
  out.ids[0] = out.ids[1] = -1;
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const int k = 32 * c + lane;
    int b = k < p.topK ? lst[k] : -1;
    if (!dbg_ok(b >= -1 && b < p.nblocks, &p.hdr_w->status)) b = -1;  // (bounds-checked build)
    const unsigned m = __ballot_sync(0xffffffffu, b >= 0);
    // compaction: the valid id of lane src goes to slot cnt + (valid lanes below src)
    for (int src = 0; src < 32; ++src) {
      const int v = __shfl_sync(0xffffffffu, b, src);
      if ((m >> src) & 1u) {
        const int dst = cnt + __popc(m & ((1u << src) - 1u));
        if ((dst & 31) == lane) {
          if (dst < 32) out.ids[0] = v;
          else out.ids[1] = v;
        }
      }
    }
    cnt += __popc(m);
  }
  return cnt;
}
__device__ __forceinline__ int block_at(const UnitIds& ids, int k) {
  const int lo = __shfl_sync(0xffffffffu, ids.ids[0], k & 31);
  const int hi = __shfl_sync(0xffffffffu, ids.ids[1], k & 31);
  return k < 32 ? lo : hi;
}

// Reduce 16 per-lane values (one per head) over the 32 lanes of a warp with 16 shuffles:
// at each step a lane keeps half of its values and receives the partner's partial of
// that half, so after 5 steps lane l holds the full result for head (l >> 1) % 16.
template <bool kMax>
__device__ __forceinline__ float warp_reduce16(const float (&v)[16], int lane) {
  auto op = [](float a, float b) { return kMax ? fmaxf(a, b) : a + b; };
  float a[8], b[4], c[2];
  bool up = lane & 16;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float keep = up ? v[j + 8] : v[j], send = up ? v[j] : v[j + 8];
    a[j] = op(keep, __shfl_xor_sync(0xffffffffu, send, 16));
  }
  up = lane & 8;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float keep = up ? a[j + 4] : a[j], send = up ? a[j] : a[j + 4];
    b[j] = op(keep, __shfl_xor_sync(0xffffffffu, send, 8));
  }
  up = lane & 4;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const float keep = up ? b[j + 2] : b[j], send = up ? b[j] : b[j + 2];
    c[j] = op(keep, __shfl_xor_sync(0xffffffffu, send, 4));
  }
  up = lane & 2;
  float d = op(up ? c[1] : c[0], __shfl_xor_sync(0xffffffffu, up ? c[0] : c[1], 2));
  return op(d, __shfl_xor_sync(0xffffffffu, d, 1));
}

// E4M3 V block (TMA layout: 128 keys x 128 bytes, 16-byte chunks swizzled by key % 8) -> f16
// in the layout the bf16 P V MMA reads ([key / 8][d / 64][key % 8][64], 128-byte swizzle).
// Thread `key` converts its key's row (exact: every E4M3 value is an f16 value).
__device__ __forceinline__ void widen_v_row(const uint8_t* src, uint8_t* dst, int key) {
  const uint8_t* row = src + key * 128;
  uint8_t* base = dst + (key >> 3) * 2048 + (key & 7) * 128;
#pragma unroll
  for (int j = 0; j < 8; ++j) {  // d = 16 j .. 16 j + 15
    const uint4 w = *reinterpret_cast<const uint4*>(row + ((j ^ (key & 7)) << 4));
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
    uint32_t h[8];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h[2 * q]) : "h"(static_cast<uint16_t>(ws[q] & 0xFFFFu)));
      asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h[2 * q + 1]) : "h"(static_cast<uint16_t>(ws[q] >> 16)));
    }
    uint8_t* half = base + (j >> 2) * 1024;
    const int c0 = (2 * j) & 7;
    *reinterpret_cast<uint4*>(half + ((c0 ^ (key & 7)) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(half + (((c0 + 1) ^ (key & 7)) << 4)) = make_uint4(h[4], h[5], h[6], h[7]);
  }
}

// kSplit: the instance for split units (p.splits > 1); the other one is the plain
// per-unit kernel (p.splits is 1 there and never read).  kFp8: E4M3 Q / K / V.
template <bool kSplit, bool kFp8>
__global__ void __launch_bounds__(kThreads, 1)
q_outer_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const QoParams p) {
  griddep_wait();
  griddep_launch();
  const int path = p.force_path ? p.force_path : p.hdr->path;
  if (path != kPathQOuter) return;
  using L = QoLay<kFp8>;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw_u & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sb = raw_u + pad;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffCtl);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffCtl + 8 * B_COUNT);
  float* red = reinterpret_cast<float*>(smem + L::kOffRed);  // [2][4 warps][16 heads]
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t units = static_cast<int64_t>(p.N) * p.Hkv;
  const int S = kSplit ? p.splits : 1;
  const int64_t nitems = units * S;

  if (tid == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(bar(B_FULL0 + s), 1);
      mbar_init(bar(B_EMPTY0 + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_QFULL0 + s), 1);
      mbar_init(bar(B_QEMPTY0 + s), 1);
      mbar_init(bar(B_SFULL0 + s), 1);
      mbar_init(bar(B_SFREE0 + s), 128);
    }
    mbar_init(bar(B_PREADY), 128);
    mbar_init(bar(B_PVDONE), 1);
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) { tma_prefetch_desc(&tmQ); tma_prefetch_desc(&tmK); tma_prefetch_desc(&tmV); }
    // Q and the K/V of blocks that several queries chose stay in L2 (evict-last) for their
    // next reader; a block only one query chose streams through (evict-first), so it does
    // not push the shared ones out.  (With one policy for all, the L2 caught 13% of the
    // repeated reads: 937 MB from DRAM against 654 MB of distinct K/V on the low-reuse
    // workload.)
    const uint64_t pol = policy_evict_normal(), pol_once = policy_evict_first(), pol_shared = policy_evict_last();
    bool ok = true;
    int item = 0, nu = 0;
    for (int64_t x = blockIdx.x; x < nitems && ok; x += gridDim.x) {
      const int64_t u = kSplit ? x / S : x;
      const int gu = static_cast<int>(u / p.N), iu = static_cast<int>(u % p.N);  // group-major order
      UnitIds mine;
      const int nb = unit_blocks(p, static_cast<int64_t>(iu) * p.Hkv + gu, lane, mine);
      int k_lo = 0, k_hi = nb;
      if constexpr (kSplit) chunk_range(nb, static_cast<int>(x % S), S, k_lo, k_hi);
      if (k_hi == k_lo) continue;
      const int i = iu, g = gu;
      const int qb = nu & 1;
      if (lane == 0) {
        // Q buffer qb was last read by the S MMAs of unit nu - 2
        if (nu >= 2) ok = mbar_wait(bar(B_QEMPTY0 + qb), ((nu >> 1) - 1) & 1);
        if (ok) {
          const uint32_t dq = sb + L::kOffQ + qb * 4096;
          if constexpr (kFp8) {
            // E4M3: the 16 heads' 128-byte rows in one box
            mbar_expect_tx(bar(B_QFULL0 + qb), 2048);
            tma_load_3d(dq, &tmQ, 0, g * kGroup, i, bar(B_QFULL0 + qb), pol);
          } else {
            mbar_expect_tx(bar(B_QFULL0 + qb), 4096);
            tma_load_3d(dq, &tmQ, 0, g * kGroup, i, bar(B_QFULL0 + qb), pol);
            tma_load_3d(dq + 2048, &tmQ, 64, g * kGroup, i, bar(B_QFULL0 + qb), pol);
          }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      for (int k = k_lo; k < k_hi && ok; ++k, ++item) {
        const int b = block_at(mine, k);
        if (lane == 0) {
          const uint64_t pol_kv = p.counts[g * p.nblocks + b] > 1 ? pol_shared : pol_once;
          // one box per tensor: the whole 128 x 128 block, both halves of each 256-byte row
          // fetched together, laid out [key / 8][D half][key % 8][64].  A slot is reused once
          // the MMA that read it (S for K, P V for V) is done; slots free in ring order.
#pragma unroll
          for (int t = 0; t < 2 && ok; ++t) {
            const int n = 2 * item + t, sl = n % kSlots;
            if (n >= kSlots) ok = mbar_wait(bar(B_EMPTY0 + sl), ((n / kSlots) - 1) & 1);
            if (ok) {
              const uint32_t fb = bar(B_FULL0 + sl);
              mbar_expect_tx(fb, L::kSlot);
              if constexpr (kFp8)  // 128 keys x 128 bytes
                tma_load_3d(sb + L::kOffKV + sl * L::kSlot, t ? &tmV : &tmK, 0, g, b * kBlock, fb, pol_kv);
              else
                tma_load_5d(sb + L::kOffKV + sl * L::kSlot, t ? &tmV : &tmK, 0, 0, 0, g, b * (kBlock / 8), fb, pol_kv);
            }
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
      ++nu;
    }
    if (!ok && lane == 0) flag_timeout(p.hdr_w);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    // S^T: M 128 keys, N 16 heads, both operands K-major (128-byte swizzle)
    constexpr uint32_t idesc_s = kFp8 ? idesc_f8(128, 16, 0, 0) : idesc_f16(128, 16, 1, 1, 0, 0);
    // O^T: M 128 (D), N 16 heads; A = V_b read MN-major, B = P^T K-major (E4M3: both f16)
    constexpr uint32_t idesc_o = kFp8 ? idesc_f16(128, 16, 0, 0, 1, 0) : idesc_f16(128, 16, 1, 1, 1, 0);
    bool ok = true;
    int item = 0, nu = 0, pending = -1;
    auto issue_pv = [&](int x) -> bool {
      const int vn = 2 * x + 1, vs = vn % kSlots;
      // (E4M3: the softmax warps waited for the slot, widened it, and are done with it)
      if (!kFp8 && !mbar_wait(bar(B_FULL0 + vs), (vn / kSlots) & 1)) return false;
      if (!mbar_wait(bar(B_PREADY), x & 1)) return false;
      tc_fence_after();
      if constexpr (kFp8) mbar_arrive(bar(B_EMPTY0 + vs));
      const uint32_t va = kFp8 ? sb + L::kOffVh + (x & 1) * kVhBytes : sb + L::kOffKV + vs * L::kSlot;
      const uint32_t pa = sb + L::kOffP;
#pragma unroll
      for (int k = 0; k < 8; ++k)
        mma_f16_ss(tmem + 32, smem_desc(va + k * 4096, 1024, 2048, 2),
                   smem_desc(pa + (k >> 2) * 2048 + (k & 3) * 32, 16, 1024, 2), idesc_o, k > 0);
      mma_commit(bar(B_PVDONE));
      if constexpr (!kFp8) mma_commit(bar(B_EMPTY0 + vs));
      return true;
    };
    for (int64_t x = blockIdx.x; x < nitems && ok; x += gridDim.x) {
      const int64_t u = kSplit ? x / S : x;
      const int gu = static_cast<int>(u / p.N), iu = static_cast<int>(u % p.N);  // group-major order
      UnitIds mine;
      const int nb = unit_blocks(p, static_cast<int64_t>(iu) * p.Hkv + gu, lane, mine);
      int k_lo = 0, k_hi = nb;
      if constexpr (kSplit) chunk_range(nb, static_cast<int>(x % S), S, k_lo, k_hi);
      if (k_hi == k_lo) continue;
      const int qb = nu & 1;
      if (lane == 0) {
        ok = mbar_wait(bar(B_QFULL0 + qb), (nu >> 1) & 1);
        for (int k = k_lo; k < k_hi && ok; ++k, ++item) {
          const int kn = 2 * item, ks = kn % kSlots, s = item & 1;
          if (!(ok = mbar_wait(bar(B_FULL0 + ks), (kn / kSlots) & 1))) break;
          // S[s] is reused: the softmax warps must have read S of item - 2
          if (item >= 2 && !(ok = mbar_wait(bar(B_SFREE0 + s), ((item >> 1) - 1) & 1))) break;
          tc_fence_after();
          const uint32_t ka = sb + L::kOffKV + ks * L::kSlot, qa = sb + L::kOffQ + qb * 4096;
          if constexpr (kFp8) {
            // E4M3: a row is one 128-byte swizzle span, 32 elements per MMA
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_f8_ss(tmem + s * 16, smem_desc(ka + kk * 32, 16, 1024, 2), smem_desc(qa + kk * 32, 16, 1024, 2),
                        idesc_s, kk > 0);
          } else {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_f16_ss(tmem + s * 16, smem_desc(ka + (kk >> 2) * 1024 + (kk & 3) * 32, 16, 2048, 2),
                         smem_desc(qa + (kk >> 2) * 2048 + (kk & 3) * 32, 16, 1024, 2), idesc_s, kk > 0);
          }
          mma_commit(bar(B_SFULL0 + s));
          mma_commit(bar(B_EMPTY0 + ks));
          if (k == k_hi - 1) mma_commit(bar(B_QEMPTY0 + qb));
          if (pending >= 0 && !(ok = issue_pv(pending))) break;
          pending = item;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      ++nu;
    }
    if (lane == 0 && ok && pending >= 0) ok = issue_pv(pending);
    if (!ok && lane == 0) flag_timeout(p.hdr_w);
  } else {
    // ------------------------------------------------------------ softmax + output (warps 2-5)
    const int q4 = warp & 3;           // TMEM lane quadrant of this warp
    const int key = 32 * q4 + lane;    // TMEM lane = key of S^T and d of O^T
    const uint32_t lane_base = static_cast<uint32_t>(32 * q4) << 16;
    const uint32_t bar_id = 1;
    const float kLn2 = 0.6931471805599453f;
    bool ok = true;
    int item = 0;
    volatile int* last_flag = reinterpret_cast<volatile int*>(smem + L::kOffCtl + 192);
    float* mscr = reinterpret_cast<float*>(smem + L::kOffP);  // merge scratch (P is free then)
    static_assert((3 * kQSplitMax + 2) * kGroup * 4 <= 4096, "merge scratch");
    // split item x of unit u done: store its partial; the last of the unit's chunks merges
    auto finish_split = [&](int64_t x, int64_t u, __nv_bfloat16* Orow, float* lse_out, const float (&m)[kGroup],
                            const float (&l)[kGroup], const float (&o)[kGroup]) {
      float* po = p.qs_o + x * (kGroup * kHeadDim);
#pragma unroll
      for (int h = 0; h < kGroup; ++h) po[h * kHeadDim + key] = o[h];
      if (key < kGroup) {
        float mk = m[0], lk = l[0];
#pragma unroll
        for (int h = 1; h < kGroup; ++h)
          if (key == h) { mk = m[h]; lk = l[h]; }
        p.qs_ml[x * kGroup + key] = make_float2(mk, lk);
      }
      // every thread's stores come before the counting thread's fence (grid-barrier pattern)
      named_bar_sync(bar_id, 128);
      if (tid == 64) {
        __threadfence();
        *last_flag = atomicAdd(p.qs_cnt + u, 1) == S - 1;
      }
      named_bar_sync(bar_id, 128);
      if (!*last_flag) return;
      __threadfence();
      const int64_t x0 = u * S;
      // (m, l) of every (chunk, head) -> weights 2^(m - M) per chunk and the denominator
      constexpr int kPairs = kQSplitMax * kGroup;
      float* mm = mscr;                // [chunk][head]
      float* ll = mscr + kPairs;       // [chunk][head]
      float* ww = mscr + 2 * kPairs;   // [chunk][head]
      float* LL = mscr + 3 * kPairs;   // [head]
      float* MM = LL + kGroup;         // [head]
      for (int q = key; q < S * kGroup; q += 128) {
        const float2 v = __ldcg(p.qs_ml + x0 * kGroup + q);
        mm[q] = v.x;
        ll[q] = v.y;
      }
      named_bar_sync(bar_id, 128);
      if (key < kGroup) {
        float M = -INFINITY;
        for (int sp = 0; sp < S; ++sp) M = fmaxf(M, mm[sp * kGroup + key]);
        float L = 0.f;
        for (int sp = 0; sp < S; ++sp) {
          const float mv = mm[sp * kGroup + key];
          const float w = mv == -INFINITY ? 0.f : ex2(mv - M);
          ww[sp * kGroup + key] = w;
          L = fmaf(w, ll[sp * kGroup + key], L);
        }
        LL[key] = L;
        MM[key] = M;
      }
      named_bar_sync(bar_id, 128);
      const float* po0 = p.qs_o + x0 * (kGroup * kHeadDim) + key;
#pragma unroll
      for (int h0 = 0; h0 < kGroup; h0 += 4) {
        float v[4][kQSplitMax];
#pragma unroll
        for (int hh = 0; hh < 4; ++hh)
#pragma unroll
          for (int sp = 0; sp < kQSplitMax; ++sp)
            v[hh][sp] = sp < S ? __ldcg(po0 + (static_cast<int64_t>(sp) * kGroup + h0 + hh) * kHeadDim) : 0.f;
#pragma unroll
        for (int hh = 0; hh < 4; ++hh) {
          const int h = h0 + hh;
          float acc = 0.f;
#pragma unroll
          for (int sp = 0; sp < kQSplitMax; ++sp)
            if (sp < S) acc = fmaf(ww[sp * kGroup + h], v[hh][sp], acc);
          const float Lh = LL[h];
          Orow[h * kHeadDim + key] = __float2bfloat16(Lh > 0.f ? p.v_descale * acc / Lh : 0.f);
        }
      }
      if (lse_out && key < kGroup) {
        const float Lk = LL[key];
        lse_out[key] = Lk > 0.f ? (MM[key] + lg2(Lk)) * kLn2 : -INFINITY;
      }
    };
    for (int64_t x = blockIdx.x; x < nitems; x += gridDim.x) {
      const int64_t u = kSplit ? x / S : x;
      const int gu = static_cast<int>(u / p.N), iu = static_cast<int>(u % p.N);  // group-major order
      UnitIds mine;
      const int nb = unit_blocks(p, static_cast<int64_t>(iu) * p.Hkv + gu, lane, mine);
      int k_lo = 0, k_hi = nb;
      if constexpr (kSplit) chunk_range(nb, static_cast<int>(x % S), S, k_lo, k_hi);
      const int i = iu, g = gu;
      __nv_bfloat16* Orow = p.O + (static_cast<int64_t>(i) * p.Hq + g * kGroup) * kHeadDim;
      float* lse_out = p.LSE ? p.LSE + static_cast<int64_t>(i) * p.Hq + g * kGroup : nullptr;
      float m[kGroup], l[kGroup], o[kGroup], aprev[kGroup];
#pragma unroll
      for (int h = 0; h < kGroup; ++h) {
        m[h] = -INFINITY;
        l[h] = 0.f;
        o[h] = 0.f;
        aprev[h] = 0.f;
      }
      if (k_hi == k_lo) {
        if constexpr (kSplit) {
          finish_split(x, u, Orow, lse_out, m, l, o);
          named_bar_sync(bar_id, 128);  // the merge scratch and the flag are read before reuse
        } else {
#pragma unroll
          for (int h = 0; h < kGroup; ++h) Orow[h * kHeadDim + key] = __float2bfloat16(0.f);
          if (lse_out && key < kGroup) lse_out[key] = -INFINITY;
        }
        continue;
      }
      const int pos = p.Lkv - p.N + i;
      for (int k = k_lo; k < k_hi; ++k, ++item) {
        const int b = block_at(mine, k);
        const int s = item & 1;
        if constexpr (kFp8) {
          // this block's V (E4M3) -> f16 buffer item % 2, whose last reader, the P V of item - 2,
          // completed before the P V of item - 1 this warpgroup has already waited for
          const int vn = 2 * item + 1, vs = vn % kSlots;
          ok = mbar_wait(bar(B_FULL0 + vs), (vn / kSlots) & 1);
          if (!named_bar_and(bar_id, 128, ok)) { ok = false; break; }
          widen_v_row(smem + L::kOffKV + vs * L::kSlot, smem + L::kOffVh + (item & 1) * kVhBytes, key);
        }
        ok = mbar_wait(bar(B_SFULL0 + s), (item >> 1) & 1);
        if (!named_bar_and(bar_id, 128, ok)) { ok = false; break; }
        tc_fence_after();
        uint32_t sv[16];
        tmem_ld16(tmem + lane_base + s * 16, sv);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(bar(B_SFREE0 + s));
        const bool vis = b * kBlock + key <= pos;
        float x[kGroup];
#pragma unroll
        for (int h = 0; h < kGroup; ++h) x[h] = vis ? __uint_as_float(sv[h]) * p.sl2 : -INFINITY;
        // per-head maximum over the 128 keys: within the warp, then across the 4 warps
        const float mx = warp_reduce16<true>(x, lane);
        float* rb = red + (k & 1) * 64;
        if (!(lane & 1)) rb[(lane >> 1) * 4 + q4] = mx;  // [head][warp]
        named_bar_sync(bar_id, 128);
        float alpha[kGroup], pv[kGroup], mn[kGroup];
#pragma unroll
        for (int h = 0; h < kGroup; ++h) {
          const float4 w4 = reinterpret_cast<const float4*>(rb)[h];
          const float bm = fmaxf(fmaxf(w4.x, w4.y), fmaxf(w4.z, w4.w));
          mn[h] = fmaxf(m[h], bm);  // finite: the block holds at least one visible key
          alpha[h] = ex2(m[h] - mn[h]);
          pv[h] = vis ? ex2(x[h] - mn[h]) : 0.f;
        }
        // per-head sum of P over the 128 keys
        const float sm = warp_reduce16<false>(pv, lane);
        float* rs = red + 128 + (k & 1) * 64;
        if (!(lane & 1)) rs[(lane >> 1) * 4 + q4] = sm;
        // the previous block's P V: accumulate it (relative to the previous maximum), then
        // the P buffer is free for this block
        if (k > k_lo) {
          ok = mbar_wait(bar(B_PVDONE), (item - 1) & 1);
          if (!named_bar_and(bar_id, 128, ok)) { ok = false; break; }
          tc_fence_after();
          uint32_t ov[16];
          tmem_ld16(tmem + lane_base + 32, ov);
          tmem_ld_wait();
#pragma unroll
          for (int h = 0; h < kGroup; ++h) o[h] = fmaf(o[h], aprev[h], __uint_as_float(ov[h]));
        } else {
          named_bar_sync(bar_id, 128);
        }
#pragma unroll
        for (int h = 0; h < kGroup; ++h) {
          const float4 w4 = reinterpret_cast<const float4*>(rs)[h];
          const float bs = (w4.x + w4.y) + (w4.z + w4.w);
          l[h] = fmaf(l[h], alpha[h], bs);
          m[h] = mn[h];
          aprev[h] = alpha[h];
        }
        // P^T[h][key] (bf16) in the K-major 128-byte-swizzled B layout: keys 0-63 and
        // 64-127 in two 2 KB halves of 16 rows
        {
          const int half = key >> 6, kk = key & 63;
          uint8_t* pb = smem + L::kOffP + half * 2048 + (kk & 7) * 2;
#pragma unroll
          for (int h = 0; h < kGroup; ++h)
            if constexpr (kFp8)  // f16 P for the f16 V
              *reinterpret_cast<__half*>(pb + h * 128 + (((kk >> 3) ^ (h & 7)) << 4)) = __float2half_rn(pv[h]);
            else
              *reinterpret_cast<__nv_bfloat16*>(pb + h * 128 + (((kk >> 3) ^ (h & 7)) << 4)) = __float2bfloat16(pv[h]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(B_PREADY));
      }
      if (!ok) break;
      // the unit's last P V
      ok = mbar_wait(bar(B_PVDONE), (item - 1) & 1);
      if (!named_bar_and(bar_id, 128, ok)) { ok = false; break; }
      tc_fence_after();
      uint32_t ov[16];
      tmem_ld16(tmem + lane_base + 32, ov);
      tmem_ld_wait();
      tc_fence_before();
#pragma unroll
      for (int h = 0; h < kGroup; ++h) o[h] = fmaf(o[h], aprev[h], __uint_as_float(ov[h]));
      if constexpr (kSplit) {
        finish_split(x, u, Orow, lse_out, m, l, o);
      } else {
#pragma unroll
        for (int h = 0; h < kGroup; ++h) Orow[h * kHeadDim + key] = __float2bfloat16(p.v_descale * o[h] / l[h]);
        if (lse_out && key < kGroup) {
          float mk = m[0], lk = l[0];
#pragma unroll
          for (int h = 1; h < kGroup; ++h)
            if (key == h) { mk = m[h]; lk = l[h]; }
          lse_out[key] = (mk + lg2(lk)) * kLn2;
        }
      }
      // all 128 threads are past this item's reads of `red` (and of the merge scratch and
      // flag) before the next item writes them
      named_bar_sync(bar_id, 128);
    }
    if (!ok && tid == 64) flag_timeout(p.hdr_w);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_q_outer(const msa_schedule* s, const void* Q, const void* K, const void* V, int Hq, float scale,
                           void* O, float* LSE, int force_path, cudaStream_t st, bool fp8, float qk_descale,
                           float v_descale) {
  if (s->topK > 64) return cudaErrorInvalidValue;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  CUtensorMap tmQ, tmK, tmV;
  if (fp8) {
    // E4M3 Q [N][Hq][128]: box = the 128-byte rows of the 16 heads of one group of one query;
    // K, V [Lkv][Hkv][128]: box = one 128-key block of one group, 128 bytes per key
    const uint64_t qd[3] = {kHeadDim, static_cast<uint64_t>(Hq), static_cast<uint64_t>(s->N)};
    const uint64_t qs[2] = {kHeadDim, static_cast<uint64_t>(Hq) * kHeadDim};
    const uint32_t qbox[3] = {128, kGroup, 1};
    if (!encode_tmap(&tmQ, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, Q, qd, qs, qbox, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
    const uint64_t kd[3] = {kHeadDim, static_cast<uint64_t>(s->Hkv), static_cast<uint64_t>(s->nblocks) * kBlock};
    const uint64_t ks[2] = {kHeadDim, static_cast<uint64_t>(s->Hkv) * kHeadDim};
    const uint32_t kbox[3] = {128, 1, kBlock};
    if (!encode_tmap(&tmK, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, K, kd, ks, kbox, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
    if (!encode_tmap(&tmV, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, V, kd, ks, kbox, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  } else {
  {
    // Q [N][Hq][128] bf16: box = 64 columns of the 16 heads of one group of one query
    const uint64_t dims[3] = {kHeadDim, static_cast<uint64_t>(Hq), static_cast<uint64_t>(s->N)};
    const uint64_t strides[2] = {kHeadDim * 2, static_cast<uint64_t>(Hq) * kHeadDim * 2};
    const uint32_t box[3] = {64, kGroup, 1};
    if (!encode_tmap(&tmQ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, Q, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  {
    // K, V [Lkv][Hkv][128] bf16 viewed as (d % 64, key % 8, d / 64, group, key / 8): one box =
    // one 128-key block of one group (32 KB), laid out [key / 8][d / 64][key % 8][64]: 8-row
    // groups of 128-byte rows 2048 bytes apart, the second D half 1024 bytes after the first
    const uint64_t row = static_cast<uint64_t>(s->Hkv) * kHeadDim * 2;  // bytes per key
    const uint64_t dims[5] = {64, 8, 2, static_cast<uint64_t>(s->Hkv), static_cast<uint64_t>(s->nblocks) * (kBlock / 8)};
    const uint64_t strides[4] = {row, 128, kHeadDim * 2, 8 * row};
    const uint32_t box[5] = {64, 8, 2, 1, kBlock / 8};
    if (!encode_tmap(&tmK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, K, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
    if (!encode_tmap(&tmV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, V, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  }
  static std::atomic<uint64_t> attr_done[4];
  {
    cudaError_t e = cudaSuccess;
    int i = 0;
    for (auto* k : {q_outer_kernel<false, false>, q_outer_kernel<true, false>})
      if (e == cudaSuccess) e = set_smem_limit(k, static_cast<int>(QoLay<false>::kSmemBytes), attr_done[i++]);
    for (auto* k : {q_outer_kernel<false, true>, q_outer_kernel<true, true>})
      if (e == cudaSuccess) e = set_smem_limit(k, static_cast<int>(QoLay<true>::kSmemBytes), attr_done[i++]);
    if (e != cudaSuccess) return e;
  }
  QoParams p;
  p.blist = s->d.blist;
  p.counts = s->d.counts;
  p.hdr = s->d.hdr;
  p.hdr_w = s->d.hdr;
  p.O = static_cast<__nv_bfloat16*>(O);
  p.LSE = LSE;
  p.N = s->N;
  p.Lkv = s->nblocks * kBlock;
  p.Hq = Hq;
  p.Hkv = s->Hkv;
  p.topK = s->topK;
  p.nblocks = s->nblocks;
  p.sl2 = scale * qk_descale * 1.4426950408889634f;
  p.v_descale = v_descale;
  p.force_path = force_path;
  const int64_t units = static_cast<int64_t>(s->N) * s->Hkv;
  // split the units' lists while the units fill at most a quarter of the SMs: the
  // merge and the counter reset cost a few microseconds, which 2 or 3 chunks per unit do
  // not win back (measured: N = 16, 64 units, 2 chunks was slower than 1)
  int splits = 1;
  if (s->qs_items > 0 && units * kQSplitMin <= sms) {
    splits = static_cast<int>(sms / units);
    if (splits > kQSplitMax) splits = kQSplitMax;
    if (splits > s->topK) splits = s->topK;
    if (static_cast<int64_t>(splits) * units > s->qs_items) splits = static_cast<int>(s->qs_items / units);
    if (splits < kQSplitMin) splits = 1;
  }
  p.splits = splits;
  p.qs_o = s->d.qs_o;
  p.qs_ml = s->d.qs_ml;
  p.qs_cnt = s->d.qs_cnt;
  if (splits > 1) {
    cudaError_t e = cudaMemsetAsync(s->d.qs_cnt, 0, static_cast<size_t>(units) * sizeof(int32_t), st);
    if (e != cudaSuccess) return e;
  }
  int64_t grid = sms;
  if (grid > units * splits) grid = units * splits;
  const uint32_t smem = fp8 ? QoLay<true>::kSmemBytes : QoLay<false>::kSmemBytes;
  void (*kern)(CUtensorMap, CUtensorMap, CUtensorMap, QoParams) =
      fp8 ? (splits > 1 ? q_outer_kernel<true, true> : q_outer_kernel<false, true>)
          : (splits > 1 ? q_outer_kernel<true, false> : q_outer_kernel<false, false>);
  MSA_LAUNCH(kern, static_cast<int>(grid), kThreads, smem, st, tmQ, tmK, tmV, p);
  return cudaGetLastError();
}

}  // namespace msa
