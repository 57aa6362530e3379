// Internal declarations shared by the libmsa translation units.
#pragma once
#include <atomic>
#include <cstdint>
#include <utility>

#include <cuda.h>
#include <cuda_runtime.h>

#include "msa.h"

namespace msa {

// Launch with a programmatic dependency on the previous work in the stream (the kernel
// must start with griddep_wait(); see ptx.cuh).  After a non-kernel stream operation the
// launch is simply ordered after it.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Raises kernel `kern`'s dynamic shared-memory limit to `bytes` on the current device.
// Function attributes belong to each device's context, so every device a process launches
// on gets its own call; `done` (one per call site, one bit per device ordinal below 64)
// skips it afterwards.  Two threads racing on a first call both set the same value.
template <class K>
inline cudaError_t set_smem_limit(K kern, int bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev >= 0 && dev < 64 ? (1ull << dev) : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
  return e;
}

// launch_pdl inside a function returning cudaError_t: returns the launch error, if any
#define MSA_LAUNCH(...)                                               \
  do {                                                                \
    const cudaError_t launch_err_ = ::msa::launch_pdl(__VA_ARGS__);   \
    if (launch_err_ != cudaSuccess) return launch_err_;               \
  } while (0)

constexpr int kBlock = 128;      // tokens per KV block
constexpr int kHeadDim = 128;    // D
constexpr int kGroup = 16;       // G = Hq / Hkv handled by the kernels
constexpr int kTileQ = 8;        // queries per tile: 8 queries x 16 heads = 128 MMA rows
constexpr int kChunk = 32;       // queries per bitmask word of the schedule
constexpr int kWindow = 2048;    // queries per work-list window (multiple of kChunk)

// Q-outer split units: at most this many splits per unit, and only while the units
// number at most kQSplitMaxUnits (more units fill the GPU without splitting)
constexpr int kQSplitMax = 8;
constexpr int kQSplitMin = 4;
constexpr int kQSplitMaxUnits = 64;

// Partial outputs of the KV-outer path (bf16 or fp32 rows of 128, one per (CSR position,
// head of the group)): positions in aligned groups of kPartGroup = 8 -- a tile's 8 entries
// are 8 consecutive positions -- and inside a group the layout is [16-byte column chunk]
// [8 positions x 16 heads], so that the attention kernel's warp store of one column chunk
// of 32 rows (after a 32x32b TMEM load: a thread per row) covers 512 contiguous bytes, and
// the combine reads 256 contiguous bytes per (position, chunk).  Chunk c of (position p,
// head h) is the uint4 at part_index(p, h, c, chunks), chunks = 16 (bf16: 8 columns) or
// 32 (fp32: 4 columns).
constexpr int kPartGroup = 8;
__host__ __device__ __forceinline__ int64_t part_index(int64_t p, int h, int c, int chunks) {
  return ((p / kPartGroup) * chunks + c) * (kPartGroup * kGroup) + (p % kPartGroup) * kGroup + h;
}
// rows (of 128 elements) the partial workspace holds for cap positions: whole groups
__host__ __device__ __forceinline__ int64_t part_rows(int64_t cap) {
  return (cap + kPartGroup - 1) / kPartGroup * kPartGroup * kGroup;
}

constexpr int kPathKvOuter = 1;
constexpr int kPathQOuter = 2;

// The AUTO dispatch: KV-outer when 10 E - 13 nsb > 35000, in exact integers (E = CSR entries,
// i.e. distinct (query, KV head, block) triples; nsb = distinct (KV head, block) pairs).
// "Kernel optimization for MiniMax M3", Q-outer vs KV-outer section and its appendix, derives
// KV-outer when nsb / N < 2.85 from a bandwidth model of its B200 kernels and asks for the
// constant to be re-derived from the machine's own numbers.  Re-derived on GB300 from
// measurement: the step time with each path forced over 36 (dtype, context, N) points
// (bench.py --dispatch-sweep) fits T_kv - T_q = 24.3 us - 6.96 ns * E + 9.04 ns * nsb --
// the KV-outer path's fixed cost (launches, pipeline fill, the combine), the Q-outer kernel's
// per-entry cost, the KV-outer kernel's per-block cost -- and the rule picks the faster path
// at all 52 measured points (16 more shapes with Hkv 1-8, topK 4-32), where nsb / N < 2.85
// picks the slower one at 19.
__host__ __device__ constexpr int dispatch_path(int64_t entries, int64_t nsb) {
  return 10 * entries - 13 * nsb > 35000 ? kPathKvOuter : kPathQOuter;
}
// True when dispatch_path picks Q-outer for every schedule of these sizes, so the host can
// launch the Q-outer kernel alone (no KV-outer or combine launch that would only exit).
// E <= E_max = N * Hkv * topK, and a (KV head, block) row holds at most N entries, so
// nsb >= E / N and 10 E - 13 nsb <= E (10 - 13 / N) <= E_max (10 - 13 / N).  Every N = 1
// call qualifies, and at Hkv 4, topK 16 every N up to 55.
constexpr bool q_outer_certain(int64_t N, int64_t Hkv, int64_t topK) {
  return N * Hkv * topK * (10 * N - 13) <= 35000 * N;
}

constexpr int kStatusBadIndex = 1;
constexpr int kStatusTimeout = 2;
constexpr int kStatusBounds = 4;  // bounds-checked builds only

// Bounds-checked build (compiled with -DMSA_DEBUG=1 into libmsa_debug.so): every gather index
// and TMA coordinate a kernel reads from device memory (schedule arrays, tile records, query
// and block ids, combine map entries) is checked against its tensor's extent before use.  A
// value out of range sets kStatusBounds in the schedule header and the access is skipped
// (stores) or redirected to element 0 (loads, so that barrier byte counts still match); no
// trap or assert.  The release build compiles the checks away.
#ifndef MSA_DEBUG
#define MSA_DEBUG 0
#endif
#ifdef __CUDACC__
__device__ __forceinline__ bool dbg_ok(bool in_range, int32_t* status) {
  if (MSA_DEBUG && !in_range) {
    atomicOr(status, kStatusBounds);
    return false;
  }
  return true;
}
#endif

// Device-resident header written by the schedule kernels and read by the attention
// kernels (the dispatch decision never leaves the device).
struct SchedHeader {
  int32_t entries;  // E
  int32_t nsb;
  int32_t ntiles;
  int32_t path;     // AUTO choice: kPathKvOuter or kPathQOuter
  int32_t status;   // sticky kStatus* bits
  // pad[0]: the KV-outer kernel's chunk counter (cleared by the combine); pad[1]: the mark
  // pass's bad-index bit, moved into status by the row scan
  int32_t pad[3];
};

struct SchedDev {
  uint32_t* mask;        // [R][C] bit (i % 32) of word (r, i / 32): query i has an entry in row r
  uint32_t* mcopy;       // [R][C] the bitmask words as the row scan read them (it clears the bitmask)
  int32_t* rowbase;      // [R][C + 1] exclusive prefix of popcounts along each row
  int32_t* counts;       // [R]
  int32_t* offsets;      // [R + 1]
  int32_t* qlist;        // [cap_entries]
  int32_t* slot;         // [cap_entries]
  int32_t* cmap;         // [N * Hkv * topK] CSR position of list slot k, or -1
  int32_t* blist;        // [N * Hkv * topK] block id of list slot k if it is an entry, else -1
  int4* tiles;           // [cap_tiles] (row, first, count, window)
  int32_t* window_tiles; // [nW + 1]
  int32_t* segoff;       // [nW * R + 1] tiles per (window, row) segment, then their exclusive prefix
  int32_t* seg_sums;     // [nseg_blocks + 1] scan scratch: per-block sums of segment tile counts
  // Q-outer split units (few units): per work item the fp32 partial output [16][128] and
  // (m, l) per head; per unit the count of finished splits
  float* qs_o;           // [qs_items * 16 * 128]
  float2* qs_ml;         // [qs_items * 16]
  int32_t* qs_cnt;       // [N * Hkv] when qs_items > 0
  SchedHeader* hdr;
};

}  // namespace msa

struct msa_schedule {
  int N, Hkv, topK, nblocks;
  int R, C, nW;
  int qs_items;  // capacity of the Q-outer split workspace in work items (0: no splitting)
  // the bitmask and the header's pad words are zero (the last multi-kernel build cleared them),
  // so the next build needs no memset
  bool mask_clean;
  int64_t cap_entries, cap_tiles, nseg, nseg_blocks;
  void* dev_base;
  size_t dev_bytes;
  msa::SchedDev d;
  // partial-output workspace (first forward call)
  void* partial;       // bf16 or fp32 [cap_entries * G, D]: raw P V of each (entry, head) row
  float2* pstat;       // [cap_entries * G]: (m, l) of each partial row, m in base-2 units
  int partial_G;
  int partial_elem;    // bytes per element the partial buffer was sized for (2 or 4)
  void* bwd_ws;  // backward workspace (first backward call)
  void* vf16;    // E4M3 forwards: V widened to f16 [Lkv][Hkv][128] (first E4M3 call)
  cudaStream_t last_stream;
};

namespace msa {

// msa_api.cu: array sizes of a schedule, and the layout of its arrays inside one
// device buffer starting at `base` (base == nullptr only computes s->dev_bytes).
void schedule_dims(msa_schedule* s, int N, int Hkv, int topK, int nblocks);
void carve_schedule(msa_schedule* s, char* base);
// msa_api.cu: maps a CUDA error to a status and records it for msa_last_cuda_error.
msa_status_t status_from_cuda(cudaError_t e);

// schedule.cu
cudaError_t enqueue_schedule(msa_schedule* s, const int32_t* indices, cudaStream_t st);
constexpr int kSegScanBlock = 4096;  // segments per block of the segment scan

// attn_kv_outer.cu
struct KvOuterArgs {
  const msa_schedule* s;
  const void* Q;
  const void* K;
  const void* V;
  int Hq, Lkv;
  float scale;
  int force_path;  // 0 auto, 1 kv, 2 q
  int num_ctas;
  bool fp8;          // E4M3 inputs
  float qk_descale;  // q descale * k descale (1 for bf16)
  bool f32p;         // fp32 partial outputs
  int debug_flags;   // msa_fwd_opts_t.debug_flags
  const void* Vf16;  // E4M3 inputs: V widened to f16 (launch_widen_e4m3), or (p8) V^T
  bool p8;           // E4M3 P V: P in E4M3 and V^T (launch_transpose_e4m3) instead of f16
};
// Whether an E4M3 call runs the E4M3 P V (kind::f8f6f4) instance of the KV-outer kernel:
// positive scales with bf16 partials, selected by msa_fwd_opts_t.debug_flags bit 1.
inline bool kv_outer_p8(bool fp8, bool f32p, float scale, int debug_flags) {
  return fp8 && !f32p && scale > 0.f && (debug_flags & 2) != 0;
}
cudaError_t launch_kv_outer(const KvOuterArgs& a, cudaStream_t st);
// E4M3 [n] -> f16 [n], exact; n a multiple of 16
// (exits at once where the device chose the Q-outer path, which widens V in shared memory)
// E4M3 V [Lkv][Hkv][128] -> V^T [Hkv * nblocks][128 d][128 keys] (exits at once on the Q-outer path)
cudaError_t launch_transpose_e4m3(const void* v, void* vt, int Hkv, int nblocks, const SchedHeader* hdr, int force_path,
                                  cudaStream_t st);
cudaError_t launch_widen_e4m3(const void* src, void* dst, int64_t n, const SchedHeader* hdr, int force_path,
                              cudaStream_t st);

// combine.cu
cudaError_t launch_combine(const msa_schedule* s, int Hq, void* O, float* LSE, float v_descale, int force_path,
                           bool f32p, cudaStream_t st);

// attn_q_outer.cu
cudaError_t launch_q_outer(const msa_schedule* s, const void* Q, const void* K, const void* V, int Hq,
                           float scale, void* O, float* LSE, int force_path, cudaStream_t st, bool fp8 = false,
                           float qk_descale = 1.f, float v_descale = 1.f);

// select.cu: block selector R1
size_t select_workspace_bytes(int N, int Hq, int Hkv, int nblocks);
uint32_t select_smem_bytes(int nblocks, int reps);
cudaError_t launch_select_r1(const void* Q, const void* K, int N, int Lkv, int Hq, int Hkv, int topK, int32_t* indices,
                             void* workspace, cudaStream_t st);
cudaError_t launch_select_r4(const void* Q, const void* K, int N, int Lkv, int Hq, int Hkv, int topK, int32_t* indices,
                             void* workspace, cudaStream_t st);

// attn_tiles.cu: forward for lists shared by tiles of consecutive queries
cudaError_t launch_tiles(const void* Q, const void* K, const void* V, int N, int Lkv, int Hq, int Hkv,
                         const int32_t* lists, int tile, int topK, float scale, void* O, float* LSE, int32_t* status,
                         int num_ctas, cudaStream_t st);

// attn_bwd.cu: backward (dQ, dK, dV) over the schedule of the forward
constexpr int kUnitEntries = 256;  // entries per KV-stationary backward unit (32 tiles)
struct BwdArgs {
  const msa_schedule* s;
  const void* Q;
  const void* K;
  const void* V;
  const void* O;
  const void* dO;
  const float* LSE;
  void* dQ;
  void* dK;
  void* dV;
  void* workspace;  // bwd_workspace_bytes(s), 256-byte aligned
  int Hq, Lkv;
  float scale;
  int num_ctas;
  cudaEvent_t ev[3];  // optional: before / after the tcgen05 kernel, after the last kernel
};
int64_t bwd_unit_capacity(const msa_schedule* s);
size_t bwd_workspace_bytes(const msa_schedule* s);
cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t st);

// tensor maps (msa_api.cpp)
bool encode_tmap(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base, const uint64_t* dims,
                 const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle swz);

}  // namespace msa
