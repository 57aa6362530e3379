// C ABI of libmsa (declared in include/msa.h): argument checks, workspace
// ownership, tensor-map encoding and the launch sequence.  No call here
// synchronises the host except msa_schedule_query / msa_schedule_export /
// msa_schedule_destroy, and nothing aborts, traps or prints.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <mutex>
#include <new>

#include "msa_internal.h"

namespace {

thread_local int g_last_cuda = 0;

msa_status_t from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return MSA_OK;
  g_last_cuda = static_cast<int>(e);
  cudaGetLastError();  // clear a sticky-free error so the next call starts clean
  return e == cudaErrorMemoryAllocation ? MSA_ERR_OOM : MSA_ERR_CUDA;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

void load_encode() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
          cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

int device_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

msa_status_t schedule_create(int N, int Hkv, int topK, int nblocks, msa_schedule** out) {
  msa_schedule* s = new (std::nothrow) msa_schedule();
  if (!s) return MSA_ERR_OOM;
  std::memset(s, 0, sizeof(*s));
  msa::schedule_dims(s, N, Hkv, topK, nblocks);
  msa::carve_schedule(s, nullptr);
  cudaError_t e = cudaMalloc(&s->dev_base, s->dev_bytes);
  if (e != cudaSuccess) {
    delete s;
    return from_cuda(e);
  }
  msa::carve_schedule(s, static_cast<char*>(s->dev_base));
  *out = s;
  return MSA_OK;
}

msa_status_t ensure_partials(msa_schedule* s, int G, int elem = 2) {
  if (s->partial && s->partial_G == G && s->partial_elem >= elem) return MSA_OK;
  if (s->partial) {
    cudaFree(s->partial);
    s->partial = nullptr;
    s->pstat = nullptr;
  }
  const size_t rows = static_cast<size_t>(msa::part_rows(s->cap_entries)) * G / msa::kGroup;
  const size_t obytes = align_up(rows * msa::kHeadDim * elem, 256);
  void* p = nullptr;
  cudaError_t e = cudaMalloc(&p, obytes + rows * sizeof(float2));
  if (e != cudaSuccess) return from_cuda(e);
  s->partial = p;
  s->pstat = reinterpret_cast<float2*>(static_cast<char*>(p) + obytes);
  s->partial_G = G;
  s->partial_elem = elem;
  return MSA_OK;
}

}  // namespace

namespace msa {
// Carves the schedule's device arrays out of one allocation.
struct Carver {
  size_t off = 0;
  char* base = nullptr;
  template <class T>
  T* take(size_t count) {
    const size_t o = off;
    off = align_up(off + count * sizeof(T), 256);
    return base ? reinterpret_cast<T*>(base + o) : nullptr;
  }
};

void carve_schedule(msa_schedule* s, char* base) {
  Carver c;
  c.base = base;
  msa::SchedDev& d = s->d;
  d.mask = c.take<uint32_t>(static_cast<size_t>(s->R) * s->C);
  d.mcopy = c.take<uint32_t>(static_cast<size_t>(s->R) * s->C);
  d.rowbase = c.take<int32_t>(static_cast<size_t>(s->R) * (s->C + 1));
  d.counts = c.take<int32_t>(s->R);
  d.offsets = c.take<int32_t>(static_cast<size_t>(s->R) + 1);
  d.qlist = c.take<int32_t>(s->cap_entries);
  d.slot = c.take<int32_t>(s->cap_entries);
  d.cmap = c.take<int32_t>(s->cap_entries);
  d.blist = c.take<int32_t>(s->cap_entries);
  d.tiles = c.take<int4>(s->cap_tiles);
  d.window_tiles = c.take<int32_t>(static_cast<size_t>(s->nW) + 1);
  d.segoff = c.take<int32_t>(static_cast<size_t>(s->nseg) + 1);
  d.seg_sums = c.take<int32_t>(static_cast<size_t>(s->nseg_blocks) + 1);
  d.qs_o = c.take<float>(static_cast<size_t>(s->qs_items) * kGroup * kHeadDim);
  d.qs_ml = c.take<float2>(static_cast<size_t>(s->qs_items) * kGroup);
  d.qs_cnt = c.take<int32_t>(s->qs_items > 0 ? static_cast<size_t>(s->N) * s->Hkv : 0);
  d.hdr = c.take<msa::SchedHeader>(1);
  s->dev_bytes = c.off;
}

// Sizes of the schedule's arrays for (N, Hkv, topK, nblocks).
void schedule_dims(msa_schedule* s, int N, int Hkv, int topK, int nblocks) {
  s->N = N;
  s->Hkv = Hkv;
  s->topK = topK;
  s->nblocks = nblocks;
  s->R = Hkv * nblocks;
  s->C = (N + kChunk - 1) / kChunk;
  s->nW = (N + kWindow - 1) / kWindow;
  s->cap_entries = static_cast<int64_t>(N) * Hkv * topK;
  s->nseg = static_cast<int64_t>(s->nW) * s->R;
  s->nseg_blocks = (s->nseg + kSegScanBlock - 1) / kSegScanBlock;
  const int64_t nonempty = s->nseg < s->cap_entries ? s->nseg : s->cap_entries;
  s->cap_tiles = s->cap_entries / kTileQ + nonempty + 1;
  const int64_t units = static_cast<int64_t>(N) * Hkv;
  s->qs_items = units <= kQSplitMaxUnits ? static_cast<int>(units * kQSplitMax) : 0;
}

msa_status_t status_from_cuda(cudaError_t e) { return from_cuda(e); }

bool encode_tmap(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base, const uint64_t* dims,
                 const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle swz) {
  std::call_once(g_encode_once, load_encode);
  if (!g_encode) return false;
  cuuint64_t gd[5], gs[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
  }
  for (int i = 0; i < rank - 1; ++i) gs[i] = strides_bytes[i];
  CUresult r = g_encode(m, dt, static_cast<cuuint32_t>(rank), const_cast<void*>(base), gd, gs, bx, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}
}  // namespace msa

extern "C" {

void msa_fwd_opts_init(msa_fwd_opts_t* opts) {
  if (!opts) return;
  std::memset(opts, 0, sizeof(*opts));
  opts->path = MSA_PATH_AUTO;
  opts->q_descale = opts->k_descale = opts->v_descale = 1.f;
}

msa_status_t msa_build_schedule(const int32_t* indices, int N, int Hkv, int topK, int nblocks, cudaStream_t stream,
                                msa_schedule_t* inout) {
  if (!indices || !inout) return MSA_ERR_INVALID_ARG;
  if (N < 1 || Hkv < 1 || topK < 1 || nblocks < 1) return MSA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(nblocks) * msa::kBlock > INT32_MAX) return MSA_ERR_CAPACITY;
  if (static_cast<int64_t>(N) > static_cast<int64_t>(nblocks) * msa::kBlock) return MSA_ERR_INVALID_ARG;
  if (topK > 64) return MSA_ERR_UNSUPPORTED;
  const int64_t rows16 = static_cast<int64_t>(N) * Hkv * topK * msa::kGroup;
  if (rows16 > INT32_MAX || static_cast<int64_t>(Hkv) * nblocks > INT32_MAX) return MSA_ERR_CAPACITY;
  msa_schedule* s = *inout;
  if (s) {
    if (s->N != N || s->Hkv != Hkv || s->topK != topK || s->nblocks != nblocks) return MSA_ERR_INVALID_ARG;
  } else {
    msa_status_t st = schedule_create(N, Hkv, topK, nblocks, &s);
    if (st != MSA_OK) return st;
  }
  cudaError_t e = msa::enqueue_schedule(s, indices, stream);
  s->last_stream = stream;
  if (!*inout) {
    if (e != cudaSuccess) {
      cudaFree(s->dev_base);
      delete s;
      return from_cuda(e);
    }
    *inout = s;
  }
  return from_cuda(e);
}

msa_status_t msa_sparse_attn_fwd(msa_tensor_t Q, msa_tensor_t K, msa_tensor_t V, msa_schedule_t s, void* O,
                                 float* LSE, float scale, const msa_fwd_opts_t* opts) {
  msa_fwd_opts_t def;
  if (!opts) {
    msa_fwd_opts_init(&def);
    opts = &def;
  }
  if (!s || !Q.ptr || !K.ptr || !V.ptr || !O) return MSA_ERR_INVALID_ARG;
  if (!aligned16(Q.ptr) || !aligned16(K.ptr) || !aligned16(V.ptr) || !aligned16(O)) return MSA_ERR_INVALID_ARG;
  if (Q.n != s->N || K.n != static_cast<int64_t>(s->nblocks) * msa::kBlock || V.n != K.n) return MSA_ERR_INVALID_ARG;
  if (K.h != s->Hkv || V.h != s->Hkv || Q.h < 1 || Q.h % K.h != 0) return MSA_ERR_INVALID_ARG;
  if (Q.d != K.d || K.d != V.d) return MSA_ERR_INVALID_ARG;
  if (Q.dtype != K.dtype || K.dtype != V.dtype) return MSA_ERR_UNSUPPORTED;
  if (Q.d != msa::kHeadDim || Q.h / K.h != msa::kGroup) return MSA_ERR_UNSUPPORTED;
  if (Q.dtype != MSA_BF16 && Q.dtype != MSA_FP8_E4M3) return MSA_ERR_UNSUPPORTED;
  if (!std::isfinite(scale)) return MSA_ERR_INVALID_ARG;
  if (opts->path != MSA_PATH_AUTO && opts->path != MSA_PATH_KV_OUTER && opts->path != MSA_PATH_Q_OUTER)
    return MSA_ERR_INVALID_ARG;
  const bool fp8 = Q.dtype == MSA_FP8_E4M3;
  if (fp8 && !(std::isfinite(opts->q_descale) && std::isfinite(opts->k_descale) && std::isfinite(opts->v_descale) &&
               opts->q_descale > 0.f && opts->k_descale > 0.f && opts->v_descale > 0.f))
    return MSA_ERR_INVALID_ARG;
  if (opts->partials_fp32 != 0 && opts->partials_fp32 != 1) return MSA_ERR_INVALID_ARG;
  const bool f32p = opts->partials_fp32 == 1;
  msa_status_t st = ensure_partials(s, msa::kGroup, f32p ? 4 : 2);
  if (st != MSA_OK) return st;
  // AUTO where the sizes alone fix the device's choice (decode sizes): the Q-outer kernel only
  const int force = opts->path != MSA_PATH_AUTO ? static_cast<int>(opts->path)
                    : msa::q_outer_certain(s->N, s->Hkv, s->topK) ? msa::kPathQOuter : 0;
  const float qk_descale = fp8 ? opts->q_descale * opts->k_descale : 1.f;
  const float v_descale = fp8 ? opts->v_descale : 1.f;
  const cudaStream_t stream = opts->stream;
  int ctas = opts->num_ctas > 0 ? opts->num_ctas : device_sms();
  if (ctas < 1) return MSA_ERR_CUDA;
  const int Hq = static_cast<int>(Q.h);
  const int64_t v_elems = static_cast<int64_t>(K.n) * K.h * K.d;
  if (fp8 && force != msa::kPathQOuter && !s->vf16) {
    // the f16 copy of E4M3 V (first E4M3 call of this schedule; later calls allocate nothing)
    void* p = nullptr;
    cudaError_t ea = cudaMalloc(&p, static_cast<size_t>(v_elems) * 2);
    if (ea != cudaSuccess) return from_cuda(ea);
    s->vf16 = p;
  }
  cudaError_t e;
  if (opts->stage_events[0] && (e = cudaEventRecord(opts->stage_events[0], stream))) return from_cuda(e);
  const bool p8 = msa::kv_outer_p8(fp8, f32p, scale, opts->debug_flags);
  if (fp8 && force != msa::kPathQOuter) {
    // the KV-outer kernel's V: widened to f16, or (E4M3 P V) transposed per block
    e = p8 ? msa::launch_transpose_e4m3(V.ptr, s->vf16, s->Hkv, s->nblocks, s->d.hdr, force, stream)
           : msa::launch_widen_e4m3(V.ptr, s->vf16, v_elems, s->d.hdr, force, stream);
    if (e) return from_cuda(e);
  }
  msa::KvOuterArgs a{s, Q.ptr, K.ptr, V.ptr, Hq, s->nblocks * msa::kBlock, scale, force, ctas, fp8, qk_descale, f32p,
                     opts->debug_flags, s->vf16, p8};
  if ((e = msa::launch_kv_outer(a, stream))) return from_cuda(e);
  if (opts->stage_events[1] && (e = cudaEventRecord(opts->stage_events[1], stream))) return from_cuda(e);
  if (force != msa::kPathQOuter && (e = msa::launch_combine(s, Hq, O, LSE, v_descale, force, f32p, stream)))
    return from_cuda(e);
  if ((e = msa::launch_q_outer(s, Q.ptr, K.ptr, V.ptr, Hq, scale, O, LSE, force, stream, fp8, qk_descale, v_descale)))
    return from_cuda(e);
  if (opts->stage_events[2] && (e = cudaEventRecord(opts->stage_events[2], stream))) return from_cuda(e);
  s->last_stream = stream;
  return MSA_OK;
}

msa_status_t msa_sparse_attn_bwd(msa_tensor_t Q, msa_tensor_t K, msa_tensor_t V, const void* O, const void* dO,
                                 const float* LSE, msa_schedule_t s, void* dQ, void* dK, void* dV, float scale,
                                 const msa_fwd_opts_t* opts) {
  msa_fwd_opts_t def;
  if (!opts) {
    msa_fwd_opts_init(&def);
    opts = &def;
  }
  if (!s || !Q.ptr || !K.ptr || !V.ptr || !O || !dO || !LSE || !dQ || !dK || !dV) return MSA_ERR_INVALID_ARG;
  for (const void* p : {Q.ptr, K.ptr, V.ptr, O, dO, static_cast<const void*>(LSE), static_cast<const void*>(dQ),
                        static_cast<const void*>(dK), static_cast<const void*>(dV)})
    if (!aligned16(p)) return MSA_ERR_INVALID_ARG;
  if (Q.n != s->N || K.n != static_cast<int64_t>(s->nblocks) * msa::kBlock || V.n != K.n) return MSA_ERR_INVALID_ARG;
  if (K.h != s->Hkv || V.h != s->Hkv || Q.h < 1 || Q.h % K.h != 0) return MSA_ERR_INVALID_ARG;
  if (Q.d != K.d || K.d != V.d) return MSA_ERR_INVALID_ARG;
  if (Q.dtype != MSA_BF16 || K.dtype != MSA_BF16 || V.dtype != MSA_BF16) return MSA_ERR_UNSUPPORTED;
  if (Q.d != msa::kHeadDim || Q.h / K.h != msa::kGroup) return MSA_ERR_UNSUPPORTED;
  if (!std::isfinite(scale)) return MSA_ERR_INVALID_ARG;
  if (opts->path == MSA_PATH_Q_OUTER) return MSA_ERR_UNSUPPORTED;
  if (opts->path != MSA_PATH_AUTO && opts->path != MSA_PATH_KV_OUTER) return MSA_ERR_INVALID_ARG;
  msa_status_t st = ensure_partials(s, msa::kGroup);
  if (st != MSA_OK) return st;
  if (!s->bwd_ws) {
    void* p = nullptr;
    cudaError_t e = cudaMalloc(&p, msa::bwd_workspace_bytes(s));
    if (e != cudaSuccess) return from_cuda(e);
    s->bwd_ws = p;
  }
  const int ctas = opts->num_ctas > 0 ? opts->num_ctas : device_sms();
  if (ctas < 1) return MSA_ERR_CUDA;
  msa::BwdArgs a{s, Q.ptr, K.ptr, V.ptr, O, dO, LSE, dQ, dK, dV, s->bwd_ws, static_cast<int>(Q.h),
                 s->nblocks * msa::kBlock, scale, ctas,
                 {opts->stage_events[0], opts->stage_events[1], opts->stage_events[2]}};
  cudaError_t e = msa::launch_bwd(a, opts->stream);
  s->last_stream = opts->stream;
  return from_cuda(e);
}

msa_status_t msa_schedule_destroy(msa_schedule_t s) {
  if (!s) return MSA_ERR_INVALID_ARG;
  cudaError_t e = cudaStreamSynchronize(s->last_stream);
  if (s->partial) cudaFree(s->partial);
  if (s->bwd_ws) cudaFree(s->bwd_ws);
  if (s->vf16) cudaFree(s->vf16);
  if (s->dev_base) cudaFree(s->dev_base);
  delete s;
  return from_cuda(e);
}

msa_status_t msa_schedule_status(msa_schedule_t s) {
  if (!s) return MSA_ERR_INVALID_ARG;
  msa_schedule_info_t info;
  return msa_schedule_query(s, &info);
}

msa_status_t msa_schedule_query(msa_schedule_t s, msa_schedule_info_t* info) {
  if (!s || !info) return MSA_ERR_INVALID_ARG;
  cudaError_t e = cudaStreamSynchronize(s->last_stream);
  if (e != cudaSuccess) return from_cuda(e);
  msa::SchedHeader h;
  e = cudaMemcpy(&h, s->d.hdr, sizeof(h), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return from_cuda(e);
  info->entries = h.entries;
  info->nsb = h.nsb;
  info->ntiles = h.ntiles;
  info->path = h.path;
  info->status = h.status;
  info->rows = s->R;
  info->windows = s->nW;
  if (h.status & msa::kStatusTimeout) return MSA_ERR_TIMEOUT;
  if (h.status & msa::kStatusBounds) return MSA_ERR_BOUNDS;
  if (h.status & msa::kStatusBadIndex) return MSA_ERR_BAD_INDEX;
  return MSA_OK;
}

msa_status_t msa_schedule_export(msa_schedule_t s, int32_t* counts, int32_t* offsets, int32_t* qlist, int32_t* slot,
                                 int32_t* cmap, int32_t* tiles, int32_t* window_tiles) {
  if (!s) return MSA_ERR_INVALID_ARG;
  msa_schedule_info_t info;
  msa_status_t st = msa_schedule_query(s, &info);
  if (st != MSA_OK && st != MSA_ERR_BAD_INDEX) return st;
  struct Item {
    void* dst;
    const void* src;
    size_t bytes;
  } items[] = {
      {counts, s->d.counts, sizeof(int32_t) * s->R},
      {offsets, s->d.offsets, sizeof(int32_t) * (static_cast<size_t>(s->R) + 1)},
      {qlist, s->d.qlist, sizeof(int32_t) * static_cast<size_t>(info.entries)},
      {slot, s->d.slot, sizeof(int32_t) * static_cast<size_t>(info.entries)},
      {cmap, s->d.cmap, sizeof(int32_t) * static_cast<size_t>(s->cap_entries)},
      {tiles, s->d.tiles, sizeof(int4) * static_cast<size_t>(info.ntiles)},
      {window_tiles, s->d.window_tiles, sizeof(int32_t) * (static_cast<size_t>(s->nW) + 1)},
  };
  for (const Item& it : items) {
    if (!it.dst || it.bytes == 0) continue;
    cudaError_t e = cudaMemcpy(it.dst, it.src, it.bytes, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return from_cuda(e);
  }
  return st;
}

size_t msa_select_workspace_bytes(int N, int Hq, int Hkv, int nblocks) {
  if (N < 1 || Hq < 1 || Hkv < 1 || nblocks < 1) return 0;
  return msa::select_workspace_bytes(N, Hq, Hkv, nblocks);
}

namespace {
msa_status_t select_blocks(int reps, msa_tensor_t Q, msa_tensor_t K, int topK, int32_t* indices, void* workspace,
                           size_t workspace_bytes, cudaStream_t stream) {
  if (!Q.ptr || !K.ptr || !indices || !workspace) return MSA_ERR_INVALID_ARG;
  if (!aligned16(Q.ptr) || !aligned16(K.ptr) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return MSA_ERR_INVALID_ARG;
  if (Q.n < 1 || K.n < msa::kBlock || K.n % msa::kBlock || Q.n > K.n || Q.h < 1 || K.h < 1 || topK < 1)
    return MSA_ERR_INVALID_ARG;
  if (Q.d != K.d) return MSA_ERR_INVALID_ARG;
  if (Q.d != msa::kHeadDim || Q.h != msa::kGroup * K.h || Q.dtype != MSA_BF16 || K.dtype != MSA_BF16 || topK > 64)
    return MSA_ERR_UNSUPPORTED;
  if (Q.n > INT32_MAX || K.n > INT32_MAX || static_cast<int64_t>(Q.n) * K.h * topK > INT32_MAX) return MSA_ERR_CAPACITY;
  const int N = static_cast<int>(Q.n), Lkv = static_cast<int>(K.n), Hq = static_cast<int>(Q.h),
            Hkv = static_cast<int>(K.h);
  if (Lkv / msa::kBlock > 40960) return MSA_ERR_UNSUPPORTED;
  if (workspace_bytes < msa::select_workspace_bytes(N, Hq, Hkv, Lkv / msa::kBlock)) return MSA_ERR_INVALID_ARG;
  return from_cuda(reps == 4 ? msa::launch_select_r4(Q.ptr, K.ptr, N, Lkv, Hq, Hkv, topK, indices, workspace, stream)
                             : msa::launch_select_r1(Q.ptr, K.ptr, N, Lkv, Hq, Hkv, topK, indices, workspace, stream));
}
}  // namespace


msa_status_t msa_select_blocks_r1(msa_tensor_t Q, msa_tensor_t K, int topK, int32_t* indices, void* workspace,
                                  size_t workspace_bytes, cudaStream_t stream) {
  return select_blocks(1, Q, K, topK, indices, workspace, workspace_bytes, stream);
}

msa_status_t msa_select_blocks_r4(msa_tensor_t Q, msa_tensor_t K, int topK, int32_t* indices, void* workspace,
                                  size_t workspace_bytes, cudaStream_t stream) {
  return select_blocks(4, Q, K, topK, indices, workspace, workspace_bytes, stream);
}

msa_status_t msa_sparse_attn_fwd_tiles(msa_tensor_t Q, msa_tensor_t K, msa_tensor_t V, const int32_t* tile_lists,
                                       int tile, int topK, void* O, float* LSE, float scale, int32_t* status,
                                       const msa_fwd_opts_t* opts) {
  msa_fwd_opts_t def;
  if (!opts) {
    msa_fwd_opts_init(&def);
    opts = &def;
  }
  if (!Q.ptr || !K.ptr || !V.ptr || !O || !tile_lists) return MSA_ERR_INVALID_ARG;
  if (!aligned16(Q.ptr) || !aligned16(K.ptr) || !aligned16(V.ptr) || !aligned16(O)) return MSA_ERR_INVALID_ARG;
  if (Q.n < 1 || K.n < msa::kBlock || K.n % msa::kBlock || V.n != K.n || Q.n > K.n) return MSA_ERR_INVALID_ARG;
  if (K.h < 1 || V.h != K.h || Q.h < 1 || Q.d != K.d || K.d != V.d) return MSA_ERR_INVALID_ARG;
  if (tile < 16 || tile % 16 || topK < 1 || !std::isfinite(scale)) return MSA_ERR_INVALID_ARG;
  if (Q.d != msa::kHeadDim || Q.h != msa::kGroup * K.h || topK > 64) return MSA_ERR_UNSUPPORTED;
  if (Q.dtype != MSA_BF16 || K.dtype != MSA_BF16 || V.dtype != MSA_BF16) return MSA_ERR_UNSUPPORTED;
  if (K.n > INT32_MAX || static_cast<int64_t>(Q.n) * Q.h > INT32_MAX) return MSA_ERR_CAPACITY;
  const int ctas = opts->num_ctas > 0 ? opts->num_ctas : device_sms();
  if (ctas < 1) return MSA_ERR_CUDA;
  return from_cuda(msa::launch_tiles(Q.ptr, K.ptr, V.ptr, static_cast<int>(Q.n), static_cast<int>(K.n),
                                     static_cast<int>(Q.h), static_cast<int>(K.h), tile_lists, tile, topK, scale, O, LSE,
                                     status, ctas, opts->stream));
}

const char* msa_status_string(msa_status_t st) {
  switch (st) {
    case MSA_OK: return "ok";
    case MSA_ERR_INVALID_ARG: return "invalid argument";
    case MSA_ERR_UNSUPPORTED: return "unsupported configuration";
    case MSA_ERR_CUDA: return "CUDA runtime error";
    case MSA_ERR_OOM: return "device allocation failed";
    case MSA_ERR_BAD_INDEX: return "block id out of range in indices (ignored)";
    case MSA_ERR_TIMEOUT: return "bounded device wait expired";
    case MSA_ERR_CAPACITY: return "size exceeds a fixed capacity";
    case MSA_ERR_BOUNDS: return "an index or TMA coordinate was out of range (bounds-checked build)";
  }
  return "unknown status";
}

int msa_last_cuda_error(void) { return g_last_cuda; }

int msa_debug_build(void) { return MSA_DEBUG; }

int msa_version(void) { return 100; }

}  // extern "C"
