// msa_sparse_attn_fwd_noalloc: the whole forward (schedule, attention, combine)
// with no device allocation.
//
// Some callers cannot call cudaMalloc at all: a serving process that reserves its
// whole device-memory budget when it starts and must not grow it later, a runtime
// that hands all device memory out through its own pool and forbids raw
// allocations, or a latency-critical loop that cannot absorb the device-wide
// synchronisation a cudaMalloc / cudaFree may cause.  msa_build_schedule and
// msa_sparse_attn_fwd allocate their workspaces; this entry point instead carves
// every scratch buffer (schedule arrays and partial outputs) out of the fixed
// file-scope array below and launches exactly the same kernels.
//
// Contract (also stated in include/msa.h):
//   - the scratch is MSA_NOALLOC_SCRATCH_BYTES of device memory that every GPU
//     loading libmsa holds until the process exits;
//   - problems whose workspace does not fit are rejected with MSA_ERR_CAPACITY;
//   - the first call on a device looks up the array's device address
//     (cudaGetSymbolAddress) with that device current; make that first call before
//     any stream capture;
//   - all calls share the array and it keeps the last call's contents: the schedule
//     kernels zero what must start at zero (the query bitmask and the status
//     header) on every call, and every other array is fully written before it is
//     read; calls whose work overlaps on the GPU (other streams, other threads)
//     race on the array and must be serialised by the caller.
#include <cmath>
#include <cstring>
#include <mutex>

#include "msa_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[MSA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_dev[kMaxDevices] = {};  // device address of g_noalloc_scratch, per device ordinal

// In host code `g_noalloc_scratch` names a host-side shadow, not device memory;
// kernels must be given the address returned here.
msa_status_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return msa::status_from_cuda(e);
  if (dev < 0 || dev >= kMaxDevices) return MSA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_dev[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return msa::status_from_cuda(e);
    g_scratch_dev[dev] = p;
  }
  *out = g_scratch_dev[dev];
  return MSA_OK;
}

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int device_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}

}  // namespace

extern "C" msa_status_t msa_sparse_attn_fwd_noalloc(const int32_t* indices, int N, int Hkv, int topK, int nblocks,
                                                    msa_tensor_t Q, msa_tensor_t K, msa_tensor_t V, void* O,
                                                    float* LSE, float scale, int32_t* status,
                                                    const msa_fwd_opts_t* opts) {
  msa_fwd_opts_t def;
  if (!opts) {
    msa_fwd_opts_init(&def);
    opts = &def;
  }
  // the checks of msa_build_schedule and msa_sparse_attn_fwd
  if (!indices || !Q.ptr || !K.ptr || !V.ptr || !O) return MSA_ERR_INVALID_ARG;
  if (N < 1 || Hkv < 1 || topK < 1 || nblocks < 1) return MSA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(nblocks) * msa::kBlock > INT32_MAX) return MSA_ERR_CAPACITY;
  if (static_cast<int64_t>(Hkv) * nblocks > INT32_MAX) return MSA_ERR_CAPACITY;
  if (static_cast<int64_t>(N) > static_cast<int64_t>(nblocks) * msa::kBlock) return MSA_ERR_INVALID_ARG;
  if (topK > 64) return MSA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(N) * Hkv * topK * msa::kGroup > INT32_MAX) return MSA_ERR_CAPACITY;
  if (!aligned16(Q.ptr) || !aligned16(K.ptr) || !aligned16(V.ptr) || !aligned16(O)) return MSA_ERR_INVALID_ARG;
  if (Q.n != N || K.n != static_cast<int64_t>(nblocks) * msa::kBlock || V.n != K.n) return MSA_ERR_INVALID_ARG;
  if (K.h != Hkv || V.h != Hkv || Q.h < 1 || Q.h % K.h != 0) return MSA_ERR_INVALID_ARG;
  if (Q.d != K.d || K.d != V.d) return MSA_ERR_INVALID_ARG;
  if (Q.dtype != K.dtype || K.dtype != V.dtype) return MSA_ERR_UNSUPPORTED;
  if (Q.d != msa::kHeadDim || Q.h / K.h != msa::kGroup || Q.dtype != MSA_BF16) return MSA_ERR_UNSUPPORTED;
  if (!std::isfinite(scale)) return MSA_ERR_INVALID_ARG;
  if (opts->path != MSA_PATH_AUTO && opts->path != MSA_PATH_KV_OUTER && opts->path != MSA_PATH_Q_OUTER)
    return MSA_ERR_INVALID_ARG;
  // the scratch holds bf16 partials only, and the test-only kernel instances stay with
  // the allocating entry points
  if (opts->partials_fp32 != 0 || opts->debug_flags != 0) return MSA_ERR_UNSUPPORTED;

  // layout inside the scratch array: schedule arrays, then partial outputs and their (m, l)
  msa_schedule s;
  std::memset(&s, 0, sizeof(s));
  msa::schedule_dims(&s, N, Hkv, topK, nblocks);
  msa::carve_schedule(&s, nullptr);
  const size_t rows = static_cast<size_t>(msa::part_rows(s.cap_entries));
  const size_t sched_bytes = round256(s.dev_bytes);
  const size_t part_bytes = round256(rows * msa::kHeadDim * 2);
  const size_t total = sched_bytes + part_bytes + rows * sizeof(float2);
  if (total > MSA_NOALLOC_SCRATCH_BYTES) return MSA_ERR_CAPACITY;

  void* base = nullptr;
  msa_status_t st = scratch_address(&base);
  if (st != MSA_OK) return st;
  char* b = static_cast<char*>(base);
  msa::carve_schedule(&s, b);
  s.dev_base = b;
  s.partial = b + sched_bytes;
  s.pstat = reinterpret_cast<float2*>(b + sched_bytes + part_bytes);
  s.partial_G = msa::kGroup;

  const cudaStream_t stream = opts->stream;
  s.last_stream = stream;
  const int ctas = opts->num_ctas > 0 ? opts->num_ctas : device_sms();
  if (ctas < 1) return MSA_ERR_CUDA;
  const int force = opts->path != MSA_PATH_AUTO ? static_cast<int>(opts->path)
                    : msa::q_outer_certain(N, Hkv, topK) ? msa::kPathQOuter : 0;
  const int Hq = static_cast<int>(Q.h);
  cudaError_t e;
  if ((e = msa::enqueue_schedule(&s, indices, stream))) return msa::status_from_cuda(e);
  if (opts->stage_events[0] && (e = cudaEventRecord(opts->stage_events[0], stream))) return msa::status_from_cuda(e);
  msa::KvOuterArgs a{&s, Q.ptr, K.ptr, V.ptr, Hq, nblocks * msa::kBlock, scale, force, ctas, false, 1.f, false, 0};
  if ((e = msa::launch_kv_outer(a, stream))) return msa::status_from_cuda(e);
  if (opts->stage_events[1] && (e = cudaEventRecord(opts->stage_events[1], stream))) return msa::status_from_cuda(e);
  if (force != msa::kPathQOuter && (e = msa::launch_combine(&s, Hq, O, LSE, 1.f, force, false, stream)))
    return msa::status_from_cuda(e);
  if ((e = msa::launch_q_outer(&s, Q.ptr, K.ptr, V.ptr, Hq, scale, O, LSE, force, stream)))
    return msa::status_from_cuda(e);
  if (opts->stage_events[2] && (e = cudaEventRecord(opts->stage_events[2], stream))) return msa::status_from_cuda(e);
  if (status && (e = cudaMemcpyAsync(status, &s.d.hdr->status, sizeof(int32_t), cudaMemcpyDefault, stream)))
    return msa::status_from_cuda(e);
  return MSA_OK;
}
