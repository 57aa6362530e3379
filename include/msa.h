/*
 * msa.h -- C ABI of libmsa: forward main branch of block-sparse attention on GQA
 * for NVIDIA GB300 (sm_103a).
 *
 * The operation ("Kernel optimization for MiniMax M3 on NVIDIA Blackwell",
 * opening section): the KV sequence is cut into 128-token blocks; for every query
 * token and every KV head (GQA group) a list of topK block ids is given; each query
 * head attends, exactly, to the keys of the blocks its group selected, and nowhere
 * else.  The softmax of a query is normalised over the union of its selected blocks
 * ("Sparse Attention", Chapter 1).  The query's own block is attended with a causal
 * mask ("Flash-MSA": the local block is always kept, sliding-window style).
 *
 * Conventions used by every call:
 *   - Q is [N, Hq, D], K and V are [Lkv, Hkv, D], all contiguous, on the device.
 *     D = 128, block = 128 tokens, Lkv = 128 * nblocks, G = Hq / Hkv = 16.
 *   - The N queries are the LAST N positions of the sequence: query i sits at
 *     pos(i) = Lkv - N + i and sees key j iff j <= pos(i).  lb(i) = pos(i) / 128 is
 *     its own (local) block.
 *   - Head h uses KV head g = h / G.
 *   - indices is int32 [N, Hkv, topK] on the device.  -1 is padding; a repeated id
 *     counts once; an id above lb(i) contributes nothing; an id >= nblocks or < -1
 *     is invalid (ignored, and reported by msa_schedule_query).
 *   - O is bf16 [N, Hq, D]; LSE is fp32 [N, Hq], the natural log of
 *     sum_j exp(scale * q.k_j) over the visible selected keys (-inf if none, with
 *     O = 0).
 *   - Every call is asynchronous on the given stream and never synchronises the
 *     host, except msa_schedule_query / msa_schedule_export (documented as such).
 *   - No call aborts, traps or prints.  Errors are returned as msa_status_t; host-
 *     checkable errors return before anything is enqueued.
 */
#ifndef MSA_H_
#define MSA_H_

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MSA_OK = 0,
  MSA_ERR_INVALID_ARG = 1,  /* null pointer, inconsistent shapes, bad sizes */
  MSA_ERR_UNSUPPORTED = 2,  /* valid but not built: D != 128, G != 16, ... */
  MSA_ERR_CUDA = 3,         /* a CUDA runtime call failed (see msa_last_cuda_error) */
  MSA_ERR_OOM = 4,          /* device allocation failed */
  MSA_ERR_BAD_INDEX = 5,    /* device saw block ids >= nblocks or < -1 (ignored) */
  MSA_ERR_TIMEOUT = 6,      /* a bounded device wait expired; outputs undefined */
  MSA_ERR_CAPACITY = 7,     /* a size exceeds a fixed capacity */
  MSA_ERR_BOUNDS = 8        /* bounds-checked build only (libmsa_debug.so, MSA_DEBUG): an index
                               or TMA coordinate read from device memory was out of range; the
                               access was skipped or redirected to element 0; outputs undefined */
} msa_status_t;

typedef enum { MSA_BF16 = 0, MSA_FP8_E4M3 = 1 } msa_dtype_t;

/* Which kernel computes the attention.  AUTO follows the crossover of "Kernel
 * optimization for MiniMax M3" (Q-outer vs KV-outer section and appendix), re-derived from
 * measurements on GB300 as the page asks: KV-outer when 10 E - 13 nsb > 35000, where E is
 * the number of distinct (query, KV head, block) entries and nsb the number of distinct
 * (KV head, block) pairs (the page's B200 rule, nsb / N < 2.85, picked the slower path at 19
 * of 52 measured GB300 points).  The choice is made on the device by msa_build_schedule;
 * no device-to-host copy is needed.  Where the sizes alone decide it (E <= N * Hkv * topK
 * and nsb >= E / N, so N * Hkv * topK * (10 N - 13) <= 35000 N means Q-outer for any lists:
 * every N = 1 call), the forward launches only the Q-outer kernel; the result is the same. */
typedef enum { MSA_PATH_AUTO = 0, MSA_PATH_KV_OUTER = 1, MSA_PATH_Q_OUTER = 2 } msa_path_t;

/* Opaque schedule: the reverse index of one indices tensor plus its device
 * workspace.  It owns device memory; destroy it with msa_schedule_destroy. */
typedef struct msa_schedule* msa_schedule_t;

/* A dense [n, h, d] device tensor. */
typedef struct {
  const void* ptr;
  msa_dtype_t dtype;
  int64_t n, h, d;
} msa_tensor_t;

typedef struct {
  cudaStream_t stream;   /* stream for every launch; 0 = legacy default stream */
  msa_path_t path;       /* AUTO, or force one kernel (tests, studies) */
  float q_descale;       /* fp8 only: real value = stored e4m3 value * descale */
  float k_descale;
  float v_descale;
  /* Optional CUDA events recorded on `stream` (NULL = skip):
   * [0] before the attention kernel, [1] after it, [2] after the combine. */
  cudaEvent_t stage_events[3];
  int num_ctas;          /* persistent grid size for the KV-outer kernel; 0 = #SMs */
  /* KV-outer partial outputs: 0 = bf16 (default), 1 = fp32 ("Sparse Attention", Chapter 5,
   * "Partial outputs and Combine": the partials' format is the main data-movement cost,
   * 16x (bf16) or 32x (fp32) the final bf16 output).  fp32 doubles the partial bytes and
   * keeps the per-block P V sums unrounded until the combine. */
  int partials_fp32;
  /* Test use only; 0 in normal calls.  Bit 0 (bf16 inputs, bf16 partials, KV-outer
   * path): a separate build of the KV-outer kernel whose scheduler warp publishes no
   * work runs instead, so every other role's bounded wait (2 s) expires: the call then
   * leaves O undefined, sets the schedule's timeout bit (msa_schedule_query returns
   * MSA_ERR_TIMEOUT until the schedule is rebuilt) and the device stays usable.  It
   * exercises the timeout path without faulting anything.  Bit 1 (E4M3 inputs, positive
   * scale, bf16 partials, KV-outer path): P V on E4M3 tensor cores, with P rounded to E4M3
   * in shared memory and V transposed per block (E4M3) by a pass before the kernel, in
   * place of f16 V and f16 P.  Measured on the 65536-query E4M3 workload: 0.3% faster
   * (3.84 vs 3.85 ms), relative L2 error 9.3e-3 instead of 1.9e-3, so it is not the
   * default. */
  int debug_flags;
} msa_fwd_opts_t;

/* Fill *opts with the defaults: stream 0, AUTO, descales 1, no events, #SMs. */
void msa_fwd_opts_init(msa_fwd_opts_t* opts);

/*
 * msa_build_schedule -- index inversion ("Sparse Attention", Chapter 5, "Reverse
 * index"; "Kernel optimization for MiniMax M3", load-balancing section).
 *
 * From indices [N, Hkv, topK] builds, on `stream`, with no host synchronisation:
 *   - the CSR over rows r = g * nblocks + b: counts[r], offsets[r], and for every
 *     entry the query (ascending within a row) and its slot in that query's list;
 *   - the combine map (i, g, k) -> CSR position (or -1);
 *   - a work list of tiles (at most 8 entries of one row) ordered by query window,
 *     so heavy blocks are split over many CTAs;
 *   - nsb and the Q-outer / KV-outer choice, kept on the device.
 *
 * *inout: NULL on entry -> a new schedule is allocated (cudaMalloc, synchronous)
 * and returned.  A schedule from an earlier call with the same (N, Hkv, topK,
 * nblocks) -> its workspace is reused and nothing is allocated.  `indices` is read
 * by kernels on `stream`: keep it alive until the stream passes this call.  The
 * schedule keeps no pointer to it.
 *
 * Returns MSA_ERR_INVALID_ARG for null pointers, N < 1, N > 128 * nblocks,
 * Hkv < 1, topK < 1 or nblocks < 1; MSA_ERR_CAPACITY when N * Hkv * topK * 16
 * exceeds 2^31 - 1; MSA_ERR_OOM / MSA_ERR_CUDA on allocation or launch failure.
 */
msa_status_t msa_build_schedule(const int32_t* indices, int N, int Hkv, int topK, int nblocks,
                                cudaStream_t stream, msa_schedule_t* inout);

/*
 * msa_sparse_attn_fwd -- the forward main branch over a built schedule.
 *
 * KV-outer path ("Kernel optimization for MiniMax M3", kernel stages): a persistent
 * warp-specialised tcgen05 kernel loads each selected K/V block with TMA, gathers
 * the queries that chose it, computes S = Q K^T and P V in tensor memory with one
 * softmax step per tile, and writes partial outputs (bf16) and their log-sum-exp in
 * contiguous tile-ordered slabs; a combine kernel gathers each query's partials and
 * merges them by LSE weighting ("Sparse Attention", Chapter 5, "Partial outputs and
 * Combine").  Q-outer path (same page, Q-outer structure): one unit per (query,
 * group) walks its own blocks with an online softmax and writes O and LSE directly.
 *
 * Q: [N, Hq, D]; K, V: [Lkv, Hkv, D]; all bf16, or all MSA_FP8_E4M3 (one byte per
 * element, real value = stored value * the tensor's descale in opts; descales must be
 * finite and > 0).  O: bf16 [N, Hq, D] device; LSE: fp32 [N, Hq] device (may be NULL).
 * scale multiplies q.k (typically 1/sqrt(D)).  opts may be NULL (defaults).
 * E4M3 inputs take either path (AUTO: the device's choice, as for bf16): S = Q K^T on
 * E4M3 tensor cores, V widened to f16 (exact) and P V in f16, output bf16.  The KV-outer
 * path widens the whole V tensor by a pass before the attention kernel; the Q-outer path
 * widens each selected block in shared memory, so the pass exits at once there.
 *
 * The first call for a given head count and partial format allocates the partial-output
 * workspace of the schedule (cudaMalloc, synchronous): N*Hkv*topK*G*(2*D + 8) bytes at most
 * for bf16 rows + float2 (m, l), N*Hkv*topK*G*(4*D + 8) with opts->partials_fp32.  A fp32
 * workspace also serves bf16 calls; the first E4M3 call that may take the KV-outer path
 * (any but a forced Q-outer) also allocates Lkv*Hkv*D*2 bytes for an f16 copy of V (each
 * such call widens V into it, exactly, when the device takes that path); later calls
 * allocate nothing.
 *
 * Returns MSA_ERR_INVALID_ARG on null pointers or shapes inconsistent with the
 * schedule or non-positive E4M3 descales; MSA_ERR_UNSUPPORTED for D != 128, G != 16 or
 * mixed dtypes; MSA_ERR_CUDA on launch failure.
 */
msa_status_t msa_sparse_attn_fwd(msa_tensor_t Q, msa_tensor_t K, msa_tensor_t V, msa_schedule_t s,
                                 void* O, float* LSE, float scale, const msa_fwd_opts_t* opts);

/*
 * msa_sparse_attn_bwd -- gradients of the forward main branch over the same schedule.
 *
 * "Flash-MSA: accelerating million-token training with sparse attention", order of
 * operations: the forward keeps its block indices and its log-sum-exp for the
 * backward, which computes the main-attention gradients over the cached blocks.  For
 * each (query i, head h) with visible keys J (the union of its selected blocks,
 * causal): P_j = exp(scale * q.k_j - LSE[i,h]), D = dO[i,h] . O[i,h],
 * dS_j = P_j (dO[i,h] . v_j - D); dQ[i,h] = scale * sum_j dS_j k_j,
 * dK_j += scale * dS_j q[i,h], dV_j += P_j dO[i,h].  Keys no query sees get 0.
 *
 * Kernels, all on opts->stream with no host synchronisation: D = rowsum(dO * O);
 * units of at most 256 entries of one (group, block) row of the schedule; a
 * KV-stationary tcgen05 kernel that holds K_b, V_b, gathers Q and dO of 8 queries x 16
 * heads per tile, forms P and dS on chip, accumulates dK_b, dV_b in tensor memory and
 * writes each entry's dQ contribution (bf16) to the schedule's partial workspace;
 * a reduction of the units' dK/dV (fp32) and a gather of each query's dQ
 * contributions, both in a fixed order (results are deterministic).
 *
 * Q, dO: bf16 [N, Hq, D]; K, V: bf16 [Lkv, Hkv, D]; O: bf16 [N, Hq, D] and LSE: fp32
 * [N, Hq] (natural log) from msa_sparse_attn_fwd on the same inputs and schedule (s
 * must still hold the lists the forward used).  Outputs dQ: bf16 [N, Hq, D]; dK, dV:
 * bf16 [Lkv, Hkv, D]; all device pointers, 16-byte aligned, caller-owned.  scale is the
 * forward's.  opts may be NULL; opts->stream, opts->num_ctas and opts->stage_events
 * ([0] before the tcgen05 kernel, [1] after it, [2] after the last kernel) are used;
 * opts->path must be AUTO or KV_OUTER.
 *
 * The first call allocates the schedule's partial-output workspace (if the forward
 * has not) and a backward workspace (cudaMalloc, synchronous): N*Hq*4 bytes for D,
 * and 128 KiB of fp32 dK/dV per unit for at most min(Hkv*nblocks, N*Hkv*topK) +
 * N*Hkv*topK/256 units.  Later calls allocate nothing.
 *
 * Returns MSA_ERR_INVALID_ARG on null or misaligned pointers or shapes inconsistent
 * with the schedule; MSA_ERR_UNSUPPORTED for E4M3, D != 128, G != 16 or a forced
 * Q-outer path; MSA_ERR_OOM / MSA_ERR_CUDA on allocation or launch failure.  A device
 * wait that exceeds its bound sets the schedule's timeout flag (msa_schedule_query).
 */
msa_status_t msa_sparse_attn_bwd(msa_tensor_t Q, msa_tensor_t K, msa_tensor_t V, const void* O, const void* dO,
                                 const float* LSE, msa_schedule_t s, void* dQ, void* dK, void* dV, float scale,
                                 const msa_fwd_opts_t* opts);

/* Frees the schedule's device memory (synchronises its last stream first). */
msa_status_t msa_schedule_destroy(msa_schedule_t s);

typedef struct {
  int64_t entries;     /* E: valid (query, group, block) entries */
  int32_t nsb;         /* distinct selected (group, block) pairs */
  int32_t ntiles;      /* tiles in the work list */
  int32_t path;        /* 1 = KV-outer, 2 = Q-outer (the AUTO choice) */
  int32_t status;      /* device-side sticky flags: bit0 bad index, bit1 timeout */
  int32_t rows;        /* Hkv * nblocks */
  int32_t windows;     /* query windows of the work list */
} msa_schedule_info_t;

/* Synchronises the schedule's last stream and reads its device header.  Returns
 * MSA_ERR_BAD_INDEX / MSA_ERR_TIMEOUT when the sticky flags are set (info is still
 * filled).  Test and debug use. */
msa_status_t msa_schedule_query(msa_schedule_t s, msa_schedule_info_t* info);

/* msa_schedule_status -- the schedule's sticky device status (test and debug use).
 * Synchronises the schedule's last stream, then returns MSA_ERR_TIMEOUT if a bounded
 * device wait of a call on this schedule expired, else MSA_ERR_BAD_INDEX if the
 * schedule build saw a block id >= nblocks or < -1 (ignored as padding), else MSA_OK.
 * MSA_ERR_INVALID_ARG for a NULL schedule; MSA_ERR_CUDA if the synchronisation or the
 * read fails.  The same bits as msa_schedule_query's info->status; they stay set until
 * the schedule is rebuilt.  Device-detected errors never abort or trap ("Kernel
 * optimization for MiniMax M3": shapes fixed per request, no device-to-host sync on the
 * hot path, so this check is kept off the hot path). */
msa_status_t msa_schedule_status(msa_schedule_t s);

/* Synchronises and copies the schedule to host arrays (any may be NULL):
 * counts[rows], offsets[rows+1], qlist[E], slot[E], cmap[N*Hkv*topK],
 * tiles[4*ntiles] as (row, first, count, window), window_tiles[windows+1].
 * Test and debug use. */
msa_status_t msa_schedule_export(msa_schedule_t s, int32_t* counts, int32_t* offsets,
                                 int32_t* qlist, int32_t* slot, int32_t* cmap, int32_t* tiles,
                                 int32_t* window_tiles);

/* Bytes of device scratch behind msa_sparse_attn_fwd_noalloc. */
#define MSA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/*
 * msa_sparse_attn_fwd_noalloc -- the whole forward (schedule, attention, combine)
 * in one call that allocates no device memory.
 *
 * The pages have no counterpart for this call: it exists for callers that cannot
 * call cudaMalloc, for example a serving process that reserves its entire device
 * memory budget at start-up and may not grow it afterwards, a runtime that owns all
 * device memory through its own pool, or a latency-critical loop that cannot absorb
 * the device-wide synchronisation of cudaMalloc / cudaFree.
 *
 * Arguments are those of msa_build_schedule followed by those of
 * msa_sparse_attn_fwd (without a schedule handle), then `status`; results are the
 * same as that pair's.  The schedule and the partial outputs live in one fixed device
 * array of MSA_NOALLOC_SCRATCH_BYTES inside libmsa, which every GPU that loads the
 * library holds until the process exits.  Limits: the workspace for N * Hkv * topK
 * list slots (about 4.2 KB per slot for the partial outputs, plus the schedule) must
 * fit in that array, else MSA_ERR_CAPACITY is returned before anything is enqueued (the
 * 1024-query, 1 KV head, topK 4 shape fits; the M3 shape does not).  Inputs must be
 * bf16; opts->partials_fp32 and opts->debug_flags must be 0 (MSA_ERR_UNSUPPORTED
 * otherwise).
 *
 * status: optional (NULL = not wanted) int32 in caller memory that the device can
 * write (device memory, or pinned / managed host memory).  After the forward, on the
 * same stream, the call copies the schedule's sticky bits into it: bit 0 = a block id
 * >= nblocks or < -1 was seen (and ignored), bit 1 = a bounded device wait expired
 * (outputs undefined).  These are the bits msa_schedule_query reports for the
 * allocating pair; here the schedule lives in the shared array, and the next call
 * clears them, so this copy is the only way to see them.
 *
 * The first call on a device looks up the array's device address with that device
 * current; make that first call before any stream capture.  Every call reuses the
 * same array and it keeps the previous call's contents: the call clears what must
 * start at zero itself.  Calls that overlap on the GPU (other streams or threads)
 * race on the array; the caller must serialise them.
 */
msa_status_t msa_sparse_attn_fwd_noalloc(const int32_t* indices, int N, int Hkv, int topK, int nblocks,
                                         msa_tensor_t Q, msa_tensor_t K, msa_tensor_t V, void* O, float* LSE,
                                         float scale, int32_t* status, const msa_fwd_opts_t* opts);

/*
 * Block selector R1 ("Sparse Attention" (dinara-dl), Chapter 4, "R1: One
 * Representative") -- the step that produces the block lists the forward reads.
 *
 * For every tile of 128 consecutive queries and every GQA group: each query head of
 * the group is summarised by the mean of its query vectors over the tile, each KV
 * block of the group by the mean of its 128 key vectors; a block's score is the
 * largest, over the group's heads, of the dot product of the two means.  The tile
 * keeps its topK best blocks: first the blocks holding the tile's own queries
 * (ascending), then by score descending, ties to the smaller block id; blocks after
 * the tile's last query are never chosen; if fewer than topK blocks are candidates the
 * list is padded with -1.  Every query of the tile gets the tile's list.
 *
 * Q: bf16 [N, Hq, 128]; K: bf16 [Lkv, Hkv, 128], Lkv a multiple of 128, N <= Lkv
 * (queries are the last N positions); Hq = 16 * Hkv.  indices: device int32
 * [N, Hkv, topK], written completely.  workspace: device memory of at least
 * msa_select_workspace_bytes(N, Hq, Hkv, Lkv / 128) bytes (enough for R1 and R4), 256-byte aligned, owned by
 * the caller; its contents are scratch.  Arithmetic is fp32 (means, dot products).
 * Asynchronous on `stream`; nothing is allocated.
 *
 * Returns MSA_ERR_INVALID_ARG for null or misaligned pointers, inconsistent shapes,
 * topK < 1 or a workspace that is too small; MSA_ERR_UNSUPPORTED for D != 128,
 * Hq != 16 * Hkv, non-bf16 inputs, topK > 64 or more than 40960 blocks; MSA_ERR_CUDA
 * on launch failure.
 */
size_t msa_select_workspace_bytes(int N, int Hq, int Hkv, int nblocks);
msa_status_t msa_select_blocks_r1(msa_tensor_t Q, msa_tensor_t K, int topK, int32_t* indices, void* workspace,
                                  size_t workspace_bytes, cudaStream_t stream);

/*
 * msa_select_blocks_r4 -- block selector R4 ("Sparse Attention" (dinara-dl), Chapter 4,
 * "R4: Four Representatives").  As msa_select_blocks_r1, except that a 128-query tile and
 * a 128-key block are each cut into four consecutive 32-token quarters summarised by
 * their means, and a block's score is the largest of the 16 quarter-pair dot products
 * over the group's query heads (a quarter of a short last tile that holds no query has no
 * representative).  Same arguments, list order, forced own blocks, padding, workspace
 * size (msa_select_workspace_bytes covers both selectors) and errors.
 */
msa_status_t msa_select_blocks_r4(msa_tensor_t Q, msa_tensor_t K, int topK, int32_t* indices, void* workspace,
                                  size_t workspace_bytes, cudaStream_t stream);

/*
 * msa_sparse_attn_fwd_tiles -- the forward main branch when consecutive queries share
 * their block lists ("Sparse Attention" (dinara-dl), Chapter 4: the selectors choose
 * the blocks of a whole 128-query tile per GQA group; Chapter 3: a query tile stays on
 * chip while its blocks stream past).  No schedule, no partial outputs, no combine:
 * each group of 8 consecutive queries x 16 heads walks its list's blocks with an online
 * softmax and writes O and LSE directly.
 *
 * Q: bf16 [N, Hq, 128]; K, V: bf16 [Lkv, Hkv, 128], Lkv a multiple of 128, N <= Lkv
 * (queries are the last N positions); Hq = 16 * Hkv.  tile_lists: device int32
 * [ceil(N / tile), Hkv, topK]: query i of group g uses list tile_lists[i / tile][g];
 * tile a multiple of 16.  The semantics per query are those of msa_sparse_attn_fwd
 * on the expanded per-query lists: -1 is padding, a repeated id counts once, keys
 * after the query are masked (ids after the last query of a 16-query group are
 * skipped), ids >= Lkv / 128 or < -1 are ignored and set bit 0 of *status.  O: bf16
 * [N, Hq, 128]; LSE: fp32 [N, Hq] (may be NULL); a query with no visible key gets
 * O = 0, LSE = -inf.  status: device int32 (may be NULL), bits OR-ed in: 1 bad id,
 * 2 a device wait timed out; the caller zeroes it.  opts: stream and num_ctas are
 * used (path, descales and stage events are ignored).  Asynchronous; nothing is
 * allocated.
 *
 * Returns MSA_ERR_INVALID_ARG for null or misaligned pointers, inconsistent shapes,
 * tile not a positive multiple of 16, topK < 1 or a non-finite scale;
 * MSA_ERR_UNSUPPORTED for D != 128, Hq != 16 * Hkv, non-bf16 inputs or topK > 64;
 * MSA_ERR_CUDA on launch failure.
 */
msa_status_t msa_sparse_attn_fwd_tiles(msa_tensor_t Q, msa_tensor_t K, msa_tensor_t V, const int32_t* tile_lists,
                                       int tile, int topK, void* O, float* LSE, float scale, int32_t* status,
                                       const msa_fwd_opts_t* opts);

/* Human-readable text for a status code (static storage). */
const char* msa_status_string(msa_status_t st);

/* The last CUDA error code seen by the library on this thread (0 if none). */
int msa_last_cuda_error(void);

/* Library version: major * 10000 + minor * 100 + patch. */
int msa_version(void);

/* 1 in the bounds-checked build (libmsa_debug.so, compiled with MSA_DEBUG=1; same entry
 * points, every device-side gather index and TMA coordinate checked, violations reported as
 * MSA_ERR_BOUNDS by msa_schedule_status / msa_schedule_query), 0 in the release build.  A
 * development aid with no counterpart in the pages. */
int msa_debug_build(void);

#ifdef __cplusplus
}
#endif
#endif /* MSA_H_ */
