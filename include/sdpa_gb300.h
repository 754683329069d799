/*
 * sdpa_gb300.h -- C ABI of the fused scaled-dot-product attention library for
 * NVIDIA GB300 (sm_103a), libsdpa_gb300.so.
 *
 * What every entry point computes
 * --------------------------------
 * For batch b, query head h and query row i:
 *
 *     G   = Hq / Hkv                 query heads per key/value head (GQA)
 *     g   = h / G                    the key/value head that query head h reads
 *     p_i = Lk - Lq + i              the row's position in the key sequence
 *                                    (causal rows are aligned bottom-right)
 *     visible keys j: (!causal || j <= p_i) && (window == 0 || p_i - j < window)
 *     out[b,h,i,:] = sum_j softmax_j(scale * q[b,h,i,:] . k[b,g,j,:]) * v[b,g,j,:]
 *
 * with the softmax taken over the visible keys only.  This is the
 * "matmul + softmax + matmul" attention of the page "fix: add head_dim=256 to
 * fused SDPA full attention kernel" (MLX PR #3293, section "Benchmark: fused vs
 * unfused SDPA for head_dim=256"), computed tile by tile so that the
 * [heads, Lq, Lk] score matrix is never stored ("Fused SDPA full-attention for
 * head_dim=192/256", MLX PR #3660, section "Microbenchmarks": the fused
 * transient stays flat as kL grows).  Grouped-query heads follow the same page
 * (n_q = 16 query heads over n_kv = 8 key/value heads); the causal flag and the
 * sliding window follow "fix: gemma-4 long-prompt prefill OOMs on CUDA"
 * (mlxcel issue #672, sections "Root cause" and "Suggested fix direction"),
 * which replaces a dense [L, L] windowed mask by in-kernel masking; the window
 * of 1024 and the bottom-right alignment of decode rows follow "fix: Gemma 4
 * MTP never engages on CUDA (GB10)" (mlxcel issue #2160, sections "Current
 * Behavior" and "Proposed Solution").
 *
 * Window convention: a window W keeps the W most recent keys including the
 * row's own (p_i - j < W).  window == 0 means no window.
 *
 * Layout and ownership (all entry points)
 * ---------------------------------------
 *  q    [B, Hq,  Lq, D]  contiguous, fp16 or bf16, device memory
 *  k    [B, Hkv, Lk, D]  contiguous, same dtype, device memory
 *  v    [B, Hkv, Lk, D]  contiguous, same dtype, device memory
 *  out  [B, Hq,  Lq, D]  contiguous, same dtype, device memory, written
 *  Every pointer is owned by the caller, must be 16-byte aligned and must stay
 *  valid until the work queued on `stream` has finished.  The library never
 *  allocates device memory: where split partials are needed the caller passes
 *  a workspace of at least the size the matching *_workspace_bytes call
 *  returns (that size does not grow with Lk).
 *  Supported: D in {128, 192, 256, 512}; dtype SDPA_F16 or SDPA_BF16.  256
 *  and 512 are the pages' head dims; 192 is the head dim "Fused SDPA
 *  full-attention for head_dim=192/256" (MLX PR #3660) also serves, and 128
 *  is kept as a regression shape.
 *
 * Errors
 * ------
 *  Calls are asynchronous on `stream`.  The return value reports argument
 *  validation and launch errors only; on any non-zero return nothing has been
 *  queued.  Device-side failures (a pipeline wait that gave up after 2 s) are
 *  recorded in a per-device status word that sdpa_device_status() returns.
 *  No entry point aborts the process.
 */
#ifndef SDPA_GB300_H_
#define SDPA_GB300_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* sdpa_stream_t;

enum sdpa_dtype { SDPA_F16 = 0, SDPA_BF16 = 1 };

enum sdpa_status {
  SDPA_OK = 0,
  SDPA_ERR_INVALID_ARG = -1,    /* bad size, mask combination, NULL pointer, scale */
  SDPA_ERR_UNSUPPORTED = -2,    /* head dim or dtype outside the supported set */
  SDPA_ERR_WORKSPACE = -3,      /* workspace missing or smaller than required */
  SDPA_ERR_CUDA = -4,           /* a CUDA runtime / driver call failed */
  SDPA_ERR_DEVICE_TIMEOUT = -5, /* a kernel wait gave up (see sdpa_device_status) */
  SDPA_ERR_ALIGNMENT = -6,      /* a pointer is not 16-byte aligned */
  SDPA_ERR_SCRATCH_LIMIT = -7   /* sdpa_decode_noalloc: the call needs more than its built-in
                                   scratch (SDPA_NOALLOC_SCRATCH_BYTES) */
};

/*
 * Prefill / full attention: any Lq >= 1 (Lq <= Lk when causal).
 *
 * scale   multiplies q.k; must be finite and >= 0 (the pages use 1/sqrt(D)).
 * causal  0 or 1; causal rows are aligned bottom-right (p_i = Lk - Lq + i).
 * window  0 (none) or > 0 with causal = 1.
 * workspace / workspace_bytes: optional.  With NULL (or too small a buffer) the
 *   whole visible key range of each query tile is processed by one CTA (pair),
 *   one launch per tile in a single grid.  With at least
 *   sdpa_prefill_workspace_bytes(...) bytes, head_dim 256 runs persistently:
 *   one unit per resident CTA slot takes the query tiles in waves and the last,
 *   partial wave is shared out by key tiles (fp32 partials merged in key
 *   order inside the kernel); head_dim 512 may split long key ranges across
 *   CTAs and merge them in a second kernel.  Either keeps all SMs busy when the
 *   query tiles do not fill whole waves.  A workspace must not be used by two
 *   calls that can run at the same time.
 * Returns SDPA_OK or a negative sdpa_status.  The return value covers argument
 * checks and launches only: call sdpa_device_status() to learn whether the
 * kernels completed.  In the persistent schedule a unit waits (at most 2 s)
 * for the partials of its tile's tail from other units; if that wait gives up
 * (for example because other work on the GPU kept those units from running),
 * the tile's rows are stored as NaN and the status reports 0x10a.
 */
int sdpa_prefill(const void* q, const void* k, const void* v, void* out, int B, int Hq, int Hkv,
                 int Lq, int Lk, int D, float scale, int causal, int window, int dtype,
                 void* workspace, size_t workspace_bytes, sdpa_stream_t stream);

/* Workspace for the persistent (head_dim 256) or split (head_dim 512) prefill
 * schedule; 0 if the call would never use one.  It does not grow with Lk: at
 * most (SM count) x 264 KiB for head_dim 256 (about 40 MB on a GB300), at most
 * 8 * B * Hq * Lq * (D + 2) * 4 bytes for head_dim 512.  Returns 0 for
 * arguments sdpa_prefill would reject. */
size_t sdpa_prefill_workspace_bytes(int B, int Hq, int Hkv, int Lq, int Lk, int D, int causal,
                                    int window);

/* Kernel launches one sdpa_prefill call makes with a workspace of
 * `workspace_bytes` bytes (0 for none): 1 (one attention kernel) or 2 (split
 * key ranges plus the merge kernel); a negative sdpa_status for arguments
 * sdpa_prefill would reject.  Host-only; queues nothing. */
int sdpa_prefill_launches(int B, int Hq, int Hkv, int Lq, int Lk, int D, int causal, int window,
                          size_t workspace_bytes);

/*
 * Decode / speculative verify: 1 <= Lq <= 8 query rows per head over Lk keys.
 *
 * Same arguments and semantics as sdpa_prefill.  The workspace must hold at
 * least sdpa_decode_workspace_bytes(B, Hq, Hkv, Lq, D) bytes; when that is 0
 * (head dims up to 256 whenever one cluster of splits covers each head group)
 * the workspace may be NULL.  The size does not depend on Lk.
 *
 * Row invariance ("fix: Gemma 4 MTP never engages on CUDA (GB10)", sections
 * "Proposed Solution" and "Acceptance Criteria"): row i of a call with Lq = M
 * is bit-identical to the Lq = 1 call with the same B, Hq, Hkv, D, dtype,
 * scale, causal and window whose key/value prefix is trimmed to
 * Lk - M + 1 + i keys.  The key range is cut into 64-key tiles at fixed
 * absolute positions, dealt round-robin over a split count that depends only
 * on (B, Hkv, Hq/Hkv, D, window) and the device, and the splits' partials are
 * merged in a fixed order (head dims up to 256: inside one launch, by the
 * thread-block cluster the splits of a head group form; head dim 512: by a
 * second kernel); a row's arithmetic never depends on the other rows of the
 * call.
 */
int sdpa_decode(const void* q, const void* k, const void* v, void* out, int B, int Hq, int Hkv,
                int Lq, int Lk, int D, float scale, int causal, int window, int dtype,
                void* workspace, size_t workspace_bytes, sdpa_stream_t stream);

/* Workspace bytes sdpa_decode needs on the current device (0 on bad arguments,
 * or when the call needs none).  It is computed without a window and is an
 * upper bound for every window: a windowed call needs at most this much. */
size_t sdpa_decode_workspace_bytes(int B, int Hq, int Hkv, int Lq, int D);

/*
 * Extended prefill / decode: a V head dim that differs from Q/K's, K/V read
 * from a caller's cache instead of packed tensors, and an additive bias.
 *
 * Head dims.  q and k have Dqk columns, v and out have Dv.  Supported: Dqk ==
 * Dv in {128, 192, 256, 512}, and Dqk = 192 with Dv = 256, the Q=192/K=192/
 * V=256 heads that "Fused SDPA full-attention for head_dim=192/256" (MLX PR
 * #3660, thread under "Additional head dimension discovered") names as gated
 * out of the fused path.  Scores are q.k over Dqk; out is the weighted sum of
 * V rows over Dv.  Workspace sizes: sdpa_prefill_workspace_bytes with Dqk,
 * sdpa_decode_workspace_bytes with Dv.
 *
 * K/V caches.  The pages' serving code decodes against KV caches: classic
 * decode and the per-row verify calls read "strided, sliced keys", and
 * sliding-window layers keep their keys in a ring addressed by a cursor ("fix:
 * Gemma 4 MTP never engages on CUDA (GB10), verify probe fails", sections
 * "Current Behavior" and "Proposed Solution"; a wrapped ring and an unwrapped
 * one are both edge cases in "Implementation Notes").
 *  k  [B, Hkv, kv_capacity, Dqk], v [B, Hkv, kv_capacity, Dv], contiguous,
 *     same dtype as q; only the rows below are read.
 *  kv_ring = 0: key j (0 <= j < Lk) is row j; kv_capacity >= Lk (kv_capacity
 *     = Lk is the packed layout of sdpa_prefill / sdpa_decode).
 *  kv_ring = 1: key j is row (j mod kv_capacity): the cache holds the last
 *     kv_capacity keys.  kv_capacity must be a multiple of 128 and hold every
 *     key some query row can see: min(Lk, Lq + window - 1) keys with a window,
 *     all Lk keys without one.  Rows of the ring that no query row can see are
 *     read but weighted by exactly 0; they must hold finite values.
 * The layout changes only which row holds a key: results equal, bit for bit,
 * the same call on packed copies of the keys, so decode row invariance holds
 * over the trimmed prefix of the same cache.
 *
 * Additive bias (a mask array).  "fix: gemma-4 long-prompt prefill OOMs on
 * CUDA" (mlxcel issue #672, sections "Root cause" and "Suggested fix
 * direction") describes models that hand attention a dense additive mask (0 for
 * a visible key, -inf for a hidden one) and cuDNN's flash path that takes such
 * a mask as a bias.  With bias != NULL the score of query row i and key j is
 *     scale * q_i . k_j + bias[b * bias_stride_b + h * bias_stride_h
 *                              + i * bias_stride_q + j]
 * for query head h, on top of the causal / window flags (keys they hide stay
 * hidden).  The bias is in q's dtype, device memory, owned by the caller and
 * only read; strides are in elements and >= 0, and a stride of 0 broadcasts
 * (a [1, 1, Lq, Lk] mask shared by all heads has bias_stride_b =
 * bias_stride_h = 0, bias_stride_q = Lk).  Key j is the logical key position
 * 0..Lk-1, also for a ring cache.  Entries may be finite or -inf (not +inf or
 * NaN); a row whose keys are all hidden outputs zeros.  Base and strides that
 * are multiples of 16 bytes are read in vectors, others element by element.
 * Negative or huge strides: SDPA_ERR_INVALID_ARG; an odd address:
 * SDPA_ERR_ALIGNMENT.  bias = NULL: no bias (strides ignored).
 *
 * Everything else is as for sdpa_prefill / sdpa_decode.  Unsupported head dims
 * return SDPA_ERR_UNSUPPORTED and layout errors SDPA_ERR_INVALID_ARG before
 * anything is queued.
 */
int sdpa_prefill_ex(const void* q, const void* k, const void* v, void* out, int B, int Hq,
                    int Hkv, int Lq, int Lk, int Dqk, int Dv, float scale, int causal, int window,
                    int dtype, int kv_capacity, int kv_ring, const void* bias,
                    long long bias_stride_b, long long bias_stride_h, long long bias_stride_q,
                    void* workspace, size_t workspace_bytes, sdpa_stream_t stream);

int sdpa_decode_ex(const void* q, const void* k, const void* v, void* out, int B, int Hq, int Hkv,
                   int Lq, int Lk, int Dqk, int Dv, float scale, int causal, int window,
                   int dtype, int kv_capacity, int kv_ring, const void* bias,
                   long long bias_stride_b, long long bias_stride_h, long long bias_stride_q,
                   void* workspace, size_t workspace_bytes, sdpa_stream_t stream);

/* Synchronises `stream`, returns SDPA_OK or SDPA_ERR_DEVICE_TIMEOUT for the
 * current device and clears the status word.  *detail (if not NULL) receives
 * the raw device code (0 if none): 0x100..0x10a identify the pipeline wait that
 * gave up, 0x10b a shared-memory window that was not 1024-byte aligned, 0x10c a
 * 2-CTA kernel that found itself outside a cluster of two (or a decode kernel
 * in a cluster of another size than planned), 0x10d a decode CTA beyond the
 * planned grid.  In every case the
 * kernel stopped without touching memory it should not and its output is
 * unspecified. */
int sdpa_device_status(sdpa_stream_t stream, int* detail);

/* Human-readable text for an sdpa_status value (static storage). */
const char* sdpa_status_string(int status);

/* Library ABI version (major * 100 + minor). */
int sdpa_version(void);

/*
 * Self-test of the device-side failure path: runs one small fp16 call
 * (B = 1, Hq = 2, Hkv = 1, Lk = 128, head_dim D in {256, 512}; prefill with
 * Lq = 128, or decode with Lq = 1 when `decode` is 1) in which the "query tile
 * ready" signal is deliberately withheld.  The kernel's bounded wait for it
 * gives up after about 2 s, every CTA drains its copies and MMAs and exits, and
 * the call returns what sdpa_device_status() then reports:
 * SDPA_ERR_DEVICE_TIMEOUT, with *detail the code (0x100..0x10a) of the first
 * wait that gave up: the query-tile wait itself (0x100) or one that depends on
 * it.  No fault, trap or hang is involved; the CUDA context stays usable.
 * q, k, v, out: device buffers of the shapes above ([1,2,Lq,D], [1,1,128,D]);
 * decode also needs a workspace of sdpa_decode_workspace_bytes(1, 2, 1, 1, D).
 *
 * decode = 2 tests the persistent prefill schedule instead: D = 256, Lq = 256,
 * Lk = 4096 (q [1,2,256,256], k and v [1,1,4096,256]) with a workspace of
 * sdpa_prefill_workspace_bytes(1, 2, 1, 256, 4096, 256, 1, 0) bytes.  The
 * pieces that compute the tail of a query tile's key range never publish
 * their "partials ready" flags, so each unit that owns such a tile gives up
 * its bounded wait for them (code 0x10a), merges nothing and stores NaN rows
 * for that tile.  SDPA_ERR_UNSUPPORTED if the device's schedule has no such
 * pieces for this shape.
 */
int sdpa_selftest_timeout(const void* q, const void* k, const void* v, void* out, int D,
                          int decode, void* workspace, size_t workspace_bytes,
                          sdpa_stream_t stream, int* detail);

/*
 * sdpa_decode_noalloc -- sdpa_decode for callers that cannot allocate device
 * memory.  (The paper, i.e. the web pages this library follows, has no
 * counterpart of this entry point; it is a convenience of this library.)
 *
 * Who needs it: code that runs inside a host runtime which owns the device
 * heap and forbids allocation on its execution path (for example a plugin
 * whose enqueue callback may only launch work), and latency-critical loops
 * where a cudaMalloc, with the device-wide synchronisation it can imply, is
 * not acceptable.  Such callers cannot hand sdpa_decode a workspace.
 *
 * Instead of a caller workspace this entry point uses a scratch array of
 * SDPA_NOALLOC_SCRATCH_BYTES that lives in the library itself (a static
 * __device__ array: every GPU that loads the library holds it until the
 * process exits).  It calls no cudaMalloc, cudaFree or other allocating
 * routine.  The caller still provides q, k, v and out exactly as for
 * sdpa_decode, and the results are those of sdpa_decode.
 *
 *  - The first call on each device looks up the device address of the scratch
 *    array (cudaGetSymbolAddress with that device current); make that first
 *    call before any stream capture on that device.
 *  - A call whose split partials need more than SDPA_NOALLOC_SCRATCH_BYTES is
 *    rejected with SDPA_ERR_SCRATCH_LIMIT before anything is queued; the need
 *    is at most what sdpa_decode_workspace_bytes(B, Hq, Hkv, Lq, D) reports
 *    (a windowed call may need less, and calls whose head groups are each
 *    covered by one cluster of splits need none).
 *  - Every call on a device shares the one array, and the array keeps the
 *    previous call's contents.  Nothing in it has to start at zero: each call
 *    writes every partial it later reads.  Two calls whose work overlaps on
 *    the GPU (different streams, no ordering between them) race on the array
 *    and give wrong results: serialise them, e.g. on one stream.
 */
#define SDPA_NOALLOC_SCRATCH_BYTES ((size_t)24 << 20)
int sdpa_decode_noalloc(const void* q, const void* k, const void* v, void* out, int B, int Hq,
                        int Hkv, int Lq, int Lk, int D, float scale, int causal, int window,
                        int dtype, sdpa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SDPA_GB300_H_ */
