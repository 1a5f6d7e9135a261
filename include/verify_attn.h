/*
 * verify_attn.h -- C ABI of libverify_attn: tree-verify attention for
 * speculative decoding over a paged MLA latent KV pool (page_size = 1), for
 * NVIDIA GB300 (sm_103a).
 *
 * The operation ("The Capture-Safe Kernel", sections The Core Problem and
 * The Design Decisions; "The Integration Chasm", sections Decision and
 * Subject Message; "The Launch Wrapper", section Input):
 *
 *   For request b of a ragged batch, T_b = qo_indptr[b+1]-qo_indptr[b] draft
 *   tokens x H heads attend to N_b = L_b + T_b keys, L_b =
 *   kv_indptr[b+1]-kv_indptr[b] (derived in-kernel, Decision 2).  Key j < L_b
 *   is pool row kv_indices[kv_indptr[b]+j]; key j >= L_b is draft token
 *   j-L_b, pool row out_cache_loc[qo_indptr[b]+j-L_b] (Decision 1: native
 *   buffers read in place).  Draft i sees key j iff bit mask_indptr[b] +
 *   i*N_b + j of custom_mask is set (Decision 5), LSB-first in each byte.
 *   With K_j = pool[slot_j, 0:576] and V_j = pool[slot_j, 0:512] (MLA latent
 *   attention after absorption: 512 no-PE + 64 RoPE dims per row, V = the
 *   no-PE part):
 *       out[t, h, :] = softmax_j( sm_scale * <q[t,h,:], K_j> ) . V_j
 *   over the visible j.  A row with no visible key gets zeros.
 *
 *   The library computes it as split-KV flash-decode ("The Integration
 *   Chasm", section Context: KV-split partial-plus-reduce; "The Capture-Safe
 *   Kernel", Decision 3): each split covers a contiguous key chunk and writes
 *   a partial output plus its log-sum-exp into the workspace; a second
 *   kernel merges the partials.
 *
 * Contract of every entry point that takes a stream:
 *   - all tensor pointers are DEVICE pointers owned by the caller;
 *   - the library keeps no per-call state, allocates no device memory and
 *     never synchronises, so a call can be captured into a CUDA graph and
 *     replayed after the caller rewrites the *contents* of its buffers
 *     (Decision 6: no replay-metadata hook needed).  Work is ordered on
 *     `stream` (0 = legacy default stream): when a call may hold requests
 *     of both tensor-core cluster shapes (max_q_per_req * num_heads > 128),
 *     the small requests' launch runs on `stream` and the large requests'
 *     launch on a library-owned second stream, forked from `stream` by an
 *     event before them and joined back by an event before the combine,
 *     which stream capture records as a fork and a join of the graph.  Per device the library holds that stream, its
 *     two events (created by verify_attn_init) and the tensor-map
 *     descriptors of the last pool it saw (host memory);
 *   - host-side argument errors are reported by a negative VA_ERR_* return
 *     and nothing is launched;
 *   - device-side data errors never trap: a slot id outside [0, pool_size)
 *     (or a null index buffer that a request needs) makes the kernel skip
 *     that key and OR bit VA_STATUS_BAD_SLOT into the 32-bit status word at
 *     byte 0 of the workspace; each run clears that word first.  The caller
 *     reads it after its own synchronisation.
 *
 * Thread safety: calls may be made from several host threads; concurrent
 * calls must use distinct workspaces.  A mixed-shape call launches its
 * large requests on a second stream that belongs to the calling host thread
 * (one per thread and device, created by that thread's first
 * verify_attn_init or mixed call), so calls and stream captures made from
 * different threads never share it, and their launches may overlap.  Within
 * one thread, a stream capture that has recorded a mixed-shape call holds
 * that thread's second stream until the capture ends (the forked stream
 * belongs to the capture): make no mixed-shape call on another stream from
 * the same thread meanwhile (its fork would wait on an event recorded in
 * the capture, and the call can fail with VA_ERR_LAUNCH).
 */
#ifndef VERIFY_ATTN_H
#define VERIFY_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Symbols of this header are the library's only exported names. */
#if defined(__GNUC__)
#define VERIFY_ATTN_API __attribute__((visibility("default")))
#else
#define VERIFY_ATTN_API
#endif

/* Opaque CUDA stream handle (the same object as cudaStream_t / CUstream). */
typedef struct CUstream_st *verify_attn_stream_t;

/* Fixed latent geometry: 576-wide rows (512 no-PE + 64 RoPE), V = first 512. */
#define VERIFY_ATTN_LATENT_DIM 576
#define VERIFY_ATTN_V_DIM 512
/* Upper bound on num_splits accepted by the run entry points. */
#define VERIFY_ATTN_MAX_SPLITS 256

enum verify_attn_status {
    VA_OK = 0,
    VA_ERR_NULL = -1,       /* a required pointer is null                          */
    VA_ERR_ALIGN = -2,      /* q/kv_pool/out not 16-B aligned, strides not x8 elems,
                               or workspace not 256-B aligned                        */
    VA_ERR_DIMS = -3,       /* batch/heads/max_q_per_req/pool_size out of range     */
    VA_ERR_WORKSPACE = -4,  /* workspace_bytes < verify_attn_workspace_size(...)   */
    VA_ERR_SPLITS = -5,     /* num_splits outside [1, VERIFY_ATTN_MAX_SPLITS]       */
    VA_ERR_LAUNCH = -6,     /* a CUDA launch or attribute call failed               */
    VA_ERR_SCALE = -7,      /* sm_scale not finite                                   */
    VA_ERR_DEVICE = -8,     /* the current device is not sm_103 or cannot be queried */
    VA_ERR_SCRATCH_LIMIT = -9, /* verify_attn_run_static: the capacities need more
                                  scratch than VERIFY_ATTN_STATIC_SCRATCH_BYTES      */
};

/* Bits of the device status word (workspace byte 0). */
#define VA_STATUS_BAD_SLOT 0x1u   /* slot outside [0,pool_size) or null index buffer */
#define VA_STATUS_BAD_META 0x2u   /* some T_b > max_q_per_req, or negative lengths;
                                     rows past the capacity are not computed        */
#define VA_STATUS_TIMEOUT 0x4u    /* a bounded wait inside a kernel expired (1 s); the
                                     output of that call is not valid               */

/*
 * Workspace bytes needed by verify_attn_run / verify_attn_run_simt for a
 * call with these capacities: a 256-B header (status word), then fp32 split
 * partials [num_splits][batch*max_q_per_req*num_heads][512] and their
 * log-sum-exp [num_splits][batch*max_q_per_req*num_heads].  The caller
 * allocates it (e.g. torch.empty(..., dtype=uint8, device="cuda")) --
 * "The Capture-Safe Kernel", Decision 4: workspace as a caller tensor, not a
 * raw cudaMalloc.  Returns 0 for invalid capacities.
 */
VERIFY_ATTN_API size_t verify_attn_workspace_size(int batch, int max_q_per_req, int num_heads, int num_splits);

/*
 * One-time per-device setup for the current device: kernel attributes such
 * as the dynamic shared-memory limit, the calling thread's second stream and
 * its events (each host thread that captures mixed-shape calls should call
 * it once before capturing), and
 * the loading of the module that holds verify_attn_run_static's 32 MiB
 * array (which commits that memory).  Every entry point calls it lazily,
 * but callers that capture CUDA graphs should call it once before
 * capturing, and callers that reserve most of the GPU's memory should call
 * it before reserving.  Returns VA_OK, VA_ERR_DEVICE or VA_ERR_LAUNCH.
 */
VERIFY_ATTN_API int verify_attn_init(void);

/*
 * Tree-verify attention, production path (tensor-core split kernel on
 * sm_103a, then the log-sum-exp combine).
 *
 *   q            [sum T_b, H, 576] bf16; element (t,h,d) at
 *                q[t*q_stride_tok + h*q_stride_head + d]; strides in
 *                elements, multiples of 8; 16-B aligned base.
 *   kv_pool      [pool_size, 576] bf16, rows contiguous (1152 B), 16-B aligned.
 *                The tensor-core kernel addresses rows with 32-bit TMA
 *                coordinates, so a pool of 2^31 rows or more (2.5 TB, more
 *                than one GPU holds) runs on the CUDA-core kernel instead.
 *   qo_indptr    [batch+1] int32, non-decreasing, qo_indptr[0] = 0, every
 *                T_b <= max_q_per_req.
 *   kv_indptr    [batch+1] int32, non-decreasing, kv_indptr[0] = 0 (prefix keys).
 *   kv_indices   [kv_indptr[batch]] int32 pool slots of the prefix keys.
 *   out_cache_loc[qo_indptr[batch]] int64 pool slots of the draft tokens.
 *   custom_mask  packed visibility bits (layout above).
 *   mask_indptr  [batch+1] int64 bit offsets; mask_indptr[b+1]-mask_indptr[b]
 *                = T_b*(L_b+T_b).
 *   sm_scale     softmax scale applied to <q, K> (e.g. 1/sqrt(192)).
 *   out          [sum T_b, H, 512] bf16 (round to nearest even), strides like q.
 *   batch, max_q_per_req, num_heads, num_splits: host capacities that fix
 *                the launch grid (so one captured graph serves every batch
 *                with these bounds).  Request b's keys are cut into chunks of
 *                c_b = max(ceil(N_b/num_splits), 256) rounded up to a multiple
 *                of 128; splits past the end exit at once (Decision 3).
 *   workspace    device scratch of workspace_bytes (see above), 256-B aligned.
 *
 * The index buffers and the mask are read in place, inside the kernels; the
 * call allocates nothing and does not synchronise.  Returns VA_OK or a
 * negative VA_ERR_*.
 */
VERIFY_ATTN_API int verify_attn_run(const void *q, int64_t q_stride_tok, int64_t q_stride_head,
                                    const void *kv_pool, int64_t pool_size,
                                    const int32_t *qo_indptr, const int32_t *kv_indptr,
                                    const int32_t *kv_indices, const int64_t *out_cache_loc,
                                    const uint8_t *custom_mask, const int64_t *mask_indptr,
                                    float sm_scale,
                                    void *out, int64_t out_stride_tok, int64_t out_stride_head,
                                    int batch, int max_q_per_req, int num_heads, int num_splits,
                                    void *workspace, size_t workspace_bytes,
                                    verify_attn_stream_t stream);

/*
 * Same operation and arguments on the portable CUDA-core kernel (fp32 FMA,
 * no tensor cores).  It is the side-by-side cross-check of the production
 * kernel on live buffers, in the spirit of the pages' "validate" mode ("The
 * Launch Wrapper", section The Design Decision: Three Modes of Operation).
 */
VERIFY_ATTN_API int verify_attn_run_simt(const void *q, int64_t q_stride_tok, int64_t q_stride_head,
                                         const void *kv_pool, int64_t pool_size,
                                         const int32_t *qo_indptr, const int32_t *kv_indptr,
                                         const int32_t *kv_indices, const int64_t *out_cache_loc,
                                         const uint8_t *custom_mask, const int64_t *mask_indptr,
                                         float sm_scale,
                                         void *out, int64_t out_stride_tok, int64_t out_stride_head,
                                         int batch, int max_q_per_req, int num_heads, int num_splits,
                                         void *workspace, size_t workspace_bytes,
                                         verify_attn_stream_t stream);

/* Kernel selectors for verify_attn_run_profiled. */
#define VERIFY_ATTN_IMPL_TC 0     /* the verify_attn_run path   */
#define VERIFY_ATTN_IMPL_SIMT 1   /* the verify_attn_run_simt path */

/*
 * verify_attn_run (impl = VERIFY_ATTN_IMPL_TC) or verify_attn_run_simt
 * (VERIFY_ATTN_IMPL_SIMT) with timing marks: events[0..3] are cudaEvent_t
 * handles created by the caller (any may be null), recorded on `stream`
 * at the start of the call, just before the split kernel (after the status
 * word is cleared), between the split kernel and the combine, and after the
 * combine.  Lets a caller time each of the two kernels on the stream they
 * run on.  Under stream capture the marks are recorded as external event
 * records (cudaEventRecordExternal), so they become event-record nodes of the
 * graph and time every replay.  Same return codes; an unknown impl gives
 * VA_ERR_DIMS.
 */
VERIFY_ATTN_API int verify_attn_run_profiled(int impl, void *const *events,
                                             const void *q, int64_t q_stride_tok, int64_t q_stride_head,
                                             const void *kv_pool, int64_t pool_size,
                                             const int32_t *qo_indptr, const int32_t *kv_indptr,
                                             const int32_t *kv_indices, const int64_t *out_cache_loc,
                                             const uint8_t *custom_mask, const int64_t *mask_indptr,
                                             float sm_scale,
                                             void *out, int64_t out_stride_tok, int64_t out_stride_head,
                                             int batch, int max_q_per_req, int num_heads, int num_splits,
                                             void *workspace, size_t workspace_bytes,
                                             verify_attn_stream_t stream);

/*
 * Largest workspace verify_attn_run_static can stand in for: 32 MiB, held in
 * a fixed array inside the library on every GPU that loads it.
 */
#define VERIFY_ATTN_STATIC_SCRATCH_BYTES ((size_t)32 << 20)

/*
 * verify_attn_run without a workspace argument, for callers that cannot
 * allocate device memory: engines that reserve almost all GPU memory for
 * their KV pool up front and allow no later allocation, host programs that
 * load this library as a plug-in without giving it an allocator, or paths
 * where an allocation would synchronise the device.  (The pages have no
 * counterpart: their workspace is always a caller tensor.)
 *
 * The library supplies the scratch itself, from a fixed 32 MiB device array
 * (VERIFY_ATTN_STATIC_SCRATCH_BYTES) compiled into it.  Capacities whose
 * verify_attn_workspace_size(...) exceeds that are rejected with
 * VA_ERR_SCRATCH_LIMIT before anything is launched.  The call allocates
 * nothing (no cudaMalloc, no cudaFree, no allocating library routine).
 *
 * Set-up: the array's memory is committed on a device when the library's
 * module holding it loads there, which verify_attn_init() forces.  Call
 * verify_attn_init() on each device at start-up, before reserving the rest
 * of its memory and before any stream capture; otherwise the first call of
 * any entry point does it (and could then fail with VA_ERR_LAUNCH for lack
 * of memory).  Each call looks the array's device address up again, so no
 * address is cached across calls.
 *
 * Sharing: all calls on a device use the one array and it keeps the last
 * call's contents; each call clears the part that must start at zero (the
 * status word).  Calls whose GPU work overlaps -- for instance on two
 * streams at once -- race on that array, so serialise them.  The status word
 * of the last call is readable through verify_attn_static_status_word().
 *
 * The library's per-device state (this array's module, the per-thread
 * second streams and events, the tensor-map cache) belongs to the device's
 * primary context:
 * after cudaDeviceReset, or under another context, it is not valid.
 *
 * Arguments, layouts and the other return codes are those of
 * verify_attn_run (a device that is not sm_103 gives VA_ERR_DEVICE).
 */
VERIFY_ATTN_API int verify_attn_run_static(const void *q, int64_t q_stride_tok, int64_t q_stride_head,
                                           const void *kv_pool, int64_t pool_size,
                                           const int32_t *qo_indptr, const int32_t *kv_indptr,
                                           const int32_t *kv_indices, const int64_t *out_cache_loc,
                                           const uint8_t *custom_mask, const int64_t *mask_indptr,
                                           float sm_scale,
                                           void *out, int64_t out_stride_tok, int64_t out_stride_head,
                                           int batch, int max_q_per_req, int num_heads, int num_splits,
                                           verify_attn_stream_t stream);

/*
 * Device address of the status word that verify_attn_run_static calls on
 * the current device write (bits VA_STATUS_*, as at workspace byte 0 of
 * verify_attn_run): after its own synchronisation a caller of
 * verify_attn_run_static reads the 32-bit word there (for instance with
 * cudaMemcpy to a host variable) to learn of bad slots, bad metadata or a
 * timed-out wait in the last call.  The pointer is device memory of the
 * library's static array; it stays valid until the process exits (see the
 * context note above).  Allocates nothing.  Returns VA_OK, VA_ERR_NULL
 * (status is null), VA_ERR_DEVICE or VA_ERR_LAUNCH.  (The pages have no
 * counterpart.)
 */
VERIFY_ATTN_API int verify_attn_static_status_word(unsigned int **status);

/*
 * KV save of the draft tokens ("The Launch Wrapper", section The KV Cache
 * Ordering Insight: the new tokens' latent rows are written into the pool
 * before the attention reads them):
 *     kv_pool[out_cache_loc[i], :] = kv_new[i, :]   for i in [0, num_tokens).
 *
 *   kv_new        [num_tokens, 576] bf16; row i at kv_new + i*kv_new_stride_tok
 *                 (elements, a multiple of 8, >= 576); 16-B aligned base.
 *   out_cache_loc [num_tokens] int64 destination slots.  Slots are expected
 *                 to be distinct (which write lands for a repeated slot is
 *                 unspecified); a slot outside [0, pool_size) is skipped and
 *                 sets VA_STATUS_BAD_SLOT.
 *   kv_pool       [pool_size, 576] bf16, written in place; 16-B aligned.
 *   workspace     at least 256 bytes, 256-B aligned: the status word at byte
 *                 0 is cleared, then set by the kernel (read it after a sync).
 *
 * One launch on `stream`; allocates nothing, does not synchronise.  Returns
 * VA_OK, VA_ERR_NULL, VA_ERR_ALIGN, VA_ERR_DIMS (num_tokens < 0 or
 * pool_size <= 0), VA_ERR_WORKSPACE, VA_ERR_DEVICE or VA_ERR_LAUNCH.
 */
VERIFY_ATTN_API int verify_attn_save_kv(const void *kv_new, int64_t kv_new_stride_tok,
                                        const int64_t *out_cache_loc, int64_t num_tokens,
                                        void *kv_pool, int64_t pool_size,
                                        void *workspace, size_t workspace_bytes,
                                        verify_attn_stream_t stream);

/*
 * The KV save of the draft tokens, then verify_attn_run, on `stream`: the
 * save kernel writes rows [0, qo_indptr[batch]) of kv_new ([sum T_b, 576]
 * bf16, row stride kv_new_stride_tok elements, a multiple of 8, >= 576) to
 * kv_pool at out_cache_loc, and the attention that follows reads them.  The
 * save grid covers batch * max_q_per_req rows and reads the real count from
 * qo_indptr on the device, so one captured graph serves every batch within
 * the capacities.  The status word collects the save's and the attention's
 * bits.  Other arguments and return codes are those of verify_attn_run.
 */
VERIFY_ATTN_API int verify_attn_save_and_run(const void *kv_new, int64_t kv_new_stride_tok,
                                             const void *q, int64_t q_stride_tok, int64_t q_stride_head,
                                             void *kv_pool, int64_t pool_size,
                                             const int32_t *qo_indptr, const int32_t *kv_indptr,
                                             const int32_t *kv_indices, const int64_t *out_cache_loc,
                                             const uint8_t *custom_mask, const int64_t *mask_indptr,
                                             float sm_scale,
                                             void *out, int64_t out_stride_tok, int64_t out_stride_head,
                                             int batch, int max_q_per_req, int num_heads, int num_splits,
                                             void *workspace, size_t workspace_bytes,
                                             verify_attn_stream_t stream);

/* Bounds of verify_attn_check_wait_timeout's limit: 1 us to 1 s. */
#define VERIFY_ATTN_WAIT_PROBE_MIN_NS 1000ull
#define VERIFY_ATTN_WAIT_PROBE_MAX_NS 1000000000ull

/*
 * Self-test of the kernels' failure path ("The Launch Wrapper", section The
 * Design Decision: Three Modes of Operation: a failed kernel must leave the
 * service able to fall back).  Every wait inside the split kernels is
 * bounded: when it expires the kernel sets VA_STATUS_TIMEOUT, unwinds and
 * returns instead of hanging the GPU.  This call launches one small kernel
 * whose single warp runs that same bounded wait on a barrier nothing ever
 * arrives on, with a limit of limit_ns nanoseconds (the split kernels use
 * 1 s), so the expiry path runs on demand.  On `stream`: clears the status
 * word at workspace byte 0, then the kernel sets VA_STATUS_TIMEOUT in it
 * and returns after about limit_ns; the caller reads the word after its own
 * synchronisation, and the context stays usable for normal calls.
 *
 *   workspace   at least 256 bytes, 256-B aligned (device memory).
 *   limit_ns    in [VERIFY_ATTN_WAIT_PROBE_MIN_NS, VERIFY_ATTN_WAIT_PROBE_MAX_NS].
 *
 * Allocates nothing, does not synchronise.  Returns VA_OK, VA_ERR_NULL,
 * VA_ERR_ALIGN, VA_ERR_WORKSPACE, VA_ERR_DIMS (limit out of bounds),
 * VA_ERR_DEVICE or VA_ERR_LAUNCH.
 */
VERIFY_ATTN_API int verify_attn_check_wait_timeout(uint64_t limit_ns, void *workspace, size_t workspace_bytes,
                                                   verify_attn_stream_t stream);

/* Short English description of a VA_* status code (static storage). */
VERIFY_ATTN_API const char *verify_attn_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* VERIFY_ATTN_H */
