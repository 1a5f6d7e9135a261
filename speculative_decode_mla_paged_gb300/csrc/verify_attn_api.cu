// Host side of the C ABI declared in include/verify_attn.h: argument
// checks, workspace carving, per-device one-time setup and the launches.
// Nothing here allocates device memory or synchronises ("The Capture-Safe
// Kernel", section The Core Problem: host syncs, raw cudaMalloc and
// temporaries are what break graph capture).
#include "verify_attn.h"
#include "va_internal.cuh"

#include <atomic>
#include <math.h>

// The ABI's constants and the kernels' own must agree.
static_assert(va::D == VERIFY_ATTN_LATENT_DIM && va::DV == VERIFY_ATTN_V_DIM, "latent row and V widths");
static_assert(va::STATUS_BAD_SLOT == VA_STATUS_BAD_SLOT && va::STATUS_BAD_META == VA_STATUS_BAD_META &&
                  va::STATUS_TIMEOUT == VA_STATUS_TIMEOUT,
              "device status bits");

namespace va {

cudaError_t tc_init();
cudaError_t tc_thread_init();
cudaError_t launch_tc_split(const Params &p, cudaStream_t stream);
bool tc_supported(const Params &p);
int static_scratch_setup();   // verify_attn_static.cu
cudaError_t launch_wait_probe(unsigned *status, uint64_t limit_ns, cudaStream_t stream);

namespace {

std::atomic<uint64_t> g_init_mask{0};   // bit d: device d initialised

int ensure_init()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return VA_ERR_DEVICE;
    const uint64_t bit = 1ull << dev;
    if (g_init_mask.load(std::memory_order_acquire) & bit) return VA_OK;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return VA_ERR_DEVICE;
    if (major != 10 || minor != 3) return VA_ERR_DEVICE;   // built for sm_103a only
    if (simt_init() != cudaSuccess) return VA_ERR_LAUNCH;
    if (tc_init() != cudaSuccess) return VA_ERR_LAUNCH;
    // The static-scratch entry point's array: its memory is committed now,
    // while the caller can still make room, not at that entry point's first call.
    if (static_scratch_setup() != VA_OK) return VA_ERR_LAUNCH;
    g_init_mask.fetch_or(bit, std::memory_order_acq_rel);
    return VA_OK;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

size_t ws_size(int batch, int max_q, int heads, int splits)
{
    if (batch < 0 || max_q < 0 || heads <= 0 || splits < 1 || splits > VERIFY_ATTN_MAX_SPLITS)
        return 0;
    const size_t rows = (size_t)batch * (size_t)max_q * (size_t)heads;
    const size_t o_bytes = (size_t)splits * rows * DV * sizeof(float);
    const size_t lse_bytes = (size_t)splits * rows * sizeof(float);
    return WS_HEADER + o_bytes + ((lse_bytes + 255) & ~(size_t)255);
}

// Validate host arguments and fill Params.  Returns VA_OK or VA_ERR_*.
int prepare(Params &p, const void *q, int64_t q_st, int64_t q_sh, const void *kv_pool,
            int64_t pool_size, const int32_t *qo_indptr, const int32_t *kv_indptr,
            const int32_t *kv_indices, const int64_t *out_cache_loc, const uint8_t *custom_mask,
            const int64_t *mask_indptr, float sm_scale, void *out, int64_t o_st, int64_t o_sh,
            int batch, int max_q, int heads, int splits, void *workspace, size_t ws_bytes)
{
    if (!q || !kv_pool || !qo_indptr || !kv_indptr || !custom_mask || !mask_indptr || !out ||
        !workspace)
        return VA_ERR_NULL;
    if (batch < 0 || max_q < 0 || heads <= 0 || pool_size <= 0) return VA_ERR_DIMS;
    if ((int64_t)batch * max_q * heads > (int64_t)1 << 31) return VA_ERR_DIMS;
    if (splits < 1 || splits > VERIFY_ATTN_MAX_SPLITS) return VA_ERR_SPLITS;
    if (!isfinite(sm_scale)) return VA_ERR_SCALE;
    if (!aligned(q, 16) || !aligned(kv_pool, 16) || !aligned(out, 16) || !aligned(workspace, 256))
        return VA_ERR_ALIGN;
    if ((q_st | q_sh | o_st | o_sh) & 7) return VA_ERR_ALIGN;
    if (q_st < 0 || q_sh < 0 || o_st < 0 || o_sh < 0) return VA_ERR_ALIGN;
    const size_t need = ws_size(batch, max_q, heads, splits);
    if (need == 0) return VA_ERR_DIMS;
    if (ws_bytes < need) return VA_ERR_WORKSPACE;

    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.q_stride_tok = q_st;
    p.q_stride_head = q_sh;
    p.kv_pool = static_cast<const __nv_bfloat16 *>(kv_pool);
    p.pool_size = pool_size;
    p.qo_indptr = qo_indptr;
    p.kv_indptr = kv_indptr;
    p.kv_indices = kv_indices;
    p.out_cache_loc = out_cache_loc;
    p.custom_mask = custom_mask;
    p.mask_indptr = mask_indptr;
    p.sm_scale = sm_scale;
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.out_stride_tok = o_st;
    p.out_stride_head = o_sh;
    p.batch = batch;
    p.max_q_per_req = max_q;
    p.num_heads = heads;
    p.num_splits = splits;
    p.rows_cap = (int64_t)batch * max_q * heads;
    p.rows_lo = -1;
    p.rows_hi = INT64_MAX;
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    p.status = reinterpret_cast<unsigned *>(ws);
    p.part_o = reinterpret_cast<float *>(ws + WS_HEADER);
    p.part_lse = reinterpret_cast<float *>(ws + WS_HEADER + (size_t)splits * p.rows_cap * DV * sizeof(float));
    return VA_OK;
}

enum class Impl { Tc, Simt };

// Draft rows to write into the pool before the attention (verify_attn_save_and_run).
struct SaveArgs {
    const void *kv_new;
    int64_t stride_tok;
};

int run(Impl impl, const void *q, int64_t q_st, int64_t q_sh, const void *kv_pool,
        int64_t pool_size, const int32_t *qo_indptr, const int32_t *kv_indptr,
        const int32_t *kv_indices, const int64_t *out_cache_loc, const uint8_t *custom_mask,
        const int64_t *mask_indptr, float sm_scale, void *out, int64_t o_st, int64_t o_sh,
        int batch, int max_q, int heads, int splits, void *workspace, size_t ws_bytes,
        verify_attn_stream_t stream, cudaEvent_t const *events = nullptr, const SaveArgs *save = nullptr)
{
    Params p;
    int rc = prepare(p, q, q_st, q_sh, kv_pool, pool_size, qo_indptr, kv_indptr, kv_indices,
                     out_cache_loc, custom_mask, mask_indptr, sm_scale, out, o_st, o_sh, batch,
                     max_q, heads, splits, workspace, ws_bytes);
    if (rc != VA_OK) return rc;
    if (save != nullptr) {
        if (save->kv_new == nullptr || out_cache_loc == nullptr) return VA_ERR_NULL;
        if (!aligned(save->kv_new, 16) || (save->stride_tok & 7) || save->stride_tok < D) return VA_ERR_ALIGN;
    }
    rc = ensure_init();
    if (rc != VA_OK) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // Under stream capture the marks are external records (event-record nodes
    // of the graph, so every replay records them); otherwise plain records.
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (events != nullptr && cudaStreamIsCapturing(s, &cap) != cudaSuccess) return VA_ERR_LAUNCH;
    const unsigned rec_flags = cap == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : cudaEventRecordDefault;
    auto mark = [&](int k) {
        return events == nullptr || events[k] == nullptr ||
               cudaEventRecordWithFlags(events[k], s, rec_flags) == cudaSuccess;
    };
    if (!mark(0)) return VA_ERR_LAUNCH;
    if (cudaMemsetAsync(p.status, 0, sizeof(unsigned), s) != cudaSuccess) return VA_ERR_LAUNCH;
    if (save != nullptr &&
        launch_kv_save(static_cast<const __nv_bfloat16 *>(save->kv_new), save->stride_tok, out_cache_loc,
                       (int64_t)batch * max_q, qo_indptr + batch, const_cast<__nv_bfloat16 *>(p.kv_pool), pool_size,
                       p.status, s) != cudaSuccess)
        return VA_ERR_LAUNCH;
    if (!mark(1)) return VA_ERR_LAUNCH;
    cudaError_t e = cudaSuccess;
    if (p.rows_cap > 0) {
        if (impl == Impl::Tc && tc_supported(p))
            e = launch_tc_split(p, s);
        else
            e = launch_simt_split(p, s);
    }
    if (e != cudaSuccess || !mark(2)) return VA_ERR_LAUNCH;
    if (p.rows_cap > 0 && launch_combine(p, s) != cudaSuccess) return VA_ERR_LAUNCH;
    if (!mark(3)) return VA_ERR_LAUNCH;
    return VA_OK;
}

}  // namespace
}  // namespace va

extern "C" {

size_t verify_attn_workspace_size(int batch, int max_q_per_req, int num_heads, int num_splits)
{
    return va::ws_size(batch, max_q_per_req, num_heads, num_splits);
}

int verify_attn_init(void)
{
    const int rc = va::ensure_init();
    if (rc != VA_OK) return rc;
    // the calling thread's second stream, made here rather than inside a capture
    return va::tc_thread_init() == cudaSuccess ? VA_OK : VA_ERR_LAUNCH;
}

int verify_attn_run(const void *q, int64_t q_stride_tok, int64_t q_stride_head, const void *kv_pool,
                    int64_t pool_size, const int32_t *qo_indptr, const int32_t *kv_indptr,
                    const int32_t *kv_indices, const int64_t *out_cache_loc,
                    const uint8_t *custom_mask, const int64_t *mask_indptr, float sm_scale,
                    void *out, int64_t out_stride_tok, int64_t out_stride_head, int batch,
                    int max_q_per_req, int num_heads, int num_splits, void *workspace,
                    size_t workspace_bytes, verify_attn_stream_t stream)
{
    return va::run(va::Impl::Tc, q, q_stride_tok, q_stride_head, kv_pool, pool_size, qo_indptr,
                   kv_indptr, kv_indices, out_cache_loc, custom_mask, mask_indptr, sm_scale, out,
                   out_stride_tok, out_stride_head, batch, max_q_per_req, num_heads, num_splits,
                   workspace, workspace_bytes, stream);
}

int verify_attn_run_simt(const void *q, int64_t q_stride_tok, int64_t q_stride_head,
                         const void *kv_pool, int64_t pool_size, const int32_t *qo_indptr,
                         const int32_t *kv_indptr, const int32_t *kv_indices,
                         const int64_t *out_cache_loc, const uint8_t *custom_mask,
                         const int64_t *mask_indptr, float sm_scale, void *out,
                         int64_t out_stride_tok, int64_t out_stride_head, int batch,
                         int max_q_per_req, int num_heads, int num_splits, void *workspace,
                         size_t workspace_bytes, verify_attn_stream_t stream)
{
    return va::run(va::Impl::Simt, q, q_stride_tok, q_stride_head, kv_pool, pool_size, qo_indptr,
                   kv_indptr, kv_indices, out_cache_loc, custom_mask, mask_indptr, sm_scale, out,
                   out_stride_tok, out_stride_head, batch, max_q_per_req, num_heads, num_splits,
                   workspace, workspace_bytes, stream);
}

int verify_attn_run_profiled(int impl, void *const *events, const void *q, int64_t q_stride_tok,
                             int64_t q_stride_head, const void *kv_pool, int64_t pool_size,
                             const int32_t *qo_indptr, const int32_t *kv_indptr,
                             const int32_t *kv_indices, const int64_t *out_cache_loc,
                             const uint8_t *custom_mask, const int64_t *mask_indptr,
                             float sm_scale, void *out, int64_t out_stride_tok,
                             int64_t out_stride_head, int batch, int max_q_per_req, int num_heads,
                             int num_splits, void *workspace, size_t workspace_bytes,
                             verify_attn_stream_t stream)
{
    if (impl != VERIFY_ATTN_IMPL_TC && impl != VERIFY_ATTN_IMPL_SIMT) return VA_ERR_DIMS;
    return va::run(impl == VERIFY_ATTN_IMPL_TC ? va::Impl::Tc : va::Impl::Simt, q, q_stride_tok,
                   q_stride_head, kv_pool, pool_size, qo_indptr, kv_indptr, kv_indices,
                   out_cache_loc, custom_mask, mask_indptr, sm_scale, out, out_stride_tok,
                   out_stride_head, batch, max_q_per_req, num_heads, num_splits, workspace,
                   workspace_bytes, stream, reinterpret_cast<cudaEvent_t const *>(events));
}

int verify_attn_save_kv(const void *kv_new, int64_t kv_new_stride_tok, const int64_t *out_cache_loc,
                        int64_t num_tokens, void *kv_pool, int64_t pool_size, void *workspace,
                        size_t workspace_bytes, verify_attn_stream_t stream)
{
    if (num_tokens < 0 || pool_size <= 0) return VA_ERR_DIMS;
    if (!kv_pool || !workspace || (num_tokens > 0 && (!kv_new || !out_cache_loc))) return VA_ERR_NULL;
    if (!va::aligned(kv_pool, 16) || !va::aligned(workspace, 256) ||
        (num_tokens > 0 && (!va::aligned(kv_new, 16) || (kv_new_stride_tok & 7) || kv_new_stride_tok < va::D)))
        return VA_ERR_ALIGN;
    if (workspace_bytes < va::WS_HEADER) return VA_ERR_WORKSPACE;
    const int rc = va::ensure_init();
    if (rc != VA_OK) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    unsigned *status = static_cast<unsigned *>(workspace);
    if (cudaMemsetAsync(status, 0, sizeof(unsigned), s) != cudaSuccess) return VA_ERR_LAUNCH;
    if (va::launch_kv_save(static_cast<const __nv_bfloat16 *>(kv_new), kv_new_stride_tok, out_cache_loc, num_tokens,
                           nullptr, static_cast<__nv_bfloat16 *>(kv_pool), pool_size, status, s) != cudaSuccess)
        return VA_ERR_LAUNCH;
    return VA_OK;
}

int verify_attn_save_and_run(const void *kv_new, int64_t kv_new_stride_tok, const void *q, int64_t q_stride_tok,
                             int64_t q_stride_head, void *kv_pool, int64_t pool_size, const int32_t *qo_indptr,
                             const int32_t *kv_indptr, const int32_t *kv_indices, const int64_t *out_cache_loc,
                             const uint8_t *custom_mask, const int64_t *mask_indptr, float sm_scale, void *out,
                             int64_t out_stride_tok, int64_t out_stride_head, int batch, int max_q_per_req,
                             int num_heads, int num_splits, void *workspace, size_t workspace_bytes,
                             verify_attn_stream_t stream)
{
    const va::SaveArgs save{kv_new, kv_new_stride_tok};
    return va::run(va::Impl::Tc, q, q_stride_tok, q_stride_head, kv_pool, pool_size, qo_indptr, kv_indptr,
                   kv_indices, out_cache_loc, custom_mask, mask_indptr, sm_scale, out, out_stride_tok,
                   out_stride_head, batch, max_q_per_req, num_heads, num_splits, workspace, workspace_bytes,
                   stream, nullptr, &save);
}

int verify_attn_check_wait_timeout(uint64_t limit_ns, void *workspace, size_t workspace_bytes,
                                   verify_attn_stream_t stream)
{
    if (workspace == nullptr) return VA_ERR_NULL;
    if (!va::aligned(workspace, 256)) return VA_ERR_ALIGN;
    if (workspace_bytes < va::WS_HEADER) return VA_ERR_WORKSPACE;
    if (limit_ns < VERIFY_ATTN_WAIT_PROBE_MIN_NS || limit_ns > VERIFY_ATTN_WAIT_PROBE_MAX_NS) return VA_ERR_DIMS;
    const int rc = va::ensure_init();
    if (rc != VA_OK) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    unsigned *status = static_cast<unsigned *>(workspace);
    if (cudaMemsetAsync(status, 0, sizeof(unsigned), s) != cudaSuccess) return VA_ERR_LAUNCH;
    if (va::launch_wait_probe(status, limit_ns, s) != cudaSuccess) return VA_ERR_LAUNCH;
    return VA_OK;
}

const char *verify_attn_status_string(int status)
{
    switch (status) {
    case VA_OK: return "ok";
    case VA_ERR_NULL: return "a required pointer is null";
    case VA_ERR_ALIGN: return "misaligned pointer or stride";
    case VA_ERR_DIMS: return "batch/heads/max_q_per_req/pool_size out of range";
    case VA_ERR_WORKSPACE: return "workspace too small";
    case VA_ERR_SPLITS: return "num_splits out of range";
    case VA_ERR_LAUNCH: return "CUDA launch failed";
    case VA_ERR_SCALE: return "sm_scale is not finite";
    case VA_ERR_DEVICE: return "current device is not sm_103";
    case VA_ERR_SCRATCH_LIMIT: return "capacities need more scratch than the static 32 MiB array";
    default: return "unknown status";
    }
}

}  // extern "C"
