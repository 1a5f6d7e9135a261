// KV save: write the draft tokens' latent rows into the pool at their own
// slots, kv_pool[out_cache_loc[i], :] = kv_new[i, :].  This is the side
// effect of the serving step that must land before the verify attention
// reads those keys ("The Launch Wrapper", section The KV Cache Ordering
// Insight: only the KV save is kept from the original step, then the
// custom kernel runs on the populated pool).  Launched on the same stream
// right before the split kernel, it allocates nothing and is capture-safe.
#include "va_internal.cuh"

namespace va {
namespace {

constexpr int ROWS_PER_BLOCK = 8;          // one warp per token row
constexpr int PIECES = D * 2 / 16;         // 72 pieces of 16 B per 1152-B row

// Rows [0, n) with n = min(*count, cap) when `count` (a device int32, e.g.
// qo_indptr[batch]) is given, else n = cap: the grid is sized by the host
// capacity so a captured graph serves every batch within it.
__global__ void __launch_bounds__(ROWS_PER_BLOCK * 32) kv_save_kernel(const __nv_bfloat16 *kv_new, int64_t stride_tok,
                                                                       const int64_t *out_cache_loc, int64_t cap,
                                                                       const int32_t *count, __nv_bfloat16 *kv_pool,
                                                                       int64_t pool_size, unsigned *status)
{
    const int64_t i = (int64_t)blockIdx.x * ROWS_PER_BLOCK + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    const int64_t n = count != nullptr ? (__ldg(count) < cap ? (int64_t)__ldg(count) : cap) : cap;
    if (i >= n) return;
    const int64_t slot = __ldg(out_cache_loc + i);
    if (slot < 0 || slot >= pool_size) {       // skipped; the caller reads the status word
        if (lane == 0) atomicOr(status, STATUS_BAD_SLOT);
        return;
    }
    const uint4 *src = reinterpret_cast<const uint4 *>(kv_new + i * stride_tok);
    uint4 *dst = reinterpret_cast<uint4 *>(kv_pool + slot * (int64_t)D);
    for (int k = lane; k < PIECES; k += 32) dst[k] = __ldg(src + k);
}

}  // namespace

cudaError_t launch_kv_save(const __nv_bfloat16 *kv_new, int64_t stride_tok, const int64_t *out_cache_loc,
                           int64_t cap, const int32_t *count, __nv_bfloat16 *kv_pool, int64_t pool_size,
                           unsigned *status, cudaStream_t stream)
{
    if (cap <= 0) return cudaSuccess;
    const int64_t blocks = (cap + ROWS_PER_BLOCK - 1) / ROWS_PER_BLOCK;
    kv_save_kernel<<<(unsigned)blocks, ROWS_PER_BLOCK * 32, 0, stream>>>(kv_new, stride_tok, out_cache_loc, cap, count,
                                                                          kv_pool, pool_size, status);
    return cudaGetLastError();
}

}  // namespace va
