// Internal declarations shared by the libverify_attn translation units.
// Nothing here is part of the C ABI (include/verify_attn.h is).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace va {

constexpr int D = 576;            // latent row: 512 no-PE + 64 RoPE dims
constexpr int DV = 512;           // V = first 512 dims of the row
constexpr int KEY_ALIGN = 128;    // split chunks are multiples of this many keys
constexpr int MIN_CHUNK = 256;    // and at least this long (a split reloads its query tile)
constexpr size_t WS_HEADER = 256; // status word + padding at the workspace start

constexpr unsigned STATUS_BAD_SLOT = 0x1u;   // slot outside the pool / null index buffer
constexpr unsigned STATUS_BAD_META = 0x2u;   // T_b > max_q_per_req or negative lengths
constexpr unsigned STATUS_TIMEOUT = 0x4u;    // a bounded wait inside a kernel expired

// Everything one call needs, by value (kernel parameter).
struct Params {
    const __nv_bfloat16 *q;
    int64_t q_stride_tok, q_stride_head;
    const __nv_bfloat16 *kv_pool;
    int64_t pool_size;
    const int32_t *qo_indptr;
    const int32_t *kv_indptr;
    const int32_t *kv_indices;
    const int64_t *out_cache_loc;
    const uint8_t *custom_mask;
    const int64_t *mask_indptr;
    float sm_scale;
    __nv_bfloat16 *out;
    int64_t out_stride_tok, out_stride_head;
    int batch, max_q_per_req, num_heads, num_splits;
    int64_t rows_cap;      // batch * max_q_per_req * num_heads
    int64_t rows_lo, rows_hi;   // tensor-core split: only requests with rows_lo < T_b * H <= rows_hi
    unsigned *status;      // workspace byte 0
    float *part_o;         // [num_splits][rows_cap][512]
    float *part_lse;       // [num_splits][rows_cap]
};

// Keys per split for a request with n keys: the pages' ceil(n / NSPLIT)
// ("The Capture-Safe Kernel", Decision 3), at least MIN_CHUNK, rounded up
// to a whole key tile.  A request uses ceil(n / chunk) <= num_splits splits.
__host__ __device__ inline int64_t split_chunk(int64_t n, int num_splits)
{
    int64_t c = (n + num_splits - 1) / num_splits;
    if (c < MIN_CHUNK) c = MIN_CHUNK;
    return (c + KEY_ALIGN - 1) / KEY_ALIGN * KEY_ALIGN;
}

// Number of non-empty splits of a request with n keys.
__host__ __device__ inline int64_t splits_used(int64_t n, int num_splits)
{
    if (n <= 0) return 0;
    int64_t c = split_chunk(n, num_splits);
    return (n + c - 1) / c;
}

// Pool slot of key j of request b, or -1 (and a status bit) when it is invalid.
__device__ inline int64_t key_slot(const Params &p, int64_t kv0, int64_t qo0, int64_t L, int64_t j)
{
    int64_t slot;
    if (j < L) {
        if (p.kv_indices == nullptr) { atomicOr(p.status, STATUS_BAD_SLOT); return -1; }
        slot = p.kv_indices[kv0 + j];
    } else {
        if (p.out_cache_loc == nullptr) { atomicOr(p.status, STATUS_BAD_SLOT); return -1; }
        slot = p.out_cache_loc[qo0 + (j - L)];
    }
    if (slot < 0 || slot >= p.pool_size) { atomicOr(p.status, STATUS_BAD_SLOT); return -1; }
    return slot;
}

cudaError_t simt_init();
cudaError_t launch_simt_split(const Params &p, cudaStream_t stream);
cudaError_t launch_combine(const Params &p, cudaStream_t stream);
cudaError_t launch_kv_save(const __nv_bfloat16 *kv_new, int64_t stride_tok, const int64_t *out_cache_loc,
                           int64_t cap, const int32_t *count, __nv_bfloat16 *kv_pool, int64_t pool_size,
                           unsigned *status, cudaStream_t stream);

}  // namespace va
