// verify_attn_run_static: the same tree-verify attention call for callers
// that cannot allocate device memory.
//
// Who needs it: a serving engine that reserves nearly all of the GPU's
// memory for its KV pool at start-up and forbids later allocations, a host
// application that loads this library as a plug-in without handing it an
// allocator, or code on a path where an allocation would synchronise the
// device.  Such callers cannot provide the workspace verify_attn_run asks
// for, so this entry point brings its own: a fixed scratch array compiled
// into the library.
//
// How: g_static_scratch below is a file-scope __device__ array.  Every GPU
// that loads the library holds one copy of it until the process exits.  In
// host code its name is only a host-side stand-in, never a device address,
// so the first call on each device asks the runtime for the real address
// (cudaGetSymbolAddress, with that device current) and caches it; later
// calls reuse the cached address.  The call then runs the production path
// (verify_attn_run) with that array as its workspace.  Nothing here calls
// cudaMalloc, cudaFree or any allocating library routine.
#include "verify_attn.h"

#include <cuda_runtime.h>
#include <mutex>

namespace {

// Scratch shared by every verify_attn_run_static call on a device.
static __device__ __align__(256) unsigned char g_static_scratch[VERIFY_ATTN_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_scratch_addr[kMaxDevices] = {};   // device address of g_static_scratch, per device

// Device address of the scratch array on the current device (set up once).
int scratch_address(void **addr)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return VA_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();   // leave no pending error behind for the caller
            return VA_ERR_LAUNCH;
        }
        g_scratch_addr[dev] = p;
    }
    *addr = g_scratch_addr[dev];
    return VA_OK;
}

}  // namespace

extern "C" int verify_attn_run_static(const void *q, int64_t q_stride_tok, int64_t q_stride_head,
                                      const void *kv_pool, int64_t pool_size,
                                      const int32_t *qo_indptr, const int32_t *kv_indptr,
                                      const int32_t *kv_indices, const int64_t *out_cache_loc,
                                      const uint8_t *custom_mask, const int64_t *mask_indptr,
                                      float sm_scale, void *out, int64_t out_stride_tok,
                                      int64_t out_stride_head, int batch, int max_q_per_req,
                                      int num_heads, int num_splits, verify_attn_stream_t stream)
{
    if (num_splits < 1 || num_splits > VERIFY_ATTN_MAX_SPLITS) return VA_ERR_SPLITS;
    const size_t need = verify_attn_workspace_size(batch, max_q_per_req, num_heads, num_splits);
    if (need == 0) return VA_ERR_DIMS;
    if (need > VERIFY_ATTN_STATIC_SCRATCH_BYTES) return VA_ERR_SCRATCH_LIMIT;
    void *scratch = nullptr;
    const int rc = scratch_address(&scratch);
    if (rc != VA_OK) return rc;
    return verify_attn_run(q, q_stride_tok, q_stride_head, kv_pool, pool_size, qo_indptr, kv_indptr,
                           kv_indices, out_cache_loc, custom_mask, mask_indptr, sm_scale, out,
                           out_stride_tok, out_stride_head, batch, max_q_per_req, num_heads,
                           num_splits, scratch, VERIFY_ATTN_STATIC_SCRATCH_BYTES, stream);
}
