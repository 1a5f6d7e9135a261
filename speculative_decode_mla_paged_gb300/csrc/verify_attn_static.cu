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
// so host code asks the runtime for the real address (cudaGetSymbolAddress,
// with the device current) and passes that to the kernels.  Under lazy
// module loading the array's memory is committed when its module first
// loads, i.e. at the first address lookup; verify_attn_init() does that
// lookup (static_scratch_setup below), so a caller that runs
// verify_attn_init() before reserving the rest of the GPU's memory never
// meets an out-of-memory failure here later.  Each call looks the address
// up again (a host-side table lookup once the module is loaded), so there is
// no cached pointer to go stale.  The call then runs the production path
// (verify_attn_run) with that array as its workspace.  Nothing here calls
// cudaMalloc, cudaFree or any allocating library routine.
#include "verify_attn.h"

#include <cuda_runtime.h>

namespace {

// Scratch shared by every verify_attn_run_static call on a device.
static __device__ __align__(256) unsigned char g_static_scratch[VERIFY_ATTN_STATIC_SCRATCH_BYTES];

// Device address of the scratch array on the current device.
int scratch_address(void **addr)
{
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) {
        cudaGetLastError();   // leave no pending error behind for the caller
        return VA_ERR_LAUNCH;
    }
    *addr = p;
    return VA_OK;
}

}  // namespace

namespace va {

// Part of verify_attn_init(): load the array's module on the current device
// (which commits its memory) by looking its address up once.
int static_scratch_setup()
{
    void *p = nullptr;
    return scratch_address(&p);
}

}  // namespace va

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
    int rc = verify_attn_init();   // device check first: a non-sm_103 device gives VA_ERR_DEVICE
    if (rc != VA_OK) return rc;
    void *scratch = nullptr;
    rc = scratch_address(&scratch);
    if (rc != VA_OK) return rc;
    return verify_attn_run(q, q_stride_tok, q_stride_head, kv_pool, pool_size, qo_indptr, kv_indptr,
                           kv_indices, out_cache_loc, custom_mask, mask_indptr, sm_scale, out,
                           out_stride_tok, out_stride_head, batch, max_q_per_req, num_heads,
                           num_splits, scratch, VERIFY_ATTN_STATIC_SCRATCH_BYTES, stream);
}

extern "C" int verify_attn_static_status_word(unsigned int **status)
{
    if (status == nullptr) return VA_ERR_NULL;
    *status = nullptr;
    int rc = verify_attn_init();
    if (rc != VA_OK) return rc;
    void *scratch = nullptr;
    rc = scratch_address(&scratch);
    if (rc != VA_OK) return rc;
    *status = static_cast<unsigned int *>(scratch);   // the status word sits at byte 0
    return VA_OK;
}
