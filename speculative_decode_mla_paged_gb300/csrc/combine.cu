// Split combine: merge the per-split partial outputs of each row by their
// log-sum-exp ("The Integration Chasm", section Context: partial-plus-reduce;
// "The Capture-Safe Kernel", Input Knowledge item 3: a reduction step
// combines the splits).
//
//   m* = max_s lse_s,  w_s = exp(lse_s - m*),  out = sum_s w_s O_s / sum_s w_s
//
// One warp per output row; each lane owns 16 of the 512 columns (four
// float4 loads per split, fully coalesced).  The lanes first read the
// splits' lse values side by side (lane k: splits k, k + 32, ...) and agree
// on the maximum and the weights with warp shuffles, so the loop over the
// splits issues its partial loads without waiting on a weight and several
// splits' loads are in flight at once; the sum still runs in split order.
// Splits past the end of the request are never read: their count follows
// from the indptrs with the same chunk rule the split kernels use.  Output
// is bf16, round to nearest even; a row whose splits all have lse = -inf (no
// visible key) gets zeros.
#include "va_internal.cuh"

#include <math.h>

namespace va {
namespace {

constexpr int WARPS = 8;

__global__ void __launch_bounds__(WARPS * 32) combine_kernel(Params p)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * WARPS + warp;      // t*H + h
    const int H = p.num_heads;
    const int64_t total_q = p.qo_indptr[p.batch];
    if (row >= total_q * H || row >= p.rows_cap) return;
    const int64_t t = row / H;
    const int h = (int)(row % H);

    int lo = 0, hi = p.batch;                 // last b with qo_indptr[b] <= t
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (p.qo_indptr[mid] <= t) lo = mid; else hi = mid;
    }
    const int b = lo;
    const int64_t T = p.qo_indptr[b + 1] - p.qo_indptr[b];
    const int64_t L = p.kv_indptr[b + 1] - p.kv_indptr[b];
    const bool processed = (t - p.qo_indptr[b]) < p.max_q_per_req && L >= 0;
    const int64_t ns = processed ? splits_used(L + T, p.num_splits) : 0;

    float m = -INFINITY;
    for (int64_t s = lane; s < ns; s += 32) m = fmaxf(m, p.part_lse[s * p.rows_cap + row]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));

    float4 acc[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f;
    if (m != -INFINITY) {
        for (int64_t s0 = 0; s0 < ns; s0 += 32) {
            // this lane's weight: split s0 + lane (0 past the end or with lse = -inf)
            float wl = 0.f;
            if (s0 + lane < ns) {
                const float lse = p.part_lse[(s0 + lane) * p.rows_cap + row];
                wl = lse == -INFINITY ? 0.f : expf(lse - m);
            }
            wsum += wl;
            const int n = ns - s0 < 32 ? (int)(ns - s0) : 32;
#pragma unroll 4
            for (int k = 0; k < n; ++k) {
                const float w = __shfl_sync(0xffffffffu, wl, k);
                const float4 *o = reinterpret_cast<const float4 *>(p.part_o + ((s0 + k) * p.rows_cap + row) * DV);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float4 v = o[j * 32 + lane];
                    if (w != 0.f) {   // a split without visible keys adds nothing
                        acc[j].x = fmaf(w, v.x, acc[j].x);
                        acc[j].y = fmaf(w, v.y, acc[j].y);
                        acc[j].z = fmaf(w, v.z, acc[j].z);
                        acc[j].w = fmaf(w, v.w, acc[j].w);
                    }
                }
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, off);
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    __nv_bfloat16 *dst = p.out + t * p.out_stride_tok + (int64_t)h * p.out_stride_head;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        __nv_bfloat162 lo2 = __floats2bfloat162_rn(acc[j].x * inv, acc[j].y * inv);
        __nv_bfloat162 hi2 = __floats2bfloat162_rn(acc[j].z * inv, acc[j].w * inv);
        uint2 packed;
        packed.x = *reinterpret_cast<unsigned *>(&lo2);
        packed.y = *reinterpret_cast<unsigned *>(&hi2);
        *reinterpret_cast<uint2 *>(dst + (j * 32 + lane) * 4) = packed;
    }
}

}  // namespace

cudaError_t launch_combine(const Params &p, cudaStream_t stream)
{
    const int64_t blocks = (p.rows_cap + WARPS - 1) / WARPS;
    if (blocks == 0) return cudaSuccess;
    combine_kernel<<<(unsigned)blocks, WARPS * 32, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace va
