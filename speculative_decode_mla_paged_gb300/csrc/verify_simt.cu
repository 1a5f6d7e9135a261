// Split-KV tree-verify attention on CUDA cores (fp32 FMA), the portable
// cross-check kernel.
//
// One CTA per (key split, 16-row tile, request).  Per 32-key tile it
// resolves slots (prefix keys through kv_indices, draft keys through
// out_cache_loc -- "The Capture-Safe Kernel", Decisions 1-2), gathers the
// scattered 1152-B rows into shared memory, decodes the packed tree-mask
// bits in place (Decision 5), and runs an online softmax over the 576-wide
// scores before accumulating V = the first 512 dims.  It writes a
// normalised partial output and its log-sum-exp per row (split-KV partial,
// "The Integration Chasm", section Context; Decision 3).
#include "va_internal.cuh"

#include <math.h>

namespace va {
namespace {

constexpr int SR = 16;            // rows per CTA
constexpr int SK = 32;            // keys per tile (one per lane)
constexpr int THREADS = 256;      // 8 warps: warp w owns rows 2w, 2w+1 in the score phase
constexpr int KT_STRIDE = SK + 2; // bf16 elements per transposed-key row (bank spread)

constexpr size_t SMEM_Q = sizeof(float) * SR * D;
constexpr size_t SMEM_KT = sizeof(__nv_bfloat16) * D * KT_STRIDE;
constexpr size_t SMEM_P = sizeof(float) * SR * SK;
constexpr size_t SMEM_SLOT = sizeof(int64_t) * SK;
constexpr size_t SMEM_ROW = sizeof(float) * SR * 3;
constexpr size_t SMEM_TOTAL = SMEM_Q + SMEM_KT + SMEM_P + SMEM_SLOT + SMEM_ROW;

__device__ inline float warp_max(float v)
{
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ inline float warp_sum(float v)
{
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__global__ void __launch_bounds__(THREADS) simt_split_kernel(Params p)
{
    extern __shared__ __align__(16) unsigned char smem[];
    float *Qs = reinterpret_cast<float *>(smem);
    __nv_bfloat16 *Kt = reinterpret_cast<__nv_bfloat16 *>(smem + SMEM_Q);
    float *Ps = reinterpret_cast<float *>(smem + SMEM_Q + SMEM_KT);
    int64_t *slot_s = reinterpret_cast<int64_t *>(smem + SMEM_Q + SMEM_KT + SMEM_P);
    float *alpha_s = reinterpret_cast<float *>(smem + SMEM_Q + SMEM_KT + SMEM_P + SMEM_SLOT);
    float *m_s = alpha_s + SR;
    float *l_s = m_s + SR;

    const int split = blockIdx.x, rt = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = p.num_heads;

    const int64_t qo0 = p.qo_indptr[b], T = p.qo_indptr[b + 1] - qo0;
    const int64_t kv0 = p.kv_indptr[b], L = p.kv_indptr[b + 1] - kv0;
    if (T < 0 || L < 0 || T > p.max_q_per_req) {
        if (split == 0 && rt == 0 && tid == 0) atomicOr(p.status, STATUS_BAD_META);
        if (T < 0 || L < 0) return;
    }
    const int64_t rows_b = (T < p.max_q_per_req ? T : p.max_q_per_req) * H;
    const int64_t r0 = (int64_t)rt * SR;
    if (r0 >= rows_b) return;
    const int64_t N = L + T;
    const int64_t chunk = split_chunk(N, p.num_splits);
    const int64_t k0 = (int64_t)split * chunk;
    if (k0 >= N) return;                       // empty split: the combine skips it
    const int64_t k1 = (k0 + chunk < N) ? k0 + chunk : N;
    const int64_t mask0 = p.mask_indptr[b];

    // Q tile -> fp32 shared memory (rows past the request are zero).
    for (int e = tid; e < SR * (D / 8); e += THREADS) {
        int rr = e / (D / 8), c = e % (D / 8);
        int64_t lr = r0 + rr;
        float v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        if (lr < rows_b) {
            int64_t t = qo0 + lr / H, h = lr % H;
            uint4 raw = *reinterpret_cast<const uint4 *>(p.q + t * p.q_stride_tok + h * p.q_stride_head + c * 8);
            const __nv_bfloat16 *x = reinterpret_cast<const __nv_bfloat16 *>(&raw);
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = __bfloat162float(x[u]);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) Qs[rr * D + c * 8 + u] = v[u];
    }

    // Per-row running max / sum, held by the owning warp (all lanes agree).
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    float acc[SR][2];
#pragma unroll
    for (int rr = 0; rr < SR; ++rr) acc[rr][0] = acc[rr][1] = 0.f;

    for (int64_t kb = k0; kb < k1; kb += SK) {
        if (warp == 0) {
            int64_t j = kb + lane;
            slot_s[lane] = (j < k1) ? key_slot(p, kv0, qo0, L, j) : -1;
        }
        __syncthreads();
        // Gather the tile's rows, transposed: Kt[d][key].
        for (int e = tid; e < SK * (D / 8); e += THREADS) {
            int key = e % SK, c = e / SK;
            int64_t slot = slot_s[key];
            uint4 raw = make_uint4(0, 0, 0, 0);
            if (slot >= 0) raw = __ldg(reinterpret_cast<const uint4 *>(p.kv_pool + slot * D + c * 8));
            const __nv_bfloat16 *x = reinterpret_cast<const __nv_bfloat16 *>(&raw);
#pragma unroll
            for (int u = 0; u < 8; ++u) Kt[(c * 8 + u) * KT_STRIDE + key] = x[u];
        }
        __syncthreads();

        // Scores for rows 2w, 2w+1 against key `lane`; mask; online softmax.
        const int64_t j = kb + lane;
        const bool key_ok = (j < k1) && (slot_s[lane] >= 0);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int rr = warp * 2 + u;
            const int64_t lr = r0 + rr;
            float s = -INFINITY;
            if (key_ok && lr < rows_b) {
                const int64_t i = lr / H;
                const int64_t bit = mask0 + i * N + j;
                if ((p.custom_mask[bit >> 3] >> (bit & 7)) & 1) {
                    const float *qr = Qs + rr * D;
                    float dot = 0.f;
#pragma unroll 8
                    for (int d = 0; d < D; ++d) dot = fmaf(qr[d], __bfloat162float(Kt[d * KT_STRIDE + lane]), dot);
                    s = dot * p.sm_scale;
                }
            }
            const float m_tile = warp_max(s);
            const float m_new = fmaxf(m_run[u], m_tile);
            float pr = 0.f, alpha = 1.f;
            if (m_new != -INFINITY) {
                pr = (s == -INFINITY) ? 0.f : expf(s - m_new);
                alpha = (m_run[u] == -INFINITY) ? 0.f : expf(m_run[u] - m_new);
            }
            l_run[u] = l_run[u] * alpha + warp_sum(pr);
            m_run[u] = m_new;
            Ps[rr * SK + lane] = pr;
            if (lane == 0) alpha_s[rr] = alpha;
        }
        __syncthreads();

        // O[rr][tid], O[rr][tid+256] += sum_k P[rr][k] * V[k][.]
#pragma unroll
        for (int rr = 0; rr < SR; ++rr) {
            const float a = alpha_s[rr];
            acc[rr][0] *= a;
            acc[rr][1] *= a;
        }
        for (int k = 0; k < SK; ++k) {
            const float v0 = __bfloat162float(Kt[tid * KT_STRIDE + k]);
            const float v1 = __bfloat162float(Kt[(tid + 256) * KT_STRIDE + k]);
#pragma unroll
            for (int rr = 0; rr < SR; ++rr) {
                const float pr = Ps[rr * SK + k];
                acc[rr][0] = fmaf(pr, v0, acc[rr][0]);
                acc[rr][1] = fmaf(pr, v1, acc[rr][1]);
            }
        }
        __syncthreads();
    }

    if (lane == 0) {
        m_s[warp * 2] = m_run[0]; m_s[warp * 2 + 1] = m_run[1];
        l_s[warp * 2] = l_run[0]; l_s[warp * 2 + 1] = l_run[1];
    }
    __syncthreads();
    for (int rr = 0; rr < SR; ++rr) {
        const int64_t lr = r0 + rr;
        if (lr >= rows_b) break;
        const int64_t row = qo0 * H + lr;
        if (row >= p.rows_cap) break;          // only when T_b > max_q_per_req (flagged)
        const float l = l_s[rr];
        const float inv = l > 0.f ? 1.f / l : 0.f;
        float *o = p.part_o + ((int64_t)split * p.rows_cap + row) * DV;
        o[tid] = acc[rr][0] * inv;
        o[tid + 256] = acc[rr][1] * inv;
        if (tid == 0) p.part_lse[(int64_t)split * p.rows_cap + row] = l > 0.f ? m_s[rr] + logf(l) : -INFINITY;
    }
}

}  // namespace

cudaError_t simt_init()
{
    return cudaFuncSetAttribute(simt_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)SMEM_TOTAL);
}

cudaError_t launch_simt_split(const Params &p, cudaStream_t stream)
{
    const int row_tiles = (p.max_q_per_req * p.num_heads + SR - 1) / SR;
    dim3 grid(p.num_splits, row_tiles, p.batch);
    simt_split_kernel<<<grid, THREADS, SMEM_TOTAL, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace va
