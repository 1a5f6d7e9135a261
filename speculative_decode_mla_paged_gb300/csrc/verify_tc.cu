// Tensor-core split kernel for tree-verify attention (sm_103a: tcgen05, TMEM).
//
// Work unit: one (key split, 128-row tile, request), the same unit as the
// pages' split-KV flash-decode partial ("The Capture-Safe Kernel",
// Decision 3), but every key tile is loaded once per 128 rows (T*H rows of
// one request share all keys: MLA latent attention, "The Integration
// Chasm", section Decision) and both contractions run on the tensor cores.
//
// Why a 2-CTA cluster per unit.  A 128 x 512 fp32 output accumulator is the
// whole of an SM's TMEM (128 lanes x 512 columns), and a 128 x 576 bf16 Q
// tile is 144 KB of shared memory, so one SM cannot hold Q, the scores S
// and O for 128 rows while feeding M = 128 MMAs at full rate.  The pair
// splits the work by role:
//
//   CTA rank 0 ("S"): Q lives in TMEM (288 columns of packed bf16, the A
//     operand of S = Q K^T from tensor memory); K tiles (64 keys x 576) are
//     gathered into shared memory; two 64-column S buffers in TMEM.  Its
//     four row warps (thread = row) read S, apply the packed tree mask, run
//     the online softmax and write P (bf16) straight into the partner's
//     shared memory.
//   CTA rank 1 ("O"): the 128 x 512 fp32 O accumulator fills its TMEM;
//     V tiles (64 keys x 512, the first 512 dims of the same rows) are
//     gathered into shared memory; O += P V on the tensor cores.
//
// Per 64-key tile the S CTA issues 36 MMAs (M128 N64 K16, A from TMEM) and
// the O CTA 8 (M128 N256 K16, both operands in shared memory), so the two
// SMs carry 576 and 512 MACs per (row, key): balanced.
//
// Online softmax uses a lazy maximum: O is rescaled only when a row's
// running maximum grows by more than 2^8 (log2 units), so P stays <= 256;
// the S CTA sends the per-row factor and a per-warp flag with each P tile
// and the O CTA's row warps rescale their TMEM rows only on flagged tiles.
//
// Each thread role, the barriers between them, and the shared-memory
// layouts (128-byte swizzle; one gathered tile serves as K-major B of
// Q K^T and as MN-major B of P V) are described where they are defined.
// Every wait is bounded (1 s of global time): on expiry the kernel sets
// STATUS_TIMEOUT, unwinds, drains its MMAs and frees TMEM.
#include "va_internal.cuh"
#include "tc_ptx.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <mutex>

namespace va {
namespace {

using namespace ptx;

constexpr int ROWS = 128;                  // rows per unit = M of every MMA
constexpr int KEYS = 64;                   // keys per O-role tile (one P half)
constexpr int KEYS_S = 128;                // keys per S-role tile (N of the score MMAs)
constexpr int STAGES = 3;                  // O role: gathered V tiles in flight
constexpr int NSLOT = 4;                   // S role: ring of 48 KB slots, 3 K chunks (128 keys x 64 dims) each
constexpr int SLOT_CHUNKS = 3;
constexpr int THREADS = 576;               // warps 0-7 rows, 8-15 gather (TMA), 16 MMA issue, 17 P sender
constexpr int SOFTMAX_THREADS = 256;       // S role: two warp groups, each owns half the keys of a tile
constexpr int PRODUCER_WARP0 = 8;          // TMA issue is serial within a warp, so 8 warps share it
constexpr int PRODUCER_WARPS = 8;
constexpr int MMA_WARP = 16;
constexpr int SENDER_WARP = 17;
constexpr uint32_t CHUNK_BYTES = KEYS * 128;          // one 64-dim column block of a tile
constexpr uint32_t K_CHUNKS = D / 64;                 // 9
constexpr uint32_t V_CHUNKS = DV / 64;                // 8
constexpr uint32_t KCHUNK_BYTES = KEYS_S * 128;       // 16384: one K chunk of an S tile
constexpr uint32_t SLOT_BYTES = SLOT_CHUNKS * KCHUNK_BYTES;
constexpr uint32_t V_STAGE = V_CHUNKS * CHUNK_BYTES;  // 65536
constexpr uint32_t P_BUF = ROWS * KEYS * 2;           // 16384
constexpr uint32_t HEADER = 2048;
constexpr uint32_t STAGE0 = HEADER;                   // both roles: gathered tiles
constexpr uint32_t PBUF0 = HEADER + STAGES * V_STAGE; // O role: two P buffers
constexpr uint32_t SMEM_USED = PBUF0 + 2 * P_BUF;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;     // room to align the base to 1 KB
constexpr uint32_t QPE0 = HEADER;                     // S role: Q's 64 RoPE dims, 128 x 128 B (A of 4 MMAs)
constexpr uint32_t RING0 = QPE0 + ROWS * 128;         // S role: K chunk ring
constexpr uint32_t S_SCRATCH = RING0 + NSLOT * SLOT_BYTES; // S role: per-row partial sums of the 2nd group
static_assert(S_SCRATCH + ROWS * 4 <= SMEM_USED, "S role layout");
static_assert(SMEM_ALLOC <= 232448, "at most 227 KB of shared memory per CTA");

constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_Q = 0;                          // S role: Q's 512 no-PE dims, 256 columns
constexpr uint32_t TM_S0 = 256;                       // S role: S buffers at 256 and 384 (128 columns each)
constexpr uint32_t IDESC_S = idesc_bf16(128, 128, false);
constexpr uint32_t IDESC_PV = idesc_bf16(128, 256, true);
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.69314718055994531f;
constexpr float RESCALE_LOG2 = 8.0f;
constexpr uint64_t TIMEOUT_NS = 1000000000ull;

// Shared-memory header at the (1 KB aligned) base; same offsets in both CTAs
// so a barrier or field can be addressed in the partner with mapa.
struct Header {
    uint64_t c_full[NSLOT];    // S: 3 K chunks landed in a ring slot (8 producer-warp arrives + TMA bytes)
    uint64_t c_empty[NSLOT];   // S: MMAs reading the slot completed (commit)
    uint64_t s_full[2];        // S: scores ready (commit) + valid-key bits published (MMA thread)
    uint64_t s_free[2];        // S: the 8 softmax warps have read the score buffer
    uint64_t p_written[2];     // S: softmax group g (4 warps) stored its P half into the partner's buffer g
    uint64_t p_empty[2];       // S: partner done with a P buffer (its commit + its 4 row-warp leaders)
    uint64_t v_full[STAGES];   // O: gathered V tile landed (8 producer-warp arrives + TMA bytes)
    uint64_t v_empty[STAGES];  // O: MMAs reading the stage completed
    uint64_t p_full[2];        // O: partner's sender warp published a P tile
    uint64_t pv_sync;          // O: every MMA issued so far completed (before a rescale)
    uint64_t rs_req;           // O: MMA thread asks the row warps to rescale O
    uint64_t rs_done;          // O: 128 row threads rescaled their rows
    uint64_t l_ready;          // O: partner's 4 row warps wrote 1/l
    uint64_t drain;            // both: all MMAs of the CTA completed
    uint64_t t_valid[2][2];    // S: bit n of an S tile's 128 keys = key n has a valid slot (tile ring of 2)
    uint64_t s_valid[2][2];    // S: the same bits, per score buffer
    uint32_t tmem_base;
    uint32_t abort;
    uint32_t flags[2];         // O: byte w != 0 if a row of warp w rescales on this P buffer
    float alpha[2][ROWS];      // O: per-row rescale factor for the tile in each P buffer
    float inv_l[ROWS];         // O: 1 / softmax denominator per row (0 if the row saw nothing)
};
static_assert(sizeof(Header) <= HEADER, "header fits");

struct Unit {
    int split, b;
    int64_t qo0, kv0, L, N, k0, k1, r0, rows_b;
    int ntiles_s;              // S tiles of 128 keys
    int ntiles;                // O tiles of 64 keys = 2 * ntiles_s (the last may be empty)
    int rot;                   // this pair starts at S tile `rot` of its split (see tile_key0)
};

// First key of the t-th S tile this pair processes.  The row tiles of one
// request read the same keys; each starts at a different tile of the split
// (rot = row tile * ntiles_s / row tiles) so they do not request the same
// rows from L2 at the same moment.  Softmax order does not change the result.
__device__ __forceinline__ int64_t tile_key0(const Unit &u, int t)
{
    int s = t + u.rot;
    if (s >= u.ntiles_s) s -= u.ntiles_s;
    return u.k0 + (int64_t)s * KEYS_S;
}

// First key of the u-th O tile (64 keys: the two halves of each S tile).
__device__ __forceinline__ int64_t otile_key0(const Unit &u, int t)
{
    return tile_key0(u, t >> 1) + (int64_t)(t & 1) * KEYS;
}

// Bounded wait on phase `parity` of a barrier.  False after a timeout (status
// bit set, abort flag raised) or when another thread of the CTA aborted.
__device__ __noinline__ bool wait_bar(Header *h, uint32_t bar, uint32_t parity, unsigned *status, bool cluster,
                                      bool stop_on_abort = true)
{
    if (cluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (cluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (stop_on_abort && *reinterpret_cast<volatile uint32_t *>(&h->abort)) return false;
            if (globaltimer_ns() - t0 > TIMEOUT_NS) {
                atomicOr(status, STATUS_TIMEOUT);
                *reinterpret_cast<volatile uint32_t *>(&h->abort) = 1u;
                return false;
            }
        }
    }
}

// The same for all 32 lanes of a warp: true only if every lane's wait succeeded
// (keeps the warp converged for the .sync.aligned tcgen05 instructions).
__device__ __forceinline__ bool warp_wait(Header *h, uint32_t bar, uint32_t parity, unsigned *status, bool cluster)
{
    return __all_sync(0xffffffffu, wait_bar(h, bar, parity, status, cluster)) != 0;
}

// nbits (<= 64) mask bits starting at bit index bit0, bit n of the result =
// bit bit0 + n; bytes are read only inside that range.
__device__ __forceinline__ uint64_t load_bits(const uint8_t *mask, int64_t bit0, int nbits)
{
    if (nbits <= 0) return 0ull;
    const int64_t first = bit0 >> 3, last = (bit0 + nbits - 1) >> 3;
    const int nb = (int)(last - first + 1);
    uint64_t lo = 0, hi = 0;
#pragma unroll
    for (int k = 0; k < 9; ++k) {
        if (k < nb) {
            const uint64_t v = __ldg(mask + first + k);
            if (k < 8) lo |= v << (8 * k); else hi = v;
        }
    }
    const int sh = (int)(bit0 & 7);
    uint64_t w = sh ? ((lo >> sh) | (hi << (64 - sh))) : lo;
    if (nbits < 64) w &= (1ull << nbits) - 1ull;
    return w;
}

// ------------------------------------------------------------------ gather (warps 8-15, both roles)
//
// Tile layout in shared memory: NCH column blocks of 64 dims; block c holds
// the 64 keys as 128-B rows (key n at n*128), 16-B pieces swizzled as
// piece q -> q ^ (n & 7) inside each 1 KB group of 8 keys (the tensor map's
// 128-byte swizzle).  Read as B of Q K^T it is K-major (rows = keys); read as
// B of P V it is MN-major (64 contiguous dims per key row, 8 keys per 1 KB
// group).  Producer warp w (0..7) owns keys 8w..8w+7: lanes 0 and 1 each
// gather four keys with one TMA gather4 per column block (a warp issues its
// TMA instructions one after another, so the tile is spread over 8 warps).
// A key without a valid slot reads row pool_size, outside the map, which
// TMA fills with zeros.  Slots are loaded two tiles ahead, without branches
// on the loaded values, so the index loads overlap the stage waits.
template <int NCH>
__device__ void gather_tiles(const Params &p, Header *h, const CUtensorMap *tmap, uint32_t stage_base,
                             uint32_t stage_bytes, uint64_t *full, uint64_t *empty, uint64_t *valid, const Unit &u)
{
    const int pw = (int)(threadIdx.x >> 5) - PRODUCER_WARP0;
    const int lane = threadIdx.x & 31;
    const int64_t oob = p.pool_size;
    struct Rows { int64_t s[4]; };
    // Raw slots of this lane's 4 keys of tile t (-1 past the split or for idle lanes).
    auto load_rows = [&](int t) -> Rows {
        Rows r;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int64_t j = (t < u.ntiles ? otile_key0(u, t) : 0) + pw * 8 + lane * 4 + k;
            const bool live = lane < 2 && t < u.ntiles && j < u.k1;
            int64_t s = -1;
            if (live) {
                if (j < u.L) s = p.kv_indices ? (int64_t)__ldg(p.kv_indices + u.kv0 + j) : -2;
                else s = p.out_cache_loc ? __ldg(p.out_cache_loc + u.qo0 + (j - u.L)) : -2;
                if (s < 0 || s >= oob) s = -2;          // invalid slot: flagged, read as zeros
            }
            r.s[k] = s;
        }
        return r;
    };
    Rows ahead1 = load_rows(0), ahead2 = load_rows(1);
    for (int t = 0; t < u.ntiles; ++t) {
        const int stage = t % STAGES;
        const Rows cur = ahead1;
        ahead1 = ahead2;
        ahead2 = load_rows(t + 2);
        if (t >= STAGES &&
            !__all_sync(0xffffffffu, wait_bar(h, smem_u32(&empty[stage]), (uint32_t)((t / STAGES) - 1) & 1u, p.status, false)))
            break;
        uint32_t nib = 0, bad = 0;
        int y[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            nib |= (cur.s[k] >= 0 ? 1u : 0u) << k;
            bad |= cur.s[k] == -2 ? 1u : 0u;
            y[k] = cur.s[k] >= 0 ? (int)cur.s[k] : (int)oob;
        }
        if (bad) atomicOr(p.status, STATUS_BAD_SLOT);
        const uint32_t nib1 = __shfl_sync(0xffffffffu, nib, 1);
        const uint32_t bar = smem_u32(&full[stage]);
        if (lane == 0) {
            if (valid != nullptr)
                reinterpret_cast<volatile uint8_t *>(&valid[stage])[pw] = (uint8_t)(nib | (nib1 << 4));
            if (pw == 0) mbar_arrive_expect_tx(bar, NCH * CHUNK_BYTES);
            else mbar_arrive(bar);
        }
        if (lane < 2) {
            const uint32_t dst = stage_base + (uint32_t)stage * stage_bytes + (uint32_t)(pw * 2 + lane) * 512u;
#pragma unroll
            for (int c = 0; c < NCH; ++c) tma_gather4(dst + c * CHUNK_BYTES, tmap, c * 64, y[0], y[1], y[2], y[3], bar);
        }
    }
}

// ------------------------------------------------------------------ S role
//
// An S tile is 128 keys.  Its K rows reach shared memory as nine 16 KB
// chunks (128 keys x 64 dims, same 128-byte swizzled key-row layout as the
// V tiles), three chunks per slot of a 4-slot ring with one barrier pair per
// slot, so the score MMAs (N = 128, the shape that runs at full tensor rate)
// can start on a tile's first chunks while its later chunks are in flight.

// Gather (warps 8-15): producer warp w owns keys 16w..16w+15 of each S tile;
// lanes 0-3 each gather four keys, one TMA gather4 per chunk.
__device__ void s_role_gather(const Params &p, Header *h, const CUtensorMap *tmap, uint32_t smem, const Unit &u)
{
    const int pw = (int)(threadIdx.x >> 5) - PRODUCER_WARP0;
    const int lane = threadIdx.x & 31;
    const int64_t oob = p.pool_size;
    struct Rows { int64_t s[4]; };
    auto load_rows = [&](int t) -> Rows {
        Rows r;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int64_t j = (t < u.ntiles_s ? tile_key0(u, t) : 0) + pw * 16 + lane * 4 + k;
            const bool live = lane < 4 && t < u.ntiles_s && j < u.k1;
            int64_t s = -1;
            if (live) {
                if (j < u.L) s = p.kv_indices ? (int64_t)__ldg(p.kv_indices + u.kv0 + j) : -2;
                else s = p.out_cache_loc ? __ldg(p.out_cache_loc + u.qo0 + (j - u.L)) : -2;
                if (s < 0 || s >= oob) s = -2;          // invalid slot: flagged, read as zeros
            }
            r.s[k] = s;
        }
        return r;
    };
    Rows ahead1 = load_rows(0), ahead2 = load_rows(1);
    for (int t = 0; t < u.ntiles_s; ++t) {
        const Rows cur = ahead1;
        ahead1 = ahead2;
        ahead2 = load_rows(t + 2);
        uint32_t nib = 0, bad = 0;
        int y[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            nib |= (cur.s[k] >= 0 ? 1u : 0u) << k;
            bad |= cur.s[k] == -2 ? 1u : 0u;
            y[k] = cur.s[k] >= 0 ? (int)cur.s[k] : (int)oob;
        }
        if (bad) atomicOr(p.status, STATUS_BAD_SLOT);
        uint32_t bits16 = 0;
#pragma unroll
        for (int l = 0; l < 4; ++l) bits16 |= __shfl_sync(0xffffffffu, nib, l) << (4 * l);
        bool ok = true;
        for (int gi = 0; gi < (int)K_CHUNKS / SLOT_CHUNKS; ++gi) {
            const int q = t * ((int)K_CHUNKS / SLOT_CHUNKS) + gi, slot = q % NSLOT, use = q / NSLOT;
            if (use > 0 &&
                !__all_sync(0xffffffffu, wait_bar(h, smem_u32(&h->c_empty[slot]), (uint32_t)(use - 1) & 1u, p.status, false))) {
                ok = false;
                break;
            }
            const uint32_t bar = smem_u32(&h->c_full[slot]);
            if (lane == 0) {
                if (gi == 0) reinterpret_cast<volatile uint16_t *>(&h->t_valid[t & 1][0])[pw] = (uint16_t)bits16;
                if (pw == 0) mbar_arrive_expect_tx(bar, SLOT_BYTES);
                else mbar_arrive(bar);
            }
            if (lane < 4) {
                const uint32_t dst = smem + RING0 + (uint32_t)slot * SLOT_BYTES + (uint32_t)(pw * 4 + lane) * 512u;
#pragma unroll
                for (int cc = 0; cc < SLOT_CHUNKS; ++cc)
                    tma_gather4(dst + (uint32_t)cc * KCHUNK_BYTES, tmap, (gi * SLOT_CHUNKS + cc) * 64, y[0], y[1], y[2],
                                y[3], bar);
            }
        }
        if (!ok) break;
    }
}

// MMA issue (warp 16, lane 0): S[buf] = Q K^T per S tile, chunk by chunk:
// 32 MMAs with Q's no-PE dims from TMEM, then 4 with Q's RoPE dims from
// shared memory; each chunk's slot is released by a commit.
__device__ void s_role_mma(const Params &p, Header *h, uint32_t smem, uint32_t tmem, const Unit &u)
{
    for (int t = 0; t < u.ntiles_s; ++t) {
        const int buf = t & 1;
        if (t >= 2 && !wait_bar(h, smem_u32(&h->s_free[buf]), (uint32_t)((t >> 1) - 1) & 1u, p.status, false)) break;
        const uint32_t d = tmem + TM_S0 + 128u * (uint32_t)buf;
        bool ok = true;
        for (int c = 0; c < (int)K_CHUNKS; ++c) {
            const int q = t * ((int)K_CHUNKS / SLOT_CHUNKS) + c / SLOT_CHUNKS, slot = q % NSLOT, use = q / NSLOT;
            if (c % SLOT_CHUNKS == 0) {
                if (!wait_bar(h, smem_u32(&h->c_full[slot]), (uint32_t)use & 1u, p.status, false)) { ok = false; break; }
                tc_fence_after_sync();   // K arrives by TMA (async proxy): no proxy fence needed before the MMAs
            }
            if (c == 0) {
                volatile uint64_t *src = &h->t_valid[t & 1][0];
                volatile uint64_t *dst = &h->s_valid[buf][0];
                dst[0] = src[0];
                dst[1] = src[1];
            }
            const uint32_t sb = smem + RING0 + (uint32_t)slot * SLOT_BYTES + (uint32_t)(c % SLOT_CHUNKS) * KCHUNK_BYTES;
            if (c < (int)V_CHUNKS) {
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_ts(d, tmem + TM_Q + 32u * (uint32_t)c + 8u * (uint32_t)k, sdesc_sw128(sb + 32u * k, 16u, 1024u),
                           IDESC_S, (c > 0 || k > 0) ? 1u : 0u);
            } else {
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_ss(d, sdesc_sw128(smem + QPE0 + 32u * k, 16u, 1024u), sdesc_sw128(sb + 32u * k, 16u, 1024u),
                           IDESC_S, 1u);
            }
            if (c % SLOT_CHUNKS == SLOT_CHUNKS - 1) mma_commit(smem_u32(&h->c_empty[slot]));
        }
        if (!ok) break;
        mma_commit(smem_u32(&h->s_full[buf]));
        mbar_arrive(smem_u32(&h->s_full[buf]));
    }
    mma_commit(smem_u32(&h->drain));
    wait_bar(h, smem_u32(&h->drain), 0u, p.status, false, false);
}

// Softmax warps 0-7 (thread = row; warp group g = warp / 4 owns keys
// [64g, 64g + 64) of every S tile and always fills the partner's P buffer g,
// i.e. the partner consumes an S tile as two 64-key P halves).  Pass 1 reads
// the whole score row (the other group's half first) for the maximum, which
// both groups therefore agree on without exchanging data; pass 2 re-reads
// the group's own 64 scores for the exponentials.  Q goes in first: the
// no-PE dims to TMEM, the RoPE dims to shared memory.  After the last tile
// the groups add their partial sums; group 0 writes the lse to the
// workspace and 1/l to the partner.
__device__ void s_role_rows(const Params &p, Header *h, uint32_t smem, uint32_t tmem, const Unit &u)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int quad = warp & 3, grp = warp >> 2;
    const int r = quad * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const int H = p.num_heads;
    const int64_t lr = u.r0 + r;
    const bool row_ok = lr < u.rows_b;
    const int64_t i = row_ok ? lr / H : 0;
    const int64_t hh = row_ok ? lr % H : 0;

    // Q row: dims 0..511 -> TMEM columns [0, 256) (32-bit column k/2 holds
    // elements k, k+1; group 0 writes dims 0..255, group 1 dims 256..511);
    // dims 512..575 -> shared memory, K-major 128-byte swizzled (group 1).
    const __nv_bfloat16 *qrow = p.q + (u.qo0 + i) * p.q_stride_tok + hh * p.q_stride_head;
#pragma unroll 1
    for (int c = grp * 4; c < grp * 4 + 4; ++c) {
        uint32_t w[32];
#pragma unroll
        for (int v = 0; v < 8; ++v) {
            uint4 x = make_uint4(0u, 0u, 0u, 0u);
            if (row_ok) x = __ldg(reinterpret_cast<const uint4 *>(qrow + c * 64 + v * 8));
            w[4 * v] = x.x; w[4 * v + 1] = x.y; w[4 * v + 2] = x.z; w[4 * v + 3] = x.w;
        }
        tmem_st32(tmem + lane_base + TM_Q + 32u * (uint32_t)c, w);
    }
    if (grp == 1) {
        uint8_t *qpe = reinterpret_cast<uint8_t *>(h) + QPE0 + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
        for (int v = 0; v < 8; ++v) {
            uint4 x = make_uint4(0u, 0u, 0u, 0u);
            if (row_ok) x = __ldg(reinterpret_cast<const uint4 *>(qrow + 512 + v * 8));
            *reinterpret_cast<uint4 *>(qpe + ((v ^ (r & 7)) << 4)) = x;
        }
        fence_proxy_async_smem();
    }
    tmem_st_wait();
    tc_fence_before_sync();
    named_barrier_sync(1, SOFTMAX_THREADS + 32);

    const int64_t mrow = p.mask_indptr[u.b] + i * u.N;
    const float sl2 = p.sm_scale * LOG2E;
    const uint32_t peer_pbuf = map_cluster(smem + PBUF0, 1) + (uint32_t)grp * P_BUF;
    const uint32_t peer_alpha = map_cluster(smem_u32(&h->alpha[grp][0]), 1);
    const uint32_t peer_flags = map_cluster(smem_u32(&h->flags[grp]), 1);
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    // Mask bits of S tile t for this row (two 64-bit words), loaded one tile ahead.
    struct Bits { uint64_t w[2]; };
    auto mask_of = [&](int t) -> Bits {
        Bits b{{0ull, 0ull}};
        if (row_ok && t < u.ntiles_s) {
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int64_t j0 = tile_key0(u, t) + 64 * hf;
                const int64_t nk = u.k1 - j0;
                b.w[hf] = load_bits(p.custom_mask, mrow + j0, (int)(nk < 64 ? (nk > 0 ? nk : 0) : 64));
            }
        }
        return b;
    };
    Bits next_bits = mask_of(0);

    for (int t = 0; t < u.ntiles_s; ++t) {
        const int buf = t & 1;
        const Bits bits = next_bits;
        next_bits = mask_of(t + 1);
        if (!warp_wait(h, smem_u32(&h->s_full[buf]), (uint32_t)(t >> 1) & 1u, p.status, false)) { ok = false; break; }
        tc_fence_after_sync();
        const uint32_t s_col = tmem + lane_base + TM_S0 + 128u * (uint32_t)buf;
        uint64_t vis[2];
        vis[0] = *reinterpret_cast<volatile uint64_t *>(&h->s_valid[buf][0]) & bits.w[0];
        vis[1] = *reinterpret_cast<volatile uint64_t *>(&h->s_valid[buf][1]) & bits.w[1];
        const bool all_vis = __all_sync(0xffffffffu, (vis[0] & vis[1]) == ~0ull);
        uint32_t sv[32];
        // pass 1: maximum over all 128 scores, the other group's half first
        float mx = -INFINITY;
#pragma unroll
        for (int part = 0; part < 4; ++part) {
            const int half = (part < 2) ? 1 - grp : grp;
            const int q = 2 * half + (part & 1);        // 32-column quarter of the row
            tmem_ld32(s_col + 32u * (uint32_t)q, sv);
            tmem_ld_wait();
            const uint32_t vq = (uint32_t)(vis[half] >> (32 * (q & 1)));
            if (all_vis) {
#pragma unroll
                for (int n = 0; n < 32; ++n) mx = fmaxf(mx, __uint_as_float(sv[n]));
            } else {
#pragma unroll
                for (int n = 0; n < 32; ++n) mx = fmaxf(mx, ((vq >> n) & 1u) ? __uint_as_float(sv[n]) : -INFINITY);
            }
        }
        mx *= sl2;                                 // maximum in log2 units (sl2 > 0 keeps the order)
        float alpha = 1.f;
        bool rescale = false;
        if (mx > m_used + RESCALE_LOG2) {        // also the first tile where the row sees a key
            alpha = (m_used == -INFINITY) ? 0.f : ex2_approx(m_used - mx);
            l *= alpha;
            m_used = mx;
            rescale = true;
        }
        // The partner must be done with P buffer grp (this group's half of the previous S tile).
        if (t >= 1 && !warp_wait(h, smem_u32(&h->p_empty[grp]), (uint32_t)(t - 1) & 1u, p.status, true)) {
            ok = false;
            break;
        }
        // pass 2: p = 2^(s * sl2 - m_used) for this group's 64 keys; masked scores give 0.
        const float neg_m = m_used == -INFINITY ? 0.f : -m_used;
        const uint32_t prow = peer_pbuf + (uint32_t)(r >> 3) * 1024u + (uint32_t)(r & 7) * 128u;
        float psum = 0.f;
#pragma unroll
        for (int part = 0; part < 2; ++part) {
            tmem_ld32(s_col + 32u * (uint32_t)(2 * grp + part), sv);
            tmem_ld_wait();
            const uint32_t vq = (uint32_t)(vis[grp] >> (32 * part));
            uint32_t pk[16];
#pragma unroll
            for (int n = 0; n < 16; ++n) {
                const float a0 = (all_vis || ((vq >> (2 * n)) & 1u)) ? __uint_as_float(sv[2 * n]) : -INFINITY;
                const float a1 = (all_vis || ((vq >> (2 * n + 1)) & 1u)) ? __uint_as_float(sv[2 * n + 1]) : -INFINITY;
                const float p0 = ex2_approx(fmaf(a0, sl2, neg_m));
                const float p1 = ex2_approx(fmaf(a1, sl2, neg_m));
                psum += p0 + p1;
                pk[n] = pack_bf16x2(p0, p1);
            }
            // keys 32*part .. 32*part+31 of this group's half: 16-B pieces 4*part .. 4*part+3 of row r
#pragma unroll
            for (int qq = 0; qq < 4; ++qq)
                st_cluster_v4(prow + ((((uint32_t)(4 * part + qq)) ^ (uint32_t)(r & 7)) << 4), pk[4 * qq],
                              pk[4 * qq + 1], pk[4 * qq + 2], pk[4 * qq + 3]);
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&h->s_free[buf]));
        l += psum;
        // The O tile of group 0's half rescales O first; group 1's half follows with the same maximum.
        st_cluster_f32(peer_alpha + (uint32_t)r * 4u, (grp == 0 && rescale) ? alpha : 1.f);
        const uint32_t any = (grp == 0 && __any_sync(0xffffffffu, rescale)) ? 1u : 0u;
        if (lane == 0) st_cluster_u8(peer_flags + (uint32_t)quad, any);
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&h->p_written[grp]));
    }

    // Partial sums of group 1 -> group 0 (both groups always reach this barrier).
    float *lpart = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(h) + S_SCRATCH);
    if (grp == 1) lpart[r] = l;
    named_barrier_sync(2, SOFTMAX_THREADS);
    if (grp == 1) return;
    l += lpart[r];
    if (ok && row_ok) {
        const int64_t row = u.qo0 * H + lr;
        if (row < p.rows_cap)
            p.part_lse[(int64_t)u.split * p.rows_cap + row] = l > 0.f ? (m_used + log2f(l)) * LN2 : -INFINITY;
    }
    st_cluster_f32(map_cluster(smem_u32(&h->inv_l[r]), 1), l > 0.f ? 1.f / l : 0.f);
    __syncwarp();
    if (lane == 0) mbar_arrive_cluster(smem_u32(&h->l_ready), 1);
}

// Sender (warp 17, lane 0): once a softmax group stored its P half into the
// partner, order those writes for the partner's tensor-core reads and
// publish the O tile.  Keeps the proxy fence and the cluster-scope release
// off the softmax warps.
__device__ void s_role_sender(const Params &p, Header *h, const Unit &u)
{
    for (int t = 0; t < u.ntiles; ++t) {
        const int buf = t & 1;
        if (!wait_bar(h, smem_u32(&h->p_written[buf]), (uint32_t)(t >> 1) & 1u, p.status, false)) break;
        fence_proxy_async_cluster();
        mbar_arrive_cluster(smem_u32(&h->p_full[buf]), 1);
    }
}

// ------------------------------------------------------------------ O role

// MMA issue (warp 16, lane 0): O += P V for every tile, both 256-column halves.
__device__ void o_role_mma(const Params &p, Header *h, uint32_t smem, uint32_t tmem, const Unit &u)
{
    uint32_t nrs = 0;
    for (int t = 0; t < u.ntiles; ++t) {
        const int stage = t % STAGES, buf = t & 1;
        if (!wait_bar(h, smem_u32(&h->v_full[stage]), (uint32_t)(t / STAGES) & 1u, p.status, false)) break;
        if (!wait_bar(h, smem_u32(&h->p_full[buf]), (uint32_t)(t >> 1) & 1u, p.status, true)) break;
        const uint32_t flags = t > 0 ? *reinterpret_cast<volatile uint32_t *>(&h->flags[buf]) : 0u;
        if (flags) {
            mma_commit(smem_u32(&h->pv_sync));
            if (!wait_bar(h, smem_u32(&h->pv_sync), nrs & 1u, p.status, false)) break;
            mbar_arrive(smem_u32(&h->rs_req));
            if (!wait_bar(h, smem_u32(&h->rs_done), nrs & 1u, p.status, false)) break;
            ++nrs;
        }
        tc_fence_after_sync();
        fence_proxy_async_smem();
        const uint32_t pb = smem + PBUF0 + (uint32_t)buf * P_BUF;
        const uint32_t vb = smem + STAGE0 + (uint32_t)stage * V_STAGE;
#pragma unroll
        for (int k = 0; k < KEYS / 16; ++k) {
            const uint64_t adesc = sdesc_sw128(pb + 32u * (uint32_t)k, 16u, 1024u);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const uint64_t bdesc =
                    sdesc_sw128(vb + (uint32_t)half * 4u * CHUNK_BYTES + (uint32_t)k * 16u * 128u, CHUNK_BYTES, 1024u);
                mma_ss(tmem + 256u * (uint32_t)half, adesc, bdesc, IDESC_PV, (t > 0 || k > 0) ? 1u : 0u);
            }
        }
        mma_commit(smem_u32(&h->v_empty[stage]));
        mma_commit_multicast(smem_u32(&h->p_empty[buf]), (uint16_t)0x1);
    }
    mma_commit(smem_u32(&h->drain));
}

// Row warps (thread = TMEM lane = row): rescale O rows on flagged tiles;
// after the last tile, O / l -> fp32 partial in the workspace.
__device__ void o_role_rows(const Params &p, Header *h, uint32_t smem, uint32_t tmem, const Unit &u)
{
    const int r = threadIdx.x, warp = r >> 5, lane = r & 31;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    uint32_t nrs = 0;
    bool ok = true;
    for (int t = 0; t < u.ntiles; ++t) {
        const int buf = t & 1;
        if (!warp_wait(h, smem_u32(&h->p_full[buf]), (uint32_t)(t >> 1) & 1u, p.status, true)) { ok = false; break; }
        const uint32_t flags = t > 0 ? *reinterpret_cast<volatile uint32_t *>(&h->flags[buf]) : 0u;
        if (flags) {
            const float a = h->alpha[buf][r];
            if (!warp_wait(h, smem_u32(&h->rs_req), nrs & 1u, p.status, false)) { ok = false; break; }
            tc_fence_after_sync();
#pragma unroll 1
            for (int c = 0; c < DV / 32; ++c) {
                uint32_t v[32];
                tmem_ld32(tmem + lane_base + 32u * (uint32_t)c, v);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * a);
                tmem_st32(tmem + lane_base + 32u * (uint32_t)c, v);
            }
            tmem_st_wait();
            tc_fence_before_sync();
            mbar_arrive(smem_u32(&h->rs_done));
            ++nrs;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(smem_u32(&h->p_empty[buf]), 0);
    }
    if (!__all_sync(0xffffffffu, wait_bar(h, smem_u32(&h->drain), 0u, p.status, false, false))) ok = false;
    if (!warp_wait(h, smem_u32(&h->l_ready), 0u, p.status, true)) ok = false;
    tc_fence_after_sync();
    const float il = h->inv_l[r];
    const int64_t lr = u.r0 + r;
    const int64_t row = u.qo0 * p.num_heads + lr;
    const bool write = ok && lr < u.rows_b && row < p.rows_cap;
    float *dst = p.part_o + ((int64_t)u.split * p.rows_cap + (write ? row : 0)) * DV;
#pragma unroll 1
    for (int c = 0; c < DV / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + 32u * (uint32_t)c, v);
        tmem_ld_wait();
        if (write) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                float4 o;
                o.x = __uint_as_float(v[4 * e]) * il;
                o.y = __uint_as_float(v[4 * e + 1]) * il;
                o.z = __uint_as_float(v[4 * e + 2]) * il;
                o.w = __uint_as_float(v[4 * e + 3]) * il;
                *reinterpret_cast<float4 *>(dst + c * 32 + 4 * e) = o;
            }
        }
    }
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    tc_split_kernel(Params p, const __grid_constant__ CUtensorMap pool_map)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t smem = (raw + 1023u) & ~1023u;
    Header *h = reinterpret_cast<Header *>(smem_raw + (smem - raw));
    const uint32_t role = cluster_rank();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // a1: segment decode.  Both CTAs of the pair compute the same unit, so
    // they leave together when it is empty.
    // Grid: x = 2 * row tile + rank in the pair, y = split, z = request.  Row
    // tiles vary fastest, so pairs that read the same key chunk run together
    // and share it through L2.
    Unit u;
    u.split = (int)blockIdx.y;
    u.b = (int)blockIdx.z;
    u.qo0 = p.qo_indptr[u.b];
    const int64_t T = p.qo_indptr[u.b + 1] - u.qo0;
    u.kv0 = p.kv_indptr[u.b];
    u.L = p.kv_indptr[u.b + 1] - u.kv0;
    if (T < 0 || u.L < 0 || T > p.max_q_per_req) {
        if (role == 0 && u.split == 0 && blockIdx.x == 0 && tid == 0) atomicOr(p.status, STATUS_BAD_META);
        if (T < 0 || u.L < 0) return;
    }
    u.rows_b = (T < p.max_q_per_req ? T : p.max_q_per_req) * p.num_heads;
    u.r0 = (int64_t)(blockIdx.x >> 1) * ROWS;
    if (u.r0 >= u.rows_b) return;
    u.N = u.L + T;
    const int64_t chunk = split_chunk(u.N, p.num_splits);
    u.k0 = (int64_t)u.split * chunk;
    if (u.k0 >= u.N) return;
    u.k1 = (u.k0 + chunk < u.N) ? u.k0 + chunk : u.N;
    u.ntiles_s = (int)((u.k1 - u.k0 + KEYS_S - 1) / KEYS_S);
    u.ntiles = 2 * u.ntiles_s;
    {
        const int64_t row_tiles = (u.rows_b + ROWS - 1) / ROWS;
        u.rot = (int)(((int64_t)(blockIdx.x >> 1) * u.ntiles_s) / row_tiles);
    }

    if (tid == 0) {
        for (int s = 0; s < NSLOT; ++s) {
            mbar_init(smem_u32(&h->c_full[s]), PRODUCER_WARPS);
            mbar_init(smem_u32(&h->c_empty[s]), 1);
        }
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&h->v_full[s]), PRODUCER_WARPS);
            mbar_init(smem_u32(&h->v_empty[s]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&h->s_full[i]), 2);
            mbar_init(smem_u32(&h->s_free[i]), SOFTMAX_THREADS / 32);
            mbar_init(smem_u32(&h->p_written[i]), SOFTMAX_THREADS / 64);
            mbar_init(smem_u32(&h->p_empty[i]), 1 + 4);
            mbar_init(smem_u32(&h->p_full[i]), 1);
            h->flags[i] = 0u;
        }
        mbar_init(smem_u32(&h->pv_sync), 1);
        mbar_init(smem_u32(&h->rs_req), 1);
        mbar_init(smem_u32(&h->rs_done), ROWS);
        mbar_init(smem_u32(&h->l_ready), 4);
        mbar_init(smem_u32(&h->drain), 1);
        h->abort = 0u;
        fence_mbar_init_cluster();
    }
    if (warp == PRODUCER_WARP0 && lane == 0) prefetch_tensormap(&pool_map);
    if (warp == MMA_WARP) {
        tmem_alloc(smem_u32(&h->tmem_base), TMEM_COLS);
        tmem_relinquish();
        tc_fence_before_sync();
    }
    __syncthreads();
    cluster_sync();
    tc_fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(&h->tmem_base);

    if (role == 0) {
        if (warp < PRODUCER_WARP0) {
            s_role_rows(p, h, smem, tmem, u);
        } else if (warp < MMA_WARP) {
            s_role_gather(p, h, &pool_map, smem, u);
        } else if (warp == MMA_WARP) {
            named_barrier_sync(1, SOFTMAX_THREADS + 32);
            tc_fence_after_sync();
            if (lane == 0) s_role_mma(p, h, smem, tmem, u);
        } else if (lane == 0) {
            s_role_sender(p, h, u);
        }
    } else {
        if (warp < 4) {
            o_role_rows(p, h, smem, tmem, u);
        } else if (warp >= PRODUCER_WARP0 && warp < MMA_WARP) {
            gather_tiles<V_CHUNKS>(p, h, &pool_map, smem + STAGE0, V_STAGE, h->v_full, h->v_empty, nullptr, u);
        } else if (warp == MMA_WARP && lane == 0) {
            o_role_mma(p, h, smem, tmem, u);
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    cluster_sync();
    if (warp == MMA_WARP) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}


PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

// 2-D tensor map over the pool [pool_size rows, 576 bf16]: box of 64
// columns x 1 row (the gather4 form), 128-byte swizzle, zero fill outside.
bool encode_pool_map(const Params &p, CUtensorMap *map)
{
    if (g_encode == nullptr || p.pool_size >= ((int64_t)1 << 31)) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)p.pool_size};
    const cuuint64_t strides[1] = {(cuuint64_t)D * sizeof(__nv_bfloat16)};
    const cuuint32_t box[2] = {64, 1};
    const cuuint32_t estr[2] = {1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<__nv_bfloat16 *>(p.kv_pool), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t tc_init()
{
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (g_encode == nullptr) return cudaErrorNotSupported;
    return cudaFuncSetAttribute(tc_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_ALLOC);
}

bool tc_supported(const Params &p) { return p.pool_size < ((int64_t)1 << 31); }

cudaError_t launch_tc_split(const Params &p, cudaStream_t stream)
{
    CUtensorMap map;
    if (!encode_pool_map(p, &map)) return cudaErrorInvalidValue;
    const int row_tiles = (int)((p.max_q_per_req * (int64_t)p.num_heads + ROWS - 1) / ROWS);
    dim3 grid(2u * (unsigned)row_tiles, (unsigned)p.num_splits, (unsigned)p.batch);
    tc_split_kernel<<<grid, THREADS, SMEM_ALLOC, stream>>>(p, map);
    return cudaGetLastError();
}

}  // namespace va
