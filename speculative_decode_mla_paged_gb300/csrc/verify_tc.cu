// Tensor-core split kernel for tree-verify attention (sm_103a: tcgen05, TMEM,
// TMA gathers, bulk copies between the CTAs of a cluster).
//
// Work unit: one (key split, pair of 128-row tiles, request), the same
// unit as the pages' split-KV flash-decode partial ("The Capture-Safe
// Kernel", Decision 3), but every key tile is loaded once per 256 rows (T*H
// rows of one request share all keys: MLA latent attention, "The
// Integration Chasm", section Decision) and both contractions run on the
// tensor cores.
//
// A 4-CTA cluster per unit: ranks 2h and 2h + 1 serve row tile h of the
// pair (a request with at most 128 rows runs on a 2-CTA cluster of one row
// tile instead: see the cluster shapes below and launch_tc_split).  A
// 128 x 512 fp32 output accumulator is the whole of an SM's TMEM
// (128 lanes x 512 columns), so one SM cannot hold Q, the scores S and O for
// 128 rows; the two CTAs of a row tile split the work by role:
//
//   even rank ("S"): Q's 512 no-PE dims live in TMEM (256 columns of packed
//     bf16, the A operand of S = Q K^T from tensor memory), its 64 RoPE dims
//     in shared memory; a 128-key tile of K arrives by TMA gather4 as three
//     rounds of three 16 KB column chunks (a ring of one tile); two
//     128-column S buffers in TMEM.  Eight softmax warps (two groups of four,
//     thread = row, group g owns keys [64g, 64g + 64) of each tile) read
//     their scores once, exchange the row maximum through shared memory,
//     write P (bf16) to a local staging slot and ship each 64-key half to
//     the partner with one bulk copy whose bytes complete the partner's
//     barrier.
//   odd rank ("O"): the fp32 O accumulator fills its TMEM; V (the first
//     512 dims of the same rows) arrives by TMA gather4 in 64-key x 256-dim
//     half tiles; P halves land in four double-buffered slots;
//     O += P V runs as N = 256 MMAs with both operands in shared memory.
//
// Per 128-key tile the S CTA issues 36 MMAs (M128 N128 K16) and the O CTA 16
// (M128 N256 K16): 576 and 512 MACs per (row, key), balanced.
//
// The gathers set the pace (a TMA gather4 moves 512 B, and one warp issues
// them one at a time, lane after lane; a ring slot comes back only after its
// refill's issue and flight and the MMAs that read it).  The two S CTAs
// need the same K tiles and the two O CTAs the same V tiles, so each
// gathers half of every tile and multicasts it into both; a ring slot is
// reused once both consumers' MMAs have released it (tensor-core commits
// multicast to both).  Each CTA runs 16 producer warps that share every
// round, and setmaxnreg moves registers from the producer warpgroups to the
// softmax / row warpgroups.
//
// Online softmax with a lazy maximum: O is rescaled only when a row's
// running maximum grows by more than 32 (log2 units), so P stays <= 2^32.
// A rescale drains the P V MMAs and round-trips O through registers, so it
// is kept rare; the bound is set by range, not precision: P is bf16 (8
// exponent bits, like fp32), rounding is relative and so independent of the
// scale, and the fp32 sums l <= n 2^32 and |O| <= n 2^32 max|v| stay finite
// for any n < 2^31 keys and |v| < 2^64.  A row's first visible key needs no
// rescale (its O and l are still exactly 0).  The P transfer of a tile's
// first half carries the per-row factor and a per-warp flag; the O CTA's
// row warps rescale their TMEM rows only when a flag is set.
//
// Synchronisation uses mbarriers only: TMA and bulk-copy bytes complete
// barriers directly, tensor-core commits arrive on them (across the pair
// with a multicast commit), and no cluster-scope release is on the per-tile
// path.  Every wait is bounded (1 s of global time): on expiry the kernel
// sets STATUS_TIMEOUT, unwinds, lets the copies it issued land, drains its
// MMAs and frees TMEM.
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
constexpr int KEYS_S = 128;                // keys per S tile (N of the score MMAs)
constexpr int KEYS_O = 64;                 // keys per O tile (one P half)
constexpr int THREADS = 896;               // 28 warps = 7 warpgroups
constexpr int SOFTMAX_THREADS = 256;       // S: warps 0-7 (warpgroups 0, 1)
constexpr int PRODUCER_WARP0 = 8;          // both: warps 8-23 (warpgroups 2-5) issue the TMA gathers
constexpr int PRODUCER_WARPS = 16;
constexpr int MMA_WARP = 24;               // both: warpgroup 6; lane 0 of warp 24 issues the MMAs
constexpr int LAUNCH_REGS = 72;            // registers per thread at launch: 65536 / 896, rounded down to 8
constexpr int REGS_WIDE = 128;             // softmax and O-row warpgroups after setmaxnreg
constexpr int REGS_NARROW = 48;            // producer, MMA and idle warpgroups
static_assert(8 * 32 * REGS_WIDE + 20 * 32 * REGS_NARROW <= THREADS * LAUNCH_REGS,
              "the register split fits the launch allocation");
static_assert(4 * 32 * REGS_WIDE + 24 * 32 * REGS_NARROW <= THREADS * LAUNCH_REGS,
              "the O CTA's split fits the launch allocation");
constexpr uint32_t K_CHUNKS = D / 64;      // 9 column chunks per S tile
constexpr uint32_t KCHUNK = KEYS_S * 128;  // 16 KB: 128 keys x 64 dims
constexpr int RCHUNKS = 3;                 // S: chunks per gather round
constexpr uint32_t KROUND = RCHUNKS * KCHUNK;   // 48 KB
constexpr int NKR = K_CHUNKS / RCHUNKS;    // S: ring of 3 rounds (one tile); round g of every tile uses slot g
constexpr uint32_t VCHUNK = KEYS_O * 128;  // 8 KB: 64 keys x 64 dims
constexpr uint32_t VHALF = 4 * VCHUNK;     // 32 KB: 64 keys x 256 dims, the B of one N = 256 MMA
constexpr int NVH = 4;                     // O: V half-tile ring
constexpr uint32_t PTILE = ROWS * KEYS_O * 2;   // 16 KB P half: 128 rows x 64 keys bf16
constexpr uint32_t SIDE_BYTES = ROWS * 4 + 16;  // alpha[128] + 4 warp flags, after P in a first-half slot
constexpr uint32_t PSLOT = PTILE + 1024;        // 17 KB (keeps every slot 1 KB aligned)
constexpr uint32_t HEADER = 2048;
// S CTA shared memory
constexpr uint32_t S_QPE = HEADER;                   // Q RoPE dims: 128 rows x 128 B, A of the 4 last MMAs
constexpr uint32_t S_STAGE = S_QPE + ROWS * 128;     // P staging, one slot per softmax group
constexpr uint32_t S_RING = S_STAGE + 2 * PSLOT;     // K round ring
constexpr uint32_t S_XMAX = S_RING + NKR * KROUND;   // row maxima exchanged by the two groups [tile parity][group][row]
constexpr uint32_t S_END = S_XMAX + 2 * 2 * ROWS * 4;
// O CTA shared memory
constexpr uint32_t O_PSLOT = HEADER;                 // P slots [group][tile parity]
constexpr uint32_t O_VRING = O_PSLOT + 4 * PSLOT;    // V half-tile ring
constexpr uint32_t O_END = O_VRING + NVH * VHALF;
constexpr uint32_t SMEM_USED = S_END > O_END ? S_END : O_END;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;    // room to align the base to 1 KB
static_assert(SMEM_ALLOC <= 232448, "at most 227 KB of shared memory per CTA");
static_assert(S_RING % 1024 == 0 && O_VRING % 1024 == 0 && PSLOT % 1024 == 0, "swizzle atoms are 1 KB aligned");

// Cluster shapes: NT row tiles of 128 rows per cluster, 2 * NT CTAs.  NT = 2
// (the shape described above) for requests of more than 128 rows; NT = 1
// (one S and one O CTA, each gathering whole tiles) when T * H <= 128, so a
// short request does not hold two SMs for an empty row tile.
template <int NT>
struct Shape {
    static_assert(NT == 1 || NT == 2, "one or two row tiles per cluster");
    static constexpr uint16_t S_MASK = NT == 2 ? 0x5 : 0x1;   // the S CTAs (ranks 0, 2 / rank 0)
    static constexpr uint16_t O_MASK = NT == 2 ? 0xA : 0x2;   // the O CTAs (ranks 1, 3 / rank 1)
};
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S0 = 256;                      // S role: S buffers at columns 256 and 384
constexpr uint32_t IDESC_S = idesc_bf16(128, 128, false);
constexpr uint32_t IDESC_PV = idesc_bf16(128, 256, true);
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.69314718055994531f;
constexpr float RESCALE_LOG2 = 32.0f;         // lazy-rescale threshold (log2 units)
constexpr uint64_t TIMEOUT_NS = 1000000000ull;

// Shared-memory header at the (1 KB aligned) base; same offsets in both CTAs
// so a barrier or field can be addressed in the partner with mapa.
struct Header {
    uint64_t c_full[NKR];      // S: K round landed (8 producer-warp arrives + TMA bytes)
    uint64_t c_empty[NKR];     // S: the MMAs of both S CTAs reading the round completed (2 multicast commits)
    uint64_t s_full[2];        // S: scores ready (commit) + the MMA thread's arrive (orders the valid bits)
    uint64_t s_free[2];        // S: the 8 softmax warps have read the score buffer
    uint64_t p_empty[2][2];    // S: the partner's P V MMAs on P slot [group][parity] completed (its commit)
    uint64_t v_full[NVH];      // O: V half tile landed (8 producer-warp arrives + TMA bytes)
    uint64_t v_empty[NVH];     // O: the MMAs of both O CTAs reading it completed (2 multicast commits)
    uint64_t p_full[2][2];     // O: P slot landed (the MMA thread's expect-tx arrive + bulk-copy bytes)
    uint64_t pv_sync;          // O: every MMA issued so far completed (before a rescale)
    uint64_t rs_req;           // O: MMA thread asks the row warps to rescale O (or to finish)
    uint64_t rs_done;          // O: the 4 row warps rescaled their rows
    uint64_t l_ready;          // O: the partner's 4 group-0 warps wrote 1/l
    uint64_t drain;            // both: all MMAs of the CTA completed
    uint8_t t_valid[4][32];    // S: [tile % 4][key group g]: bit k = key 4g + k of the tile has a valid slot
    uint32_t tmem_base;
    uint32_t abort;
    int32_t rs_slot;           // O: tile parity of the P slot whose factors to apply; -1: finish
    uint32_t pad;
    float inv_l[ROWS];         // O: 1 / softmax denominator per row (0 if the row saw nothing)
    float lpart[ROWS];         // S: group 1's partial sums
};
static_assert(sizeof(Header) <= HEADER, "header fits");

struct Unit {
    int split, b, half;        // half: row tile of the cluster (cluster rank >> 1)
    int64_t qo0, kv0, L, N, k0, k1, r0, rows_b;
    int ntiles;                // S tiles of 128 keys; the O CTA processes 2 * ntiles 64-key halves
};

// First key of the t-th S tile of a unit.  The units of one split of a
// request (its pairs of row tiles) walk the same tiles in the same order,
// run together (pairs are the fastest grid index) and so share each tile
// through L2 instead of re-reading it from DRAM.
__device__ __forceinline__ int64_t tile_key0(const Unit &u, int t)
{
    return u.k0 + (int64_t)t * KEYS_S;
}

// ------------------------------------------------------------------ bounded waits

__device__ __forceinline__ bool wait_slow(Header *h, uint32_t bar, uint32_t parity, unsigned *status, bool cluster,
                                       bool stop_on_abort, uint64_t limit_ns)
{
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (cluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (stop_on_abort && *reinterpret_cast<volatile uint32_t *>(&h->abort)) return false;
            if (globaltimer_ns() - t0 > limit_ns) {
                if (stop_on_abort) {
                    atomicOr(status, STATUS_TIMEOUT);
                    *reinterpret_cast<volatile uint32_t *>(&h->abort) = 1u;
                }
                return false;
            }
        }
    }
}

// Wait for phase `parity` of a barrier.  False after a timeout (status bit
// set, abort flag raised) or when another thread of the CTA aborted.
__device__ __forceinline__ bool wait_bar(Header *h, uint32_t bar, uint32_t parity, unsigned *status,
                                         bool cluster = false, bool stop_on_abort = true,
                                         uint64_t limit_ns = TIMEOUT_NS)
{
    if (cluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
    return wait_slow(h, bar, parity, status, cluster, stop_on_abort, limit_ns);
}

// The same for all 32 lanes of a warp (keeps the warp converged for the
// .sync.aligned tcgen05 instructions that follow).
__device__ __forceinline__ bool warp_wait(Header *h, uint32_t bar, uint32_t parity, unsigned *status,
                                          bool cluster = false, uint64_t limit_ns = TIMEOUT_NS,
                                          bool stop_on_abort = true)
{
    return __all_sync(0xffffffffu, wait_bar(h, bar, parity, status, cluster, stop_on_abort, limit_ns)) != 0;
}

// For waits off the critical path (the O row warps, idle until a rescale or
// the epilogue): the thread sleeps between polls, so it takes no issue
// slots or ALU cycles from the warps doing the work.  Same bound and abort
// handling as wait_bar.
__device__ __forceinline__ bool wait_idle(Header *h, uint32_t bar, uint32_t parity, unsigned *status)
{
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        __nanosleep(256);
        if ((it & 15u) == 0) {
            if (*reinterpret_cast<volatile uint32_t *>(&h->abort)) return false;
            if (globaltimer_ns() - t0 > TIMEOUT_NS) {
                atomicOr(status, STATUS_TIMEOUT);
                *reinterpret_cast<volatile uint32_t *>(&h->abort) = 1u;
                return false;
            }
        }
    }
}

// Self-test of the failure path: one warp waits, with the split kernel's
// own bounded wait, on an mbarrier that nothing ever arrives on.  The wait
// must give up after `limit_ns`, set STATUS_TIMEOUT and the abort flag, and
// the kernel must return, leaving the context usable.
__global__ void __launch_bounds__(32, 1) wait_probe_kernel(unsigned *status, uint64_t limit_ns)
{
    __shared__ __align__(16) Header hs;
    Header *h = &hs;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&h->drain), 1);
        h->abort = 0u;
    }
    __syncthreads();
    if (warp_wait(h, smem_u32(&h->drain), 0u, status, false, limit_ns))
        atomicOr(status, 0x80000000u);   // cannot happen: nothing arrives; a set top bit would show it did
}

// After a timeout: TMA gathers and bulk copies already issued into this
// CTA's shared memory finish within microseconds; wait 50 us before the
// CTA may exit so none lands in memory that is no longer this CTA's.
__device__ __forceinline__ void settle_copies()
{
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 50000ull) {
    }
}

// ------------------------------------------------------------------ slots of four keys

// Raw slots of keys j0..j0+3 of the unit's request; bit k of `live` = key
// j0+k is inside the split.  Loads are issued here and used a tile later.
struct RawSlots {
    int64_t s[4];
    uint32_t live;
};

__device__ __forceinline__ RawSlots load_slots(const Params &p, const Unit &u, int64_t j0, bool lane_active)
{
    RawSlots r;
    r.live = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int64_t j = j0 + k;
        r.s[k] = -1;
        if (lane_active && j < u.k1) {
            r.live |= 1u << k;
            if (j < u.L) r.s[k] = p.kv_indices ? (int64_t)__ldg(p.kv_indices + u.kv0 + j) : -1;
            else r.s[k] = p.out_cache_loc ? __ldg(p.out_cache_loc + u.qo0 + (j - u.L)) : -1;
        }
    }
    return r;
}

// Gather rows of the four keys (a key without a valid slot reads row
// pool_size, outside the tensor map, which TMA fills with zeros) and the
// valid-bit nibble; a live key with an invalid slot raises STATUS_BAD_SLOT.
struct Slots {
    int y[4];
    uint32_t nib;
};

__device__ __forceinline__ Slots resolve_slots(const Params &p, const RawSlots &r)
{
    Slots o;
    o.nib = 0;
    bool bad = false;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const bool ok = r.s[k] >= 0 && r.s[k] < p.pool_size;
        o.y[k] = ok ? (int)r.s[k] : (int)p.pool_size;
        o.nib |= (ok ? 1u : 0u) << k;
        bad |= ((r.live >> k) & 1u) && !ok;
    }
    if (bad) atomicOr(p.status, STATUS_BAD_SLOT);
    return o;
}

// Slot of key j of the unit's request (-1 for a missing index buffer).
__device__ __forceinline__ int64_t slot_of(const Params &p, const Unit &u, int64_t j)
{
    if (j < u.L) return p.kv_indices ? (int64_t)__ldg(p.kv_indices + u.kv0 + j) : -1;
    return p.out_cache_loc ? __ldg(p.out_cache_loc + u.qo0 + (j - u.L)) : -1;
}

// True when every key of the unit, [k0, k1), sits in consecutive valid pool
// slots (a defragmented pool).  Called by all 512 producer threads of a CTA:
// the slots of the first and last key decide at once for every thread alike
// (so a fragmented pool costs two cached loads and no barrier); only if they
// line up do the threads check every consecutive pair and vote once.
__device__ bool unit_contiguous(const Params &p, const Unit &u, int pt)
{
    const int64_t first = slot_of(p, u, u.k0), last = slot_of(p, u, u.k1 - 1);
    if (first < 0 || last >= p.pool_size || last - first != u.k1 - 1 - u.k0) return false;
    bool ok = true;
#pragma unroll 1
    for (int64_t j = u.k0 + 1 + pt; j < u.k1; j += PRODUCER_WARPS * 32) ok &= slot_of(p, u, j) == slot_of(p, u, j - 1) + 1;
    return named_barrier_and(7, PRODUCER_WARPS * 32, ok);
}

// ------------------------------------------------------------------ S role: gather (warps 8-23)
//
// K chunk layout: 128 keys as 128-B rows (key n at n*128) of one 64-dim
// column block, 16-B pieces swizzled q -> q ^ (n & 7) inside each 1 KB group
// of 8 keys (the tensor map's 128-byte swizzle): the K-major B operand of
// the score MMAs.  A tile arrives as three rounds of three chunks; round g
// of tile t goes to ring slot g.  Producer warp w (0-15) resolves key
// groups w and w + 16 (four keys each) of every tile and, in the S CTA of
// row tile h, gathers group w + 16h: one TMA gather4 per chunk of every
// round, multicast to both S CTAs.  (A warp issues its TMA instructions one
// after another, so each warp issues only three per round.)
//
// Contiguous fast path: when all the unit's keys sit in consecutive pool
// slots (a defragmented pool; decided once per unit), one lane loads each
// chunk of a full tile with a single plain TMA tile of this CTA's 64 rows
// (run_map: box 64 x 64) instead of 16 gather4s.  A partial last tile is
// gathered, so no row past the unit's last key is read.
template <int NT>
__device__ void s_gather(const Params &p, Header *h, const CUtensorMap *tmap, const CUtensorMap *run_map,
                         uint32_t smem, const Unit &u)
{
    const int pw = (int)(threadIdx.x >> 5) - PRODUCER_WARP0;
    const int lane = threadIdx.x & 31;
    const bool act = lane < 2;
    const int kg = pw + 16 * lane;                 // lane 0: group pw (keys 0-63), lane 1: group pw + 16
    const bool issuer = act && (NT == 1 || lane == u.half);   // one S CTA: both lanes gather
    RawSlots raw = load_slots(p, u, tile_key0(u, 0) + kg * 4, act);
    Slots cur = resolve_slots(p, raw);
    if (u.ntiles > 1) raw = load_slots(p, u, tile_key0(u, 1) + kg * 4, act);
    const bool contiguous = unit_contiguous(p, u, pw * 32 + lane);
    bool ok = true;
    for (int t = 0; t < u.ntiles && ok; ++t) {
        const bool run = contiguous && tile_key0(u, t) + KEYS_S <= u.k1;
        const int base = cur.y[0];                       // warp 0, lane l: the slot of key 64 l
#pragma unroll 1
        for (int g = 0; g < NKR; ++g) {
            if (t > 0 && !__all_sync(0xffffffffu, wait_bar(h, smem_u32(&h->c_empty[g]), (uint32_t)(t - 1) & 1u, p.status))) {
                ok = false;
                break;
            }
            const uint32_t bar = smem_u32(&h->c_full[g]);
            if (g == 0) {
                if (act) reinterpret_cast<volatile uint8_t *>(&h->t_valid[t & 3][0])[kg] = (uint8_t)cur.nib;
                __syncwarp();                                 // lane 1's byte before lane 0's release
            }
            if (lane == 0) {
                if (pw == 0) mbar_arrive_expect_tx(bar, KROUND);   // both halves land here
                else mbar_arrive(bar);
            }
            if (run) {
                if (pw == 0 && issuer) {   // lane l loads keys [64 l, 64 l + 64)
                    const uint32_t dst = smem + S_RING + (uint32_t)g * KROUND + (uint32_t)lane * 64u * 128u;
#pragma unroll
                    for (int cc = 0; cc < RCHUNKS; ++cc) {
                        if constexpr (NT == 2)
                            tma_tile_multicast(dst + (uint32_t)cc * KCHUNK, run_map, (g * RCHUNKS + cc) * 64, base, bar,
                                               Shape<NT>::S_MASK);
                        else
                            tma_tile(dst + (uint32_t)cc * KCHUNK, run_map, (g * RCHUNKS + cc) * 64, base, bar);
                    }
                }
            } else if (issuer) {
                const uint32_t dst = smem + S_RING + (uint32_t)g * KROUND + (uint32_t)kg * 512u;
#pragma unroll
                for (int cc = 0; cc < RCHUNKS; ++cc) {
                    if constexpr (NT == 2)
                        tma_gather4_multicast(dst + (uint32_t)cc * KCHUNK, tmap, (g * RCHUNKS + cc) * 64, cur.y[0],
                                              cur.y[1], cur.y[2], cur.y[3], bar, Shape<NT>::S_MASK);
                    else
                        tma_gather4(dst + (uint32_t)cc * KCHUNK, tmap, (g * RCHUNKS + cc) * 64, cur.y[0], cur.y[1],
                                    cur.y[2], cur.y[3], bar);
                }
            }
        }
        if (!ok) break;
        if (t + 1 < u.ntiles) {
            cur = resolve_slots(p, raw);                        // loaded one tile ago
            if (t + 2 < u.ntiles) raw = load_slots(p, u, tile_key0(u, t + 2) + kg * 4, act);
        }
    }
    // Every round issued was consumed, unless a wait timed out: then give
    // the gathers in flight time to land before the CTA can exit.
    if (!ok) settle_copies();
}

// ------------------------------------------------------------------ S role: MMA issue (warp 24)
//
// S[buf] = Q K^T round by round: 32 MMAs with Q's no-PE dims from TMEM, then
// 4 with Q's RoPE dims from shared memory; each round is released by a commit.
//
// One lane issues every MMA, and the tensor pipe accepts only a few ahead
// of the one it runs, so the issuing lane's instruction stream sets the MMA
// rate: an M = 128, N = 128, K = 16 MMA occupies the pipe for 64 cycles,
// while the softmax warps on the same scheduler keep it busy.  So the issue
// path is kept short: the whole warp runs the loop and its waits (the
// operands are warp-uniform values), one lane issues, and the descriptors are
// built once and advanced by constants: the start address sits in the low 14
// bits in 16-B units, and shared-memory offsets below 256 KB never carry out
// of it, so desc(addr + off) = desc(addr) + off / 16.
static_assert(SMEM_ALLOC < (256u << 10), "descriptor arithmetic needs shared-memory offsets below 256 KB");

__device__ __forceinline__ uint64_t desc_add(uint64_t desc, uint32_t byte_off)
{
    return desc + (uint64_t)(byte_off >> 4);
}

template <int NT>
__device__ void s_mma(const Params &p, Header *h, uint32_t smem, uint32_t tmem, const Unit &u)
{
    // The whole warp runs the loop and waits, so the operands are warp-uniform
    // values; one lane issues each round's MMAs and commits.
    const bool issuer = (threadIdx.x & 31) == 0;
    const uint64_t ring_desc = sdesc_sw128(smem + S_RING, 16u, 1024u);
    const uint64_t qpe_desc = sdesc_sw128(smem + S_QPE, 16u, 1024u);
    for (int t = 0; t < u.ntiles; ++t) {
        const int buf = t & 1;
        if (t >= 2 && !warp_wait(h, smem_u32(&h->s_free[buf]), (uint32_t)((t >> 1) - 1) & 1u, p.status)) break;
        const uint32_t d = tmem + TM_S0 + 128u * (uint32_t)buf;
        bool ok = true;
#pragma unroll 1
        for (int g = 0; g < NKR; ++g) {
            if (!warp_wait(h, smem_u32(&h->c_full[g]), (uint32_t)t & 1u, p.status)) { ok = false; break; }
            tc_fence_after_sync();
            const uint64_t b0 = desc_add(ring_desc, (uint32_t)g * KROUND);
            const uint32_t a0 = tmem + 32u * (uint32_t)(g * RCHUNKS);
            if (issuer) {
#pragma unroll
                for (int cc = 0; cc < RCHUNKS; ++cc) {
                    const uint64_t b = desc_add(b0, (uint32_t)cc * KCHUNK);
                    if (g * RCHUNKS + cc < 8) {
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            mma_ts(d, a0 + 32u * (uint32_t)cc + 8u * (uint32_t)k, desc_add(b, 32u * (uint32_t)k), IDESC_S,
                                   (g | cc | k) ? 1u : 0u);
                    } else {
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            mma_ss(d, desc_add(qpe_desc, 32u * (uint32_t)k), desc_add(b, 32u * (uint32_t)k), IDESC_S, 1u);
                    }
                }
                mma_commit_multicast(smem_u32(&h->c_empty[g]), Shape<NT>::S_MASK);   // every S CTA may refill the slot
            }
            __syncwarp();
        }
        if (!ok) break;
        if (issuer) {
            mma_commit(smem_u32(&h->s_full[buf]));
            mbar_arrive(smem_u32(&h->s_full[buf]));
        }
        __syncwarp();
    }
    if (issuer) mma_commit(smem_u32(&h->drain));
    __syncwarp();
    warp_wait(h, smem_u32(&h->drain), 0u, p.status, false, TIMEOUT_NS, false);
}

// ------------------------------------------------------------------ S role: softmax (warps 0-7)

// Valid-slot bits of softmax group `grp`'s 64 keys of tile t (bit n = key
// 64 grp + n), from the producers' per-key-group nibbles: eight bytes, each
// holding one nibble, are packed into 32 bits by three shift-or-mask steps.
// The ring of four tiles is never overwritten too early: the producers write
// tile t + 4's entry after the score MMAs of tile t + 3 began, which waited
// for the softmax to free the score buffer of tile t + 1, so every softmax
// thread has read tile t's entry by then.  The producers' bytes reach this
// thread through c_full (their arrive, the MMA thread's wait) and s_full
// (the MMA thread's arrive, this thread's wait).
__device__ __forceinline__ uint64_t pack_nibbles(uint64_t x)
{
    x = (x | (x >> 4)) & 0x00FF00FF00FF00FFull;
    x = (x | (x >> 8)) & 0x0000FFFF0000FFFFull;
    return (x | (x >> 16)) & 0xFFFFFFFFull;
}

__device__ __forceinline__ uint64_t valid_bits(const Header *h, int t, int grp)
{
    const volatile uint64_t *v = reinterpret_cast<const volatile uint64_t *>(&h->t_valid[t & 3][16 * grp]);
    return pack_nibbles(v[0]) | (pack_nibbles(v[1]) << 32);
}


// nbits (<= 64) mask bits starting at bit index bit0, loaded as the one or
// two aligned 8-byte words that hold them (loads only), and their
// combination into a word (bit n = bit bit0 + n).  An aligned word that
// holds at least one of the wanted bytes lies in the same page as that byte,
// so the surplus bytes it carries never reach unmapped memory.
struct MaskBytes {
    uint64_t w0, w1;
    int sh, nbits;
};

__device__ __forceinline__ MaskBytes load_mask(const uint8_t *mask, int64_t bit0, int nbits)
{
    MaskBytes m;
    m.w0 = m.w1 = 0;
    m.nbits = nbits;
    const uintptr_t addr = reinterpret_cast<uintptr_t>(mask) + (uintptr_t)(bit0 >> 3);
    const uintptr_t aligned = addr & ~(uintptr_t)7;
    m.sh = (int)((addr - aligned) * 8 + (uintptr_t)(bit0 & 7));   // 0..63
    if (nbits > 0) {
        m.w0 = __ldg(reinterpret_cast<const unsigned long long *>(aligned));
        if (m.sh + nbits > 64) m.w1 = __ldg(reinterpret_cast<const unsigned long long *>(aligned) + 1);
    }
    return m;
}

__device__ __forceinline__ uint64_t mask_word(const MaskBytes &m)
{
    uint64_t w = m.sh ? ((m.w0 >> m.sh) | (m.w1 << (64 - m.sh))) : m.w0;
    if (m.nbits < 64) w &= m.nbits > 0 ? (1ull << m.nbits) - 1ull : 0ull;
    return w;
}

// Thread = row r (TMEM lane), group g = warp / 4 owns keys [64g, 64g + 64)
// of every S tile.  Per tile: read the group's 64 scores once into
// registers (which frees the S buffer for the next MMAs), exchange the
// row's partial maximum with the other group through shared memory, write
// P = 2^(s*scale*log2e - m) as bf16 into the group's staging slot (K-major,
// 128-byte swizzled: the A operand of the partner's P V MMAs), and the
// group's leader ships it with one bulk copy.  Q goes in first: no-PE dims
// to TMEM, RoPE dims to shared memory.
__device__ void s_softmax(const Params &p, Header *h, uint32_t smem, uint32_t tmem, const Unit &u)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int quad = warp & 3, grp = warp >> 2;
    const int r = quad * 32 + lane;
    const bool leader = (threadIdx.x & 127) == 0;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const int H = p.num_heads;
    const int64_t lr = u.r0 + r;
    const bool row_ok = lr < u.rows_b;
    const int64_t i = row_ok ? lr / H : 0;
    // A negative scale is folded into Q (exact sign flips) so the score
    // scale below is >= 0 and the maximum of s is the maximum of s * scale.
    const uint32_t qsign = p.sm_scale < 0.f ? 0x80008000u : 0u;
    const float sl2 = fabsf(p.sm_scale) * LOG2E;

    // Q rows: dims 0..511 -> TMEM columns [0, 256) (column k/2 holds
    // elements k, k+1; group 0 writes dims 0..255, group 1 dims 256..511);
    // dims 512..575 -> shared memory, K-major 128-byte swizzled (group 1).
    // The loads are coalesced: for each 64-dim chunk, lanes 8s..8s+7 read
    // the 128 contiguous bytes of row 4j + s of the warp's 32 rows (j = 0..7),
    // so one instruction covers four rows; the chunk goes through a 4 KB
    // per-warp stage (the P staging area, idle until the first tile; 16-B
    // pieces swizzled by row so writes and reads avoid bank conflicts) and
    // each thread then reads its own row for the TMEM store.
    const int sub = lane >> 3, piece = lane & 7;
    const __nv_bfloat16 *qsrc[8];      // row 4j + sub of this warp's 32 (null: past the request's rows)
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int64_t lrj = u.r0 + quad * 32 + 4 * j + sub;
        qsrc[j] = lrj < u.rows_b ? p.q + (u.qo0 + lrj / H) * p.q_stride_tok + (lrj % H) * p.q_stride_head + piece * 8
                                 : nullptr;
    }
    uint8_t *qst = reinterpret_cast<uint8_t *>(h) + S_STAGE + (uint32_t)warp * 4096u;
#pragma unroll 1
    for (int c = grp * 4; c < grp * 4 + 4; ++c) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            uint4 x = make_uint4(0u, 0u, 0u, 0u);
            if (qsrc[j] != nullptr) x = __ldg(reinterpret_cast<const uint4 *>(qsrc[j] + c * 64));
            const int k = 4 * j + sub;
            *reinterpret_cast<uint4 *>(qst + k * 128 + ((piece ^ (k & 7)) << 4)) = x;
        }
        __syncwarp();
        uint32_t w[32];
#pragma unroll
        for (int v = 0; v < 8; ++v) {
            const uint4 x = *reinterpret_cast<const uint4 *>(qst + lane * 128 + ((v ^ (lane & 7)) << 4));
            w[4 * v] = x.x ^ qsign; w[4 * v + 1] = x.y ^ qsign; w[4 * v + 2] = x.z ^ qsign; w[4 * v + 3] = x.w ^ qsign;
        }
        __syncwarp();                  // the next chunk reuses the stage
        tmem_st32(tmem + lane_base + 32u * (uint32_t)c, w);
    }
    if (grp == 1) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            uint4 x = make_uint4(0u, 0u, 0u, 0u);
            if (qsrc[j] != nullptr) x = __ldg(reinterpret_cast<const uint4 *>(qsrc[j] + 512));
            x.x ^= qsign; x.y ^= qsign; x.z ^= qsign; x.w ^= qsign;
            const int rr = quad * 32 + 4 * j + sub;
            *reinterpret_cast<uint4 *>(reinterpret_cast<uint8_t *>(h) + S_QPE + (rr >> 3) * 1024 + (rr & 7) * 128 +
                                       ((piece ^ (rr & 7)) << 4)) = x;
        }
        fence_proxy_async_smem();
    }
    tmem_st_wait();
    tc_fence_before_sync();
    named_barrier_sync(1, SOFTMAX_THREADS + 32);

    const int64_t mrow = p.mask_indptr[u.b] + i * u.N;
    uint8_t *stage = reinterpret_cast<uint8_t *>(h) + S_STAGE + (uint32_t)grp * PSLOT;
    uint8_t *prow = stage + (r >> 3) * 1024 + (r & 7) * 128;
    const uint32_t stage_u32 = smem + S_STAGE + (uint32_t)grp * PSLOT;
    const uint32_t copy_bytes = grp == 0 ? PTILE + SIDE_BYTES : PTILE;
    const uint32_t partner = 2u * (uint32_t)u.half + 1u;   // the O CTA of this row tile
    float *xmax = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(h) + S_XMAX);
    float m_used = -INFINITY, l = 0.f;
    bool ok = true, slot_failed = false;

    // This group's mask bits of a tile: bytes loaded a tile ahead, combined after use.
    auto mask_of = [&](int t) -> MaskBytes {
        const int64_t j0 = tile_key0(u, t) + 64 * grp;
        const int64_t nk = u.k1 - j0;
        return load_mask(p.custom_mask, mrow + j0, row_ok ? (int)(nk < 64 ? (nk > 0 ? nk : 0) : 64) : 0);
    };
    uint64_t bits = mask_word(mask_of(0));
    MaskBytes nm = mask_of(u.ntiles > 1 ? 1 : 0);

    for (int t = 0; t < u.ntiles; ++t) {
        const int buf = t & 1;
        const bool got = warp_wait(h, smem_u32(&h->s_full[buf]), (uint32_t)(t >> 1) & 1u, p.status);
        tc_fence_after_sync();
        const uint32_t s_col = tmem + lane_base + TM_S0 + 128u * (uint32_t)buf + 64u * (uint32_t)grp;
        uint32_t sa[32], sb[32];
        tmem_ld32(s_col, sa);
        tmem_ld32(s_col + 32u, sb);
        const uint64_t vis = valid_bits(h, t, grp) & bits;
        tmem_ld_wait();
        // The scores are in registers: the MMAs may refill this S buffer.
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&h->s_free[buf]));
        const bool all_vis = __all_sync(0xffffffffu, vis == ~0ull);
        const uint32_t v0 = (uint32_t)vis, v1 = (uint32_t)(vis >> 32);

        float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};   // independent chains
        if (all_vis) {
#pragma unroll
            for (int n = 0; n < 32; ++n) mx4[n & 3] = max3f(mx4[n & 3], __uint_as_float(sa[n]), __uint_as_float(sb[n]));
        } else {
#pragma unroll
            for (int n = 0; n < 32; ++n) {
                const float a = ((v0 >> n) & 1u) ? __uint_as_float(sa[n]) : -INFINITY;
                const float b = ((v1 >> n) & 1u) ? __uint_as_float(sb[n]) : -INFINITY;
                mx4[n & 3] = max3f(mx4[n & 3], a, b);
            }
        }
        const float lmax = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
        xmax[(buf * 2 + grp) * ROWS + r] = lmax;
        // The staging slot is free once the previous bulk copy has read it.
        if (leader) bulk_wait_read_all();
        // Both groups: maxima exchanged, staging slots free; all agree to go on
        // (a P slot wait that gave up in either group on the previous tile
        // votes no here, so the groups always leave the loop together).
        if (!named_barrier_and(5, SOFTMAX_THREADS, got && !slot_failed)) { ok = false; break; }
        float mx = fmaxf(lmax, xmax[(buf * 2 + (1 - grp)) * ROWS + r]);
        mx = mx == -INFINITY ? -INFINITY : mx * sl2;   // log2 units
        float alpha = 1.f;
        bool rescale = false;
        if (m_used == -INFINITY) {
            m_used = mx;                               // first visible key (or none yet): O and l are 0
        } else if (mx > m_used + RESCALE_LOG2) {
            alpha = ex2_approx(m_used - mx);
            l *= alpha;
            m_used = mx;
            rescale = true;
        }

        // p = 2^(s * sl2 - m_used) for this group's 64 keys; masked keys give
        // 0.  Scaling and summing run on key pairs (packed fp32 FMA and add).
        const float neg_m = m_used == -INFINITY ? 0.f : -m_used;
        const uint64_t sl2x2 = f2_pack(sl2, sl2), negm2 = f2_pack(neg_m, neg_m);
        uint64_t ps2[4] = {0ull, 0ull, 0ull, 0ull};   // independent chains of pair sums (+0.0f bits)
        // All 64 scalings first, then all 64 exponentials back to back, then
        // sums and bf16 packing (more independent work per warp).
        float x[64];
#pragma unroll
        for (int n = 0; n < 16; ++n) {
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sa[2 * n]), __uint_as_float(sa[2 * n + 1])), sl2x2, negm2),
                      x[2 * n], x[2 * n + 1]);
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sb[2 * n]), __uint_as_float(sb[2 * n + 1])), sl2x2, negm2),
                      x[32 + 2 * n], x[32 + 2 * n + 1]);
        }
#pragma unroll
        for (int n = 0; n < 64; ++n) x[n] = ex2_approx(x[n]);
        if (!all_vis) {
#pragma unroll
            for (int n = 0; n < 32; ++n) {
                x[n] = ((v0 >> n) & 1u) ? x[n] : 0.f;
                x[32 + n] = ((v1 >> n) & 1u) ? x[32 + n] : 0.f;
            }
        }
#pragma unroll
        for (int part = 0; part < 2; ++part) {
            uint32_t pk[16];
#pragma unroll
            for (int n = 0; n < 16; ++n) {
                const float p0 = x[32 * part + 2 * n], p1 = x[32 * part + 2 * n + 1];
                ps2[n & 3] = f2_add(ps2[n & 3], f2_pack(p0, p1));
                pk[n] = pack_bf16x2(p0, p1);
            }
            // keys 32*part .. +31 of this half: 16-B pieces 4*part .. 4*part+3 of row r
#pragma unroll
            for (int qq = 0; qq < 4; ++qq)
                *reinterpret_cast<uint4 *>(prow + ((((uint32_t)(4 * part + qq)) ^ (uint32_t)(r & 7)) << 4)) =
                    make_uint4(pk[4 * qq], pk[4 * qq + 1], pk[4 * qq + 2], pk[4 * qq + 3]);
        }
        {
            float a0, a1;
            f2_unpack(f2_add(f2_add(ps2[0], ps2[1]), f2_add(ps2[2], ps2[3])), a0, a1);
            l += a0 + a1;
        }
        if (grp == 0) {
            // The first half's O tile rescales O; the second half follows with the same maximum.
            reinterpret_cast<float *>(stage + PTILE)[r] = rescale ? alpha : 1.f;
            const uint32_t any = __any_sync(0xffffffffu, rescale) ? 1u : 0u;
            if (lane == 0) reinterpret_cast<uint32_t *>(stage + PTILE + ROWS * 4)[quad] = any;
        }
        fence_proxy_async_smem();
        // The partner must be done with P slot [grp][t & 1] (its use two tiles
        // ago).  Each group waits for its own slot and its own 128 threads'
        // P stores; the other group does not wait for it here.
        bool slot_free = true;
        if (leader && t >= 2)
            slot_free = wait_bar(h, smem_u32(&h->p_empty[grp][buf]), (uint32_t)((t >> 1) - 1) & 1u, p.status);
        const bool group_ok = grp == 0 ? named_barrier_and(6, SOFTMAX_THREADS / 2, slot_free)
                                       : named_barrier_and(9, SOFTMAX_THREADS / 2, slot_free);
        if (!group_ok) slot_failed = true;
        if (leader && !slot_failed) {
            bulk_copy_to_cluster(map_cluster(smem + O_PSLOT + (uint32_t)(2 * grp + buf) * PSLOT, partner), stage_u32,
                                 copy_bytes, map_cluster(smem_u32(&h->p_full[grp][buf]), partner));
            bulk_commit_group();
        }
        // mask bits of tile t + 1 (loaded during this tile), then the loads for t + 2
        bits = mask_word(nm);
        if (t + 2 < u.ntiles) nm = mask_of(t + 2);
    }
    if (slot_failed) ok = false;
    if (leader) bulk_wait_read_all();

    // Partial sums of group 1 -> group 0 (both groups always reach this barrier).
    if (grp == 1) h->lpart[r] = l;
    named_barrier_sync(4, SOFTMAX_THREADS);
    if (grp == 1) return;
    l += h->lpart[r];
    if (ok && row_ok) {
        const int64_t row = u.qo0 * H + lr;
        if (row < p.rows_cap)
            p.part_lse[(int64_t)u.split * p.rows_cap + row] = l > 0.f ? (m_used + log2f(l)) * LN2 : -INFINITY;
    }
    st_cluster_f32(map_cluster(smem_u32(&h->inv_l[r]), partner), l > 0.f ? 1.f / l : 0.f);
    __syncwarp();
    if (lane == 0) mbar_arrive_cluster(smem_u32(&h->l_ready), partner);
}

// ------------------------------------------------------------------ O role: gather (warps 8-23)
//
// V half tile layout: four 64-dim column blocks of 64 keys (8 KB each, key
// rows of 128 B swizzled as above): the MN-major B operand of one N = 256
// P V MMA.  Round R = 2 * (O tile) + value half goes to ring slot R % 4.
// With two row tiles, in the O CTA of row tile h, producer warp w gathers
// key group 8h + (w & 7) (four keys of the 64), column blocks 2 (w >> 3) and
// 2 (w >> 3) + 1 of every round, multicast to both O CTAs; with one row
// tile, warp w gathers key group w for all four column blocks.  Contiguous
// fast path as for K (decided once per unit, full O tiles only): one lane
// loads each column block with a plain TMA tile of this CTA's 32 rows
// (two row tiles; run_map: box 64 x 32) or of all 64 (one; box 64 x 64).
template <int NT>
__device__ void o_gather(const Params &p, Header *h, const CUtensorMap *tmap, const CUtensorMap *run_map,
                         uint32_t smem, const Unit &u)
{
    constexpr int NB = NT == 2 ? 2 : 4;            // column blocks per warp and round
    const int pw = (int)(threadIdx.x >> 5) - PRODUCER_WARP0;
    const int lane = threadIdx.x & 31;
    const bool act = lane == 0;
    const int kg = NT == 2 ? 8 * u.half + (pw & 7) : pw, blk0 = NT == 2 ? 2 * (pw >> 3) : 0;
    const int nt = 2 * u.ntiles;
    auto key0 = [&](int ot) { return tile_key0(u, ot >> 1) + (int64_t)(ot & 1) * KEYS_O + kg * 4; };
    RawSlots raw = load_slots(p, u, key0(0), act);
    Slots cur = resolve_slots(p, raw);
    raw = load_slots(p, u, key0(1), act);
    const bool contiguous = unit_contiguous(p, u, pw * 32 + lane);
    bool ok = true;
    int slot = 0;
    uint32_t phase = 0;
    for (int ot = 0; ot < nt && ok; ++ot) {
        const bool run = contiguous && key0(ot) - kg * 4 + KEYS_O <= u.k1;
        const int base = cur.y[0];                       // warp 0, lane 0: the first key this CTA loads
#pragma unroll 1
        for (int hf = 0; hf < 2; ++hf) {
            const int R = 2 * ot + hf;
            if (R >= NVH && !__all_sync(0xffffffffu, wait_bar(h, smem_u32(&h->v_empty[slot]), phase ^ 1u, p.status))) {
                ok = false;
                break;
            }
            const uint32_t bar = smem_u32(&h->v_full[slot]);
            if (lane == 0) {
                if (pw == 0) mbar_arrive_expect_tx(bar, VHALF);   // every O CTA's key groups land here
                else mbar_arrive(bar);
            }
            if (run) {
                if (pw == 0 && lane == 0) {
                    const uint32_t dst = smem + O_VRING + (uint32_t)slot * VHALF + (uint32_t)u.half * 32u * 128u;
#pragma unroll
                    for (int blk = 0; blk < 4; ++blk) {
                        if constexpr (NT == 2)
                            tma_tile_multicast(dst + (uint32_t)blk * VCHUNK, run_map, (4 * hf + blk) * 64, base, bar,
                                               Shape<NT>::O_MASK);
                        else
                            tma_tile(dst + (uint32_t)blk * VCHUNK, run_map, (4 * hf + blk) * 64, base, bar);
                    }
                }
            } else if (act) {
                const uint32_t dst = smem + O_VRING + (uint32_t)slot * VHALF + (uint32_t)kg * 512u;
#pragma unroll
                for (int j = 0; j < NB; ++j) {
                    if constexpr (NT == 2)
                        tma_gather4_multicast(dst + (uint32_t)(blk0 + j) * VCHUNK, tmap, (4 * hf + blk0 + j) * 64,
                                              cur.y[0], cur.y[1], cur.y[2], cur.y[3], bar, Shape<NT>::O_MASK);
                    else
                        tma_gather4(dst + (uint32_t)(blk0 + j) * VCHUNK, tmap, (4 * hf + blk0 + j) * 64, cur.y[0],
                                    cur.y[1], cur.y[2], cur.y[3], bar);
                }
            }
            if (++slot == NVH) { slot = 0; phase ^= 1u; }
        }
        if (!ok) break;
        if (ot + 1 < nt) {
            cur = resolve_slots(p, raw);
            if (ot + 2 < nt) raw = load_slots(p, u, key0(ot + 2), act);
        }
    }
    if (!ok) settle_copies();
}

// ------------------------------------------------------------------ O role: MMA issue (warp 24)
//
// O += P V per 64-key O tile: two halves of the value dims, N = 256 each.
// P slot [g][par] of O tile ot: g = ot & 1 (softmax group), par = (ot >> 1) & 1.
template <int NT>
__device__ void o_mma(const Params &p, Header *h, uint32_t smem, uint32_t tmem, const Unit &u)
{
    // Run by the whole warp like s_mma: uniform operands, one issuing lane.
    const bool issuer = (threadIdx.x & 31) == 0;
    const int nt = 2 * u.ntiles;
    const uint64_t p_desc = sdesc_sw128(smem + O_PSLOT, 16u, 1024u);   // A: P, K-major
    const uint64_t v_desc = sdesc_sw128(smem + O_VRING, VCHUNK, 1024u);  // B: V, MN-major
    int slot = 0;
    uint32_t phase = 0, nrs = 0;
    uint32_t pphase = 0;       // bit 2g + par: parity of P slot [g][par]'s pending transfer
    bool ok = true;
    for (int ot = 0; ot < nt && ok; ++ot) {
        const int g = ot & 1, par = (ot >> 1) & 1;
        if (!warp_wait(h, smem_u32(&h->p_full[g][par]), (pphase >> (2 * g + par)) & 1u, p.status)) { ok = false; break; }
        pphase ^= 1u << (2 * g + par);
        if (g == 0 && ot > 0) {
            const volatile uint32_t *f = reinterpret_cast<const volatile uint32_t *>(
                reinterpret_cast<uint8_t *>(h) + O_PSLOT + (2 * g + par) * PSLOT + PTILE + ROWS * 4);
            if (f[0] | f[1] | f[2] | f[3]) {
                if (issuer) mma_commit(smem_u32(&h->pv_sync));
                __syncwarp();
                if (!warp_wait(h, smem_u32(&h->pv_sync), nrs & 1u, p.status)) { ok = false; break; }
                if (issuer) {
                    *reinterpret_cast<volatile int32_t *>(&h->rs_slot) = par;
                    mbar_arrive(smem_u32(&h->rs_req));
                }
                __syncwarp();
                if (!warp_wait(h, smem_u32(&h->rs_done), nrs & 1u, p.status)) { ok = false; break; }
                ++nrs;
            }
        }
        tc_fence_after_sync();
        const uint64_t a = desc_add(p_desc, (uint32_t)(2 * g + par) * PSLOT);
#pragma unroll 1
        for (int hf = 0; hf < 2; ++hf) {
            if (!warp_wait(h, smem_u32(&h->v_full[slot]), phase, p.status)) { ok = false; break; }
            tc_fence_after_sync();
            const uint64_t b = desc_add(v_desc, (uint32_t)slot * VHALF);
            if (issuer) {
#pragma unroll
                for (int k = 0; k < KEYS_O / 16; ++k)
                    mma_ss(tmem + 256u * (uint32_t)hf, desc_add(a, 32u * (uint32_t)k),
                           desc_add(b, (uint32_t)k * 16u * 128u), IDESC_PV, (ot | k) ? 1u : 0u);
                mma_commit_multicast(smem_u32(&h->v_empty[slot]), Shape<NT>::O_MASK);   // every O CTA may refill the slot
            }
            __syncwarp();
            if (++slot == NVH) { slot = 0; phase ^= 1u; }
        }
        if (!ok) break;
        if (issuer) {
            mma_commit_multicast(smem_u32(&h->p_empty[g][par]), (uint16_t)(1u << (2 * u.half)));   // this row tile's S CTA
            // arm this slot for its next P transfer
            mbar_arrive_expect_tx(smem_u32(&h->p_full[g][par]), g == 0 ? PTILE + SIDE_BYTES : PTILE);
        }
        __syncwarp();
    }
    if (issuer) {
        mma_commit(smem_u32(&h->drain));
        *reinterpret_cast<volatile int32_t *>(&h->rs_slot) = -1;
        mbar_arrive(smem_u32(&h->rs_req));
    }
    __syncwarp();
    if (!ok) settle_copies();   // P transfers already on their way land before the CTA can exit
}

// Row warps 0-3 (thread = TMEM lane = row): rescale O rows when asked;
// after the last tile, O / l -> fp32 partial in the workspace.
__device__ void o_rows(const Params &p, Header *h, uint32_t smem, uint32_t tmem, const Unit &u)
{
    const int r = threadIdx.x, warp = r >> 5, lane = r & 31;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    bool ok = true;
    for (uint32_t n = 0;; ++n) {
        if (!__all_sync(0xffffffffu, wait_idle(h, smem_u32(&h->rs_req), n & 1u, p.status))) { ok = false; break; }
        const int par = *reinterpret_cast<volatile int32_t *>(&h->rs_slot);
        if (par < 0) break;
        const float a = reinterpret_cast<const float *>(reinterpret_cast<uint8_t *>(h) + O_PSLOT +
                                                        (uint32_t)par * PSLOT + PTILE)[r];
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
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&h->rs_done));
    }
    if (!__all_sync(0xffffffffu, wait_bar(h, smem_u32(&h->drain), 0u, p.status, false, false))) ok = false;
    if (!warp_wait(h, smem_u32(&h->l_ready), 0u, p.status, true)) ok = false;
    tc_fence_after_sync();
    // O / l -> fp32 partial rows, 32 columns at a time.  Each warp stages its
    // 32 rows x 32 columns in shared memory (the V ring, idle once the MMAs
    // have drained; rows padded to 36 floats so the 16-B writes and reads
    // below are free of bank conflicts) and writes them back four rows per
    // instruction: lanes 8k..8k+7 store one row's 128 contiguous bytes,
    // where a thread storing its own row would scatter 32 16-B pieces.
    const float il = h->inv_l[r];
    float *stage = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(h) + O_VRING) + warp * 32 * 36;
    const int sub = lane >> 3, col4 = (lane & 7) * 4;
    float *dst[8];                    // row 4i + sub of this warp's 32, or null when not written
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t lr = u.r0 + warp * 32 + 4 * i + sub;
        const int64_t row = u.qo0 * p.num_heads + lr;
        dst[i] = ok && lr < u.rows_b && row < p.rows_cap ? p.part_o + ((int64_t)u.split * p.rows_cap + row) * DV + col4
                                                         : nullptr;
    }
#pragma unroll 1
    for (int c = 0; c < DV / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + 32u * (uint32_t)c, v);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 8; ++e)
            *reinterpret_cast<float4 *>(stage + lane * 36 + 4 * e) =
                make_float4(__uint_as_float(v[4 * e]) * il, __uint_as_float(v[4 * e + 1]) * il,
                            __uint_as_float(v[4 * e + 2]) * il, __uint_as_float(v[4 * e + 3]) * il);
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 x = *reinterpret_cast<const float4 *>(stage + (4 * i + sub) * 36 + col4);
            if (dst[i] != nullptr) *reinterpret_cast<float4 *>(dst[i] + c * 32) = x;
        }
        __syncwarp();                 // the next chunk reuses the stage
    }
}

// Launched with clusters of 2 * NT CTAs (a launch attribute).
template <int NT>
__global__ void __launch_bounds__(THREADS, 1)
    tc_split_kernel(Params p, const __grid_constant__ CUtensorMap pool_map,
                    const __grid_constant__ CUtensorMap run_map_k, const __grid_constant__ CUtensorMap run_map_v)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t smem = (raw + 1023u) & ~1023u;
    Header *h = reinterpret_cast<Header *>(smem_raw + (smem - raw));
    const uint32_t rank = cluster_rank();
    const uint32_t role = rank & 1u;        // 0: S, 1: O
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // Segment decode.  All CTAs of the cluster compute the same unit, so
    // they leave together when it is empty.  Grid: x = 2 NT * (group of NT
    // row tiles) + rank, y = split, z = request; row groups vary fastest, so
    // clusters that read the same key chunk run together and share it
    // through L2.  With NT = 2 the second row tile may be past the request's
    // rows: its CTAs still take part (their gathers feed the first row tile)
    // on zero rows.
    Unit u;
    u.split = (int)blockIdx.y;
    u.b = (int)blockIdx.z;
    u.half = (int)(rank >> 1);
    u.qo0 = p.qo_indptr[u.b];
    const int64_t T = p.qo_indptr[u.b + 1] - u.qo0;
    u.kv0 = p.kv_indptr[u.b];
    u.L = p.kv_indptr[u.b + 1] - u.kv0;
    if (T < 0 || u.L < 0 || T > p.max_q_per_req) {
        if (role == 0 && u.split == 0 && blockIdx.x == 0 && tid == 0) atomicOr(p.status, STATUS_BAD_META);
        if (T < 0 || u.L < 0) return;
    }
    u.rows_b = (T < p.max_q_per_req ? T : p.max_q_per_req) * p.num_heads;
    if (u.rows_b <= p.rows_lo || u.rows_b > p.rows_hi) return;   // served by the other cluster shape
    const int64_t first_row = (int64_t)(blockIdx.x / (2 * NT)) * (NT * ROWS);   // the cluster's first row
    if (first_row >= u.rows_b) return;
    u.r0 = first_row + (int64_t)u.half * ROWS;
    u.N = u.L + T;
    const int64_t chunk = split_chunk(u.N, p.num_splits);
    u.k0 = (int64_t)u.split * chunk;
    if (u.k0 >= u.N) return;
    u.k1 = (u.k0 + chunk < u.N) ? u.k0 + chunk : u.N;
    u.ntiles = (int)((u.k1 - u.k0 + KEYS_S - 1) / KEYS_S);

    if (tid == 0) {
        for (int s = 0; s < NKR; ++s) {
            mbar_init(smem_u32(&h->c_full[s]), PRODUCER_WARPS);
            mbar_init(smem_u32(&h->c_empty[s]), NT);
        }
        for (int s = 0; s < NVH; ++s) {
            mbar_init(smem_u32(&h->v_full[s]), PRODUCER_WARPS);
            mbar_init(smem_u32(&h->v_empty[s]), NT);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&h->s_full[i]), 2);
            mbar_init(smem_u32(&h->s_free[i]), SOFTMAX_THREADS / 32);
            for (int j = 0; j < 2; ++j) {
                mbar_init(smem_u32(&h->p_empty[i][j]), 1);
                mbar_init(smem_u32(&h->p_full[i][j]), 1);
            }
        }
        mbar_init(smem_u32(&h->pv_sync), 1);
        mbar_init(smem_u32(&h->rs_req), 1);
        mbar_init(smem_u32(&h->rs_done), 4);
        mbar_init(smem_u32(&h->l_ready), 4);
        mbar_init(smem_u32(&h->drain), 1);
        h->abort = 0u;
        h->rs_slot = 0;
        fence_mbar_init_cluster();
        if (role == 1)   // the P slots expect their first transfers
            for (int i = 0; i < 2; ++i)
                for (int j = 0; j < 2; ++j)
                    mbar_arrive_expect_tx(smem_u32(&h->p_full[i][j]), i == 0 ? PTILE + SIDE_BYTES : PTILE);
    }
    if (warp == PRODUCER_WARP0 && lane == 0) {
        prefetch_tensormap(&pool_map);
        prefetch_tensormap(role == 0 || NT == 1 ? &run_map_k : &run_map_v);
    }
    if (warp == MMA_WARP) {
        tmem_alloc(smem_u32(&h->tmem_base), TMEM_COLS);
        tmem_relinquish();
        tc_fence_before_sync();
    }
    __syncthreads();
    cluster_sync();
    tc_fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(&h->tmem_base);

    // Roles by warpgroup; setmaxnreg moves registers from the producer, MMA
    // and idle warpgroups to the softmax / row warpgroups, once.  No
    // warpgroup changes its budget again: an increase waits until the pool
    // covers it, so a narrow warpgroup that handed its registers back and then
    // asked for them again (an idle one at once, a producer when done) could
    // take them before a wide warpgroup's increase was served, and in the S
    // CTA the pool cannot cover both (8 softmax warps at 128, 17 warps at 48
    // and the MMA warpgroup's 3 idle warps back at 72 need 1280 registers more
    // than the 896 x 72 launch allocation): a softmax warpgroup would wait
    // forever.
    // With decreases only on the narrow side, the one increase per wide
    // warpgroup is always covered once the decreases have run.
    const bool wide = role == 0 ? warp < PRODUCER_WARP0 : warp < 4;
    if (wide) {
        regs_inc<REGS_WIDE>();
        if (role == 0) s_softmax(p, h, smem, tmem, u);
        else o_rows(p, h, smem, tmem, u);
    } else {
        regs_dec<REGS_NARROW>();
        if (warp >= PRODUCER_WARP0 && warp < MMA_WARP) {
            if (role == 0) s_gather<NT>(p, h, &pool_map, &run_map_k, smem, u);
            else o_gather<NT>(p, h, &pool_map, NT == 2 ? &run_map_v : &run_map_k, smem, u);
        } else if (warp == MMA_WARP) {
            if (role == 0) {
                named_barrier_sync(1, SOFTMAX_THREADS + 32);
                tc_fence_after_sync();
                s_mma<NT>(p, h, smem, tmem, u);
            } else {
                o_mma<NT>(p, h, smem, tmem, u);
            }
        }
        __syncwarp();
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
// columns x `rows` rows (1 row: the gather4 form; 64 / 32 rows: the
// contiguous fast path's tiles), 128-byte swizzle, zero fill outside.
bool encode_pool_map(const Params &p, CUtensorMap *map, uint32_t rows = 1)
{
    if (g_encode == nullptr || p.pool_size >= ((int64_t)1 << 31)) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)p.pool_size};
    const cuuint64_t strides[1] = {(cuuint64_t)D * sizeof(__nv_bfloat16)};
    const cuuint32_t box[2] = {64, rows};
    const cuuint32_t estr[2] = {1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<__nv_bfloat16 *>(p.kv_pool), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t side_init();

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
    // setmaxnreg.inc waits for registers the CTA does not have if the
    // launch allocation is smaller than the split assumes: refuse to run.
    for (const void *fn : {reinterpret_cast<const void *>(tc_split_kernel<1>),
                           reinterpret_cast<const void *>(tc_split_kernel<2>)}) {
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, fn);
        if (e != cudaSuccess) return e;
        if (fa.numRegs < LAUNCH_REGS || fa.maxThreadsPerBlock < THREADS) return cudaErrorNotSupported;
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_ALLOC);
        if (e != cudaSuccess) return e;
    }
    return side_init();
}

bool tc_supported(const Params &p) { return p.pool_size < ((int64_t)1 << 31); }

cudaError_t tc_thread_init() { return side_init(); }

cudaError_t launch_wait_probe(unsigned *status, uint64_t limit_ns, cudaStream_t stream)
{
    wait_probe_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
    return cudaGetLastError();
}

namespace {

// Grid: `groups` row groups of NT row tiles (0: enough for max_q_per_req * H rows).
template <int NT>
cudaError_t launch_shape(const Params &p, const CUtensorMap &map, const CUtensorMap &run_k, const CUtensorMap &run_v,
                         cudaStream_t stream, int groups = 0)
{
    if (groups == 0) groups = (int)((p.max_q_per_req * (int64_t)p.num_heads + NT * ROWS - 1) / (NT * ROWS));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2u * NT * (unsigned)groups, (unsigned)p.num_splits, (unsigned)p.batch);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = SMEM_ALLOC;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2 * NT;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tc_split_kernel<NT>, p, map, run_k, run_v);
}

// Per device: a second stream and the two events that fork the 4-CTA launch
// of a mixed call onto it and join it back (created once, before capture).
// The second stream of mixed-shape calls, with its fork and join events:
// one per host thread and device, so that calls (and stream captures) made
// from different threads never share it.  A thread's calls are sequential,
// so it needs no lock; the objects live until the process ends.
struct SideStream {
    cudaStream_t stream = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};
thread_local SideStream t_side[64];

cudaError_t side_init()
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    SideStream &ss = t_side[dev];
    if (ss.join != nullptr) return cudaSuccess;
    if (ss.stream == nullptr && (e = cudaStreamCreateWithFlags(&ss.stream, cudaStreamNonBlocking)) != cudaSuccess)
        return e;
    if (ss.fork == nullptr && (e = cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming)) != cudaSuccess)
        return e;
    return cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming);
}

// The three pool tensor maps of the last pool seen on each device (a pool is
// normally one long-lived allocation, so a call reuses them).
struct MapCache {
    const void *pool = nullptr;
    int64_t pool_size = -1;
    CUtensorMap map, run_k, run_v;
    std::mutex lock;
};
MapCache g_maps[64];

bool pool_maps(const Params &p, CUtensorMap *map, CUtensorMap *run_k, CUtensorMap *run_v)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    MapCache &mc = g_maps[dev];
    std::lock_guard<std::mutex> g(mc.lock);
    if (mc.pool != p.kv_pool || mc.pool_size != p.pool_size) {
        mc.pool = nullptr;
        if (!encode_pool_map(p, &mc.map) || !encode_pool_map(p, &mc.run_k, 64) || !encode_pool_map(p, &mc.run_v, 32))
            return false;
        mc.pool = p.kv_pool;
        mc.pool_size = p.pool_size;
    }
    *map = mc.map;
    *run_k = mc.run_k;
    *run_v = mc.run_v;
    return true;
}

}  // namespace

// Requests with T * H <= 128 run on 2-CTA clusters (one row tile), larger
// ones on 4-CTA clusters.  When a call may hold both, the 4-CTA launch takes
// the large requests on the caller's stream and the 2-CTA launch the small
// ones on a second stream forked from it and joined back, so the two grids
// share the GPU (including the SMs that 4-CTA clusters leave over).
cudaError_t launch_tc_split(const Params &p, cudaStream_t stream)
{
    CUtensorMap map, run_k, run_v;
    if (!pool_maps(p, &map, &run_k, &run_v)) return cudaErrorInvalidValue;
    if (p.max_q_per_req * (int64_t)p.num_heads <= ROWS) return launch_shape<1>(p, map, run_k, run_v, stream);
    if (p.max_q_per_req < 1 || p.num_heads > ROWS) return launch_shape<2>(p, map, run_k, run_v, stream);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    cudaError_t e = side_init();   // this thread's first mixed call on the device creates its second stream
    if (e != cudaSuccess) return e;
    SideStream &ss = t_side[dev];
    Params big = p, small = p;
    big.rows_lo = ROWS;
    small.rows_hi = ROWS;
    // The small requests' grid must start first: its clusters take SMs before
    // the large grid fills the GPU, so short units do not end up in the tail
    // (measured: 635 against 671 us per graph replay of the ragged workload).
    // So it goes on the caller's stream, where it depends on nothing new, and
    // the large grid on the side stream behind the fork event; the other way
    // round the large grid started first in direct calls, whatever the
    // enqueue order.
    if ((e = cudaEventRecord(ss.fork, stream)) != cudaSuccess) return e;
    if ((e = launch_shape<1>(small, map, run_k, run_v, stream, 1)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(ss.stream, ss.fork, 0)) != cudaSuccess) return e;
    if ((e = launch_shape<2>(big, map, run_k, run_v, ss.stream)) != cudaSuccess) return e;
    if ((e = cudaEventRecord(ss.join, ss.stream)) != cudaSuccess) return e;
    return cudaStreamWaitEvent(stream, ss.join, 0);
}

}  // namespace va
