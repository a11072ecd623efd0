// ssd_chunk_tc.cu -- the fused chunked SSD scan on Blackwell tensor cores (bf16).
//
// One CTA walks one (segment, head) work item piece by piece with the running
// state kept in tensor memory (TMEM) for the whole segment, so chunk states
// never travel through HBM.  A piece is a tile of at most 128 tokens: pieces
// are cut at absolute multiples of the tile size Qi and also end where a
// segment or a request ends.  Per piece the kernel evaluates the SSD chunk
// decomposition of h_t = exp(dt'_t A) h_{t-1} + dt'_t x_t (outer) B_t:
//   cs_t      = inclusive sum of dt'_s A over the piece, from its first token
//   CB        = C B^T                                  (bmm_chunk, tcgen05)
//   M[t,s]    = CB[t,s] exp(cs_t - cs_s) dt'_s, s <= t (the causal mask L o CB)
//   y_intra   = M x                                    (tcgen05, M read from TMEM)
//   y_inter   = exp(cs_t) C h_prev^T                   (tcgen05)
//   y         = (y_intra + y_inter + D x) * silu(z)
//   h_new^T   = exp(cs_last) h_prev^T + B^T (w x),  w_t = exp(cs_last - cs_t) dt'_t
// cs is measured from the piece's first valid token, so an initial state (or
// the state carried in from the previous piece) decays from exactly that
// token: the initial-state decay fix of the "[Bugfix] Mamba2 SSD varlen bug fix
// initstates decay" page.  Exported chunk states, block checkpoints and final
// states are read out of TMEM at the piece boundaries where they fall.
//
// D x is folded into the diagonal of M, so y_intra already carries the skip.
//
// Precision: rounding an operand to bf16 loses 8 bits, which breaks the 5e-3
// tolerance on y.  The three operands that are not exact bf16 inputs -- M,
// the carried state h and the weighted inputs w x -- are each split into
// bf16 hi + lo parts and their products issued twice into the fp32
// accumulator.  CB, x, B and C are exact bf16 and go in once.
//
// Roles (640 threads, warp-specialised):
//   warp 0  producer: draws the work items (a ticket counter in the scan), the
//           x tiles by TMA into a double-buffered stage (P = 64), and per piece
//           dt' and the cumulative decay, computed once and published beside
//           the x tile;
//   warp 1  MMA issuer (one lane) and TMEM owner;
//   G1      warps 2-9: w x split tiles, causal mask;
//   G2      warps 10-17: state bookkeeping, epilogue (z read from global memory,
//           y staged in the piece's x tile and stored with coalesced writes),
//           chunk/block/final states;
//   warp 18 B and C tiles by TMA into double buffers (P = 64), each buffer
//           reloaded as soon as its last MMA has read it (C after y_inter, B
//           after the state update), so the next piece's tiles load while this
//           piece computes;
//   warp 19 z tiles by TMA when the layout stages z (no current layout does).
// Each of G1 and G2 has two warps per TMEM lane quadrant (thread r owns tile
// row / TMEM lane r) that split the columns; many warps per role hide the
// latency of TMEM and shared-memory traffic.
// G1 can run a piece ahead of G2, and the y accumulators are double-buffered in
// TMEM (P = 64), so the mask of one piece overlaps the epilogue of the last.
// Every wait is a bounded mbarrier wait; on a timeout the CTA records
// SSD_DEVERR_TIMEOUT, drains what it issued and exits.
//
// A second mode (STATE_ONLY) computes, for each segment that is not the last
// of its request, the segment's end state from a zero state and its total
// decay; seg_pass_kernel chains them so that all segments of a long request
// run in parallel.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstddef>
#include <mutex>

#include "sm100.cuh"
#include "pdl.cuh"
#include "ssd_internal.cuh"
#include "tc_util.cuh"

namespace ssd {
namespace {
using namespace sm100;
using namespace tc;

constexpr int kMathPerRole = 8;              // G1 and G2 warps each (two per TMEM lane quadrant)
constexpr int kWarpBC = 2 + 2 * kMathPerRole;   // B/C loader warp
constexpr int kWarpZ = kWarpBC + 1;               // z loader warp
constexpr int kThreads = 32 * (kWarpZ + 1);       // x/dt producer, MMA, G1, G2, B/C loader, z loader
constexpr int kRows = 128;                   // tile rows (tokens per piece, at most)
constexpr uint64_t kWaitNs = 1000000000ull;  // bounded waits: 1 s, then abort

// Per-P layout choices.  P = 64 has room to double-buffer the x stage, the B
// and C tiles and the y accumulators and to keep the state update S in its own
// TMEM columns (z is then read by the epilogue and y staged in the x tile, which
// is what makes the second B and C tiles fit: 232,448 bytes, the limit);
// P = 128 fills shared memory and TMEM with one of each and updates the state
// in place.
template <int P>
struct TcCfg {
    static constexpr int kNS = (P == 64) ? 2 : 1;     // x stages
    static constexpr int kNY = (P == 64) ? 2 : 1;     // y_intra / y_inter accumulator pairs in TMEM
    static constexpr bool kSepS = (P == 64);          // state update in its own columns
    static constexpr bool kZTile = false;             // z read by the epilogue
    static constexpr bool kSepY = false;              // y staged in the x tile
    static constexpr int kNBC = (P == 64) ? 2 : 1;    // B and C tiles each
    // Slots of the per-piece decay values.  With y in its own tile G2 does not
    // hold the x stage, so the values G2 reads get their own deeper ring (and
    // barriers); otherwise they live and die with the x stage.
    static constexpr int kNC = kSepY ? 4 : kNS;
    static constexpr int kXBytes = kRows * P * 2;
    // TMEM columns: CB/M [0,128), then kNY pairs (y_intra, y_inter), then h^T, then S.
    __host__ __device__ static constexpr uint32_t col_yi(int yb) { return 128 + yb * 2 * P; }
    __host__ __device__ static constexpr uint32_t col_ye(int yb) { return 128 + yb * 2 * P + P; }
    static constexpr uint32_t kColH = 128 + kNY * 2 * P;
    static constexpr uint32_t kColS = kColH + P;      // only when kSepS
    static_assert(kColH + P * (kSepS ? 2 : 1) <= 512, "TMEM columns");
};

template <int P>
struct __align__(1024) TcSmem {
    using Cfg = TcCfg<P>;
    uint8_t x[Cfg::kNS * Cfg::kXBytes];  // x tiles; a finished stage also stages y for the store
    uint8_t b[Cfg::kNBC * kRows * 128 * 2];  // B tiles: 2 sub-tiles each (n 0-63, 64-127)
    uint8_t c[Cfg::kNBC * kRows * 128 * 2];  // C tiles
    uint8_t xd_hi[Cfg::kXBytes];         // w x, hi and lo parts (MN-major B operand)
    uint8_t xd_lo[Cfg::kXBytes];
    uint8_t h_hi[128 * P * 2];           // h^T (rows n, P columns), hi and lo parts
    uint8_t h_lo[128 * P * 2];
    uint8_t ystage[Cfg::kSepY ? Cfg::kXBytes : 0];           // y of the piece, for coalesced stores
    uint8_t z[Cfg::kZTile ? Cfg::kNS * Cfg::kXBytes : 16];  // last: a stub must not shift the tiles
    float cs2[Cfg::kNC][kRows];          // per slot: the piece's cumulative decay (log2 units)
    float dtp[Cfg::kNC][kRows];          // per slot: dt' (zero beyond the piece's length)
    float cslast[Cfg::kNC];              // per slot: the piece's total decay (log2 units)
    uint64_t full_x[2], empty_x[2], full_z[2], empty_z[2];
    uint64_t full_b[2], empty_b[2], full_c[2], empty_c[2];
    uint64_t full_cs[4], empty_cs[4];    // decay-value ring (kSepY only)
    uint64_t cb_full, m_full, m_done;
    uint64_t y_full[2], y_empty[2];
    uint64_t xd_full, s_free, s_full, h_full;
    uint64_t hin_bar;                    // G2's eight warps meet while building an entering state
    uint64_t hin_full;                   // the entering state's bulk copy has landed
    int32_t item_ring[8];                // work items in the order the CTA processes them (-1: none left)
    uint64_t item_full[8], item_empty[8];
    uint32_t tmem_base;
    int abort_flag;
};

// Every operand tile must start on a 1024-byte swizzle-atom boundary.
#define SSD_TILE_ALIGNED(P_, m) static_assert(offsetof(TcSmem<P_>, m) % 1024 == 0, "tile " #m " misaligned")
SSD_TILE_ALIGNED(64, b); SSD_TILE_ALIGNED(64, c); SSD_TILE_ALIGNED(64, xd_hi); SSD_TILE_ALIGNED(64, xd_lo);
SSD_TILE_ALIGNED(64, h_hi); SSD_TILE_ALIGNED(64, h_lo); SSD_TILE_ALIGNED(64, z); SSD_TILE_ALIGNED(64, ystage);
SSD_TILE_ALIGNED(128, b); SSD_TILE_ALIGNED(128, c); SSD_TILE_ALIGNED(128, xd_hi); SSD_TILE_ALIGNED(128, xd_lo);
SSD_TILE_ALIGNED(128, h_hi); SSD_TILE_ALIGNED(128, h_lo);
// the h^T tiles also take a raw (P, 128) fp32 state, as one region
static_assert(offsetof(TcSmem<64>, h_lo) == offsetof(TcSmem<64>, h_hi) + 128 * 64 * 2, "h^T tiles not adjacent");
static_assert(offsetof(TcSmem<128>, h_lo) == offsetof(TcSmem<128>, h_hi) + 128 * 128 * 2, "h^T tiles not adjacent");
static_assert(kWarpBC == 18, "G2 is warps 10-17 (its eight warps share the entering-state load)");
static_assert(sizeof(TcSmem<64>) <= 232448, "P = 64 tiles exceed the 227 KB shared-memory limit");
static_assert(sizeof(TcSmem<128>) <= 232448, "P = 128 tiles exceed the 227 KB shared-memory limit");
#undef SSD_TILE_ALIGNED

struct TcMaps {
    CUtensorMap x, b, c, z;
};

struct Item {
    int seg, head, req;
    int tok, len;
    int64_t abs0;            // absolute position of the segment's first token
    int64_t req_s, req_end;  // request's num_computed and absolute end
    bool first_seg, last_seg;
};

__device__ __forceinline__ bool load_item(const FwdParams &p, int w, bool state_only, Item &it) {
    const int nseg = p.hdr[kHdrSegs];
    const int pos = w / p.H;
    it.head = w % p.H;
    if (pos >= nseg) return false;
    it.seg = p.seg_order[pos];
    const Seg sg = p.segs[it.seg];
    it.req = sg.req;
    it.tok = sg.tok;
    it.len = sg.len;
    it.abs0 = sg.abs_start;
    it.first_seg = it.seg == p.req_first_seg[it.req];
    it.last_seg = it.seg == p.req_first_seg[it.req + 1] - 1;
    it.req_s = p.num_computed ? (int64_t)p.num_computed[it.req] : 0;
    it.req_end = it.req_s + (int64_t)p.cu_seqlens[it.req + 1] - p.cu_seqlens[it.req];
    if (state_only && it.last_seg) return false;  // the last segment's end state is never chained
    return true;
}

// Pieces of a segment: tiles of at most Qi tokens cut at absolute multiples of Qi.
struct Pieces {
    int64_t abs, end;
    int tok, Qi;
    __device__ bool next(int &t0, int &len, int64_t &abs_end) {
        if (abs >= end) return false;
        const int64_t e = min(end, (abs / Qi + 1) * (int64_t)Qi);
        t0 = tok;
        len = (int)(e - abs);
        abs_end = e;
        tok += len;
        abs = e;
        return true;
    }
};

extern __shared__ __align__(1024) uint8_t tc_smem[];


// The first wait of a launch to time out leaves where it was: header word
// kHdrTimeoutAt = 1 + the waited barrier's byte offset in shared memory, the
// next two words its block and thread.
__device__ __noinline__ void record_timeout(int32_t *hdr, int site) {
    atomicOr(hdr + kHdrErr, SSD_DEVERR_TIMEOUT);
    if (atomicCAS(hdr + kHdrTimeoutAt, 0, 1 + site) == 0) {
        hdr[kHdrTimeoutAt + 1] = (int32_t)blockIdx.x;
        hdr[kHdrTimeoutAt + 2] = (int32_t)threadIdx.x;
    }
}

__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, volatile int *abort_flag, int32_t *hdr) {
    if (*abort_flag) return false;
    if (mbar_wait(bar, parity, kWaitNs)) return true;
    *abort_flag = 1;
    record_timeout(hdr, (int)(smem_u32(bar) - smem_u32(tc_smem)));
    return false;
}

// A wait by every lane of a warp, with one outcome for the whole warp (each lane
// acquires the barrier itself; if any gave up, every lane takes the abort path).
__device__ __forceinline__ bool wait_bar_warp(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                              int32_t *hdr) {
    return __all_sync(0xffffffffu, wait_bar(bar, parity, abort_flag, hdr));
}

// A wait for the state of the previous segment (chained mode), recorded as
// site kSiteSegState when it gives up.
__device__ __forceinline__ bool wait_counter(const int32_t *counter, int target, volatile int *abort_flag,
                                             int32_t *hdr) {
    if (*abort_flag) return false;
    if (poll_counter(counter, target, kWaitNs)) return true;
    *abort_flag = 1;
    record_timeout(hdr, kSiteSegState);
    return false;
}

// ---- work items -----------------------------------------------------------
// Every role walks the same items in the same order.  The producer warp draws
// them -- in the scan from a global ticket counter, so CTAs that run faster
// take more items and neighbouring CTAs work on neighbouring (segment, head)
// items; in the state pre-pass by striding over the grid -- and publishes each
// through a ring in shared memory that the other roles read.
constexpr int kItemRing = 8;

// Producer: the next item index for this CTA (-1: none left), published.
// Only items with pieces are published (the state pre-pass has none for a
// request's last segment; an empty request's final state is written by
// seg_pass_kernel), so every published item holds a piece and a ring of 8
// covers the producer's look-ahead of two pieces: publishing item n waits for
// item n - 8, which every role reaches with inputs already issued.
template <bool STATE_ONLY, class Smem>
__device__ __forceinline__ int publish_item(Smem &s, const FwdParams &p, uint32_t n_work, uint32_t &n,
                                            uint32_t &drawn, volatile int *abort_flag) {
    int item = -1;
    while (true) {
        const uint32_t w = STATE_ONLY ? blockIdx.x + drawn++ * gridDim.x : (uint32_t)atomicAdd(p.hdr + kHdrTicket, 1);
        if (w >= n_work) break;
        Item it;
        if (load_item(p, (int)w, STATE_ONLY, it) && it.len > 0) {
            item = (int)w;
            break;
        }
    }
    const int slot = n % kItemRing;
    if (n >= (uint32_t)kItemRing && !wait_bar(&s.item_empty[slot], par(n / kItemRing - 1), abort_flag, p.hdr))
        return -2;
    s.item_ring[slot] = item;
    mbar_arrive(&s.item_full[slot]);
    ++n;
    return item;
}

// Other roles (one lane): the next item (-1: none left, -2: aborted).
template <class Smem>
__device__ __forceinline__ int take_item(Smem &s, uint32_t &n, volatile int *abort_flag, int32_t *hdr) {
    const int slot = n % kItemRing;
    if (!wait_bar(&s.item_full[slot], par(n / kItemRing), abort_flag, hdr)) return -2;
    const int item = s.item_ring[slot];
    mbar_arrive(&s.item_empty[slot]);
    ++n;
    return item;
}

// The same for a whole warp (lane 0 takes, every lane gets it).
template <class Smem>
__device__ __forceinline__ int take_item_warp(Smem &s, uint32_t &n, volatile int *abort_flag, int32_t *hdr,
                                              int lane) {
    int item = 0;
    if (lane == 0) item = take_item(s, n, abort_flag, hdr);
    return __shfl_sync(0xffffffffu, item, 0);
}

// The CTA's pieces in order across its items (used to look ahead).  One lane
// draws or takes the items; the piece fields are that lane's.
struct Cursor {
    uint32_t n, drawn;
    Item it;
    Pieces pcs;
    bool in_item, done;
};
template <bool PUBLISH, bool STATE_ONLY, class Smem>
__device__ __forceinline__ bool cursor_next(Cursor &c, Smem &s, const FwdParams &p, uint32_t n_work, int Qi,
                                            volatile int *abort_flag, int &t0, int &len, int64_t &ae) {
    while (!c.done) {
        if (c.in_item && c.pcs.next(t0, len, ae)) return true;
        c.in_item = false;
        const int w = PUBLISH ? publish_item<STATE_ONLY>(s, p, n_work, c.n, c.drawn, abort_flag)
                              : take_item(s, c.n, abort_flag, p.hdr);
        if (w < 0) {
            c.done = true;
            break;
        }
        if (!load_item(p, w, STATE_ONLY, c.it)) continue;
        c.pcs = Pieces{c.it.abs0, c.it.abs0 + c.it.len, c.it.tok, Qi};
        c.in_item = true;
    }
    return false;
}

// 16 columns (p0 .. p0+15) of state row n -> bf16 hi/lo copies of h^T row n.
template <int P>
__device__ __forceinline__ void write_h_copy16(TcSmem<P> &s, int n, int pcol0, const uint32_t (&v)[16]) {
#pragma unroll
    for (int c8 = 0; c8 < 2; ++c8) {
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
            split_pair(f2(__uint_as_float(v[c8 * 8 + 2 * e]), __uint_as_float(v[c8 * 8 + 2 * e + 1])), hi[e], lo[e]);
        const int pcol = pcol0 + c8 * 8;
        const uint32_t off = (pcol >> 6) * 16384 + sw128_off(n, (pcol & 63) >> 3);
        *reinterpret_cast<uint4 *>(s.h_hi + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4 *>(s.h_lo + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
}

// Barrier phases.  Every barrier completes once per piece of the CTA's running
// piece count pc, or once per use of a ring slot (x/z stages, decay-value
// slots, y accumulator pairs: pc / depth; work items: per item).  No waiter
// can fall two phases behind: each barrier's next phase needs an arrival that
// comes after every waiter of the current one.
//
// Per piece the MMA warp issues CB = C B^T, y_inter = C h^T (after which C is
// reloaded), the state update B^T (w x) (after which B is reloaded) and last
// y_intra = M x, which waits for the mask.  G2 reads the state out (which
// frees the state columns and the h^T copy for the next piece) before it runs
// the epilogue, so the state chain never waits for a mask or an epilogue.

template <int P, bool STATE_ONLY>
__global__ void __launch_bounds__(kThreads, 1)
ssd_chunk_tc_kernel(const FwdParams p, const __grid_constant__ TcMaps maps, int Qi) {
    using Cfg = TcCfg<P>;
    using Smem = TcSmem<P>;
    // The state-only pass is the first kernel of a forward: it waits for the plan
    // (or the previous forward) before anything else; the scan waits after its
    // shared-memory and TMEM set-up.
    if (STATE_ONLY) pdl_wait();
    // The first kernel of a forward rewinds the scan's work ticket and counts the
    // forward (the chained mode's publication counters grow by one round per forward).
    if (STATE_ONLY && blockIdx.x == 0 && threadIdx.x == 0) {
        p.hdr[kHdrTicket] = 0;
        p.hdr[kHdrEpoch] += 1;
    }
    // The tiles need 1024-byte alignment (swizzle atoms); the dynamic shared
    // window starts there on this architecture.  Refuse to run otherwise.
    // The state pre-pass has nothing to do for batches whose requests each fit
    // one segment: leave before setting up barriers and TMEM.
    if (STATE_ONLY && (p.hdr[kHdrNonFinal] == 0 || p.hdr[kHdrMode] == kModeChained)) return;
    if ((smem_u32(tc_smem) & 1023u) != 0) {
        pdl_wait();
        if (threadIdx.x == 0) atomicOr(p.hdr + kHdrErr, SSD_DEVERR_INTERNAL);
        return;
    }
    Smem &s = *reinterpret_cast<Smem *>(tc_smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int *abort_flag = &s.abort_flag;
    constexpr int kNS = Cfg::kNS, kNY = Cfg::kNY;
    constexpr int kPB = P / 64;  // 64-column blocks of P
    const size_t slot_elems = (size_t)p.H * P * 128;
    const bool z_tile = Cfg::kZTile && !STATE_ONLY && p.z != nullptr;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s.full_x[i], 2);  // TMA bytes + the producer warp's dt stores
            // x is released by the MMA that last reads it, plus G2 when it stages y in
            // the x tile (G2 then also reads the decay values of the stage)
            mbar_init(&s.empty_x[i], 1 + (Cfg::kSepY ? 0 : kMathPerRole));
            mbar_init(&s.full_z[i], 1);
            mbar_init(&s.empty_z[i], kMathPerRole);
            mbar_init(&s.y_full[i], 1);
            mbar_init(&s.y_empty[i], kMathPerRole);
        }
        for (int i = 0; i < 4; ++i) {
            mbar_init(&s.full_cs[i], 1);
            mbar_init(&s.empty_cs[i], kMathPerRole);
        }
        for (int i = 0; i < kItemRing; ++i) {
            mbar_init(&s.item_full[i], 1);
            // every role but the producer takes each item: MMA, G1 and G2 warps, loaders
            mbar_init(&s.item_empty[i], 2 + 2 * kMathPerRole + (z_tile ? 1 : 0));
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s.full_b[i], 1);
            mbar_init(&s.empty_b[i], 1);
            mbar_init(&s.full_c[i], 1);
            mbar_init(&s.empty_c[i], 1);
        }
        mbar_init(&s.cb_full, 1);
        mbar_init(&s.m_full, kMathPerRole);
        mbar_init(&s.m_done, 1);
        mbar_init(&s.xd_full, kMathPerRole);
        mbar_init(&s.s_free, kMathPerRole);
        mbar_init(&s.s_full, 1);
        mbar_init(&s.h_full, kMathPerRole);
        mbar_init(&s.hin_bar, kMathPerRole);
        mbar_init(&s.hin_full, 1);
        s.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&s.tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (!STATE_ONLY) pdl_wait();  // the segment-state passes have finished
    const uint32_t tbase = s.tmem_base;
    const uint32_t n_work = (uint32_t)p.hdr[kHdrSegs] * (uint32_t)p.H;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        // Draws the work items.  Per piece lane 0 issues the x TMA and the whole
        // warp turns the piece's 128 dt values (strided in HBM, loaded into
        // registers two pieces ahead) into dt' and the cumulative decay, which
        // it publishes beside the x tile.
        const uint16_t *__restrict__ dt16 = static_cast<const uint16_t *>(p.dt);
        if (lane == 0) prefetch_tmap(&maps.x);
        struct Ahead {
            bool have;
            int t0, len, head;
            float dtb, Ah2;
            uint16_t d[4];
        };
        Cursor cur{0, 0, Item{}, Pieces{}, false, false};
        auto next_piece = [&](Ahead &a) {
            int t0 = 0, len = 0, head = 0;
            int64_t ae = 0;
            bool have = false;
            if (lane == 0) {
                have = cursor_next<true, STATE_ONLY>(cur, s, p, n_work, Qi, abort_flag, t0, len, ae);
                head = cur.it.head;
            }
            a.have = __shfl_sync(0xffffffffu, have, 0);
            a.t0 = __shfl_sync(0xffffffffu, t0, 0);
            a.len = __shfl_sync(0xffffffffu, len, 0);
            a.head = __shfl_sync(0xffffffffu, head, 0);
            a.dtb = a.have ? p.dt_bias[a.head] : 0.f;
            a.Ah2 = a.have ? p.A[a.head] * kLog2e : 0.f;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                a.d[k] = 0;
                if (a.have && lane * 4 + k < a.len) a.d[k] = dt16[(size_t)(a.t0 + lane * 4 + k) * p.H + a.head];
            }
        };
        Ahead a0, a1, a2;
        next_piece(a0);
        next_piece(a1);
        uint32_t pc = 0;
        bool ok = true;
        const uint32_t xbytes = Cfg::kXBytes;
        while (ok && a0.have) {
            next_piece(a2);  // its dt loads stay in flight for two pieces
            const int st = pc % kNS;
            bool good = true;
            if (lane == 0 && pc >= (uint32_t)kNS) good = wait_bar(&s.empty_x[st], par(pc / kNS - 1), abort_flag, p.hdr);
            if (!__shfl_sync(0xffffffffu, good, 0)) { ok = false; break; }
            if (lane == 0) {
                mbar_arrive_expect_tx(&s.full_x[st], xbytes);
                uint8_t *xs = s.x + st * Cfg::kXBytes;
                for (int q = 0; q < kPB; ++q) tma_load_3d(xs + q * 16384, &maps.x, &s.full_x[st], q * 64, a0.head, a0.t0);
            }
            // dt' = softplus(dt + dt_bias) and its inclusive cumulative decay
            // dt' A (log2 units) over the piece; lane l holds rows 4l .. 4l+3.
            const int cslot = pc % Cfg::kNC;
            if (Cfg::kSepY && pc >= (uint32_t)Cfg::kNC) {
                bool free_ok = true;
                if (lane == 0) free_ok = wait_bar(&s.empty_cs[cslot], par(pc / Cfg::kNC - 1), abort_flag, p.hdr);
                if (!__shfl_sync(0xffffffffu, free_ok, 0)) { ok = false; break; }
            }
            float dl[4], cl[4], run = 0.f;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                dl[k] = lane * 4 + k < a0.len ? softplus_fast(__uint_as_float((uint32_t)a0.d[k] << 16) + a0.dtb) : 0.f;
                run += dl[k] * a0.Ah2;
                cl[k] = run;
            }
            float incl = run;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += v;
            }
            const float excl = incl - run;
            *reinterpret_cast<float4 *>(&s.cs2[cslot][lane * 4]) =
                make_float4(cl[0] + excl, cl[1] + excl, cl[2] + excl, cl[3] + excl);
            *reinterpret_cast<float4 *>(&s.dtp[cslot][lane * 4]) = make_float4(dl[0], dl[1], dl[2], dl[3]);
            if (lane == 31) s.cslast[cslot] = incl;
            __syncwarp();
            if (lane == 0) {
                if (Cfg::kSepY) mbar_arrive(&s.full_cs[cslot]);
                mbar_arrive(&s.full_x[st]);
            }
            a0 = a1;
            a1 = a2;
            ++pc;
        }
        // Never leave a copy in flight: wait for the last issued loads.
        if (lane == 0 && pc > 0) mbar_wait(&s.full_x[(pc - 1) % kNS], par((pc - 1) / kNS), kWaitNs);
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t sb = smem_u32(s.b), sc = smem_u32(s.c);
            const uint32_t sxh = smem_u32(s.xd_hi), sxl = smem_u32(s.xd_lo);
            const uint32_t shh = smem_u32(s.h_hi), shl = smem_u32(s.h_lo);
            constexpr uint32_t i_cb = idesc_bf16_f32(128, 128, false, false);  // C (K-major) x B^T (K-major)
            constexpr uint32_t i_y = idesc_bf16_f32(128, P, false, true);      // K-major A x MN-major B
            constexpr uint32_t i_s = idesc_bf16_f32(128, P, true, true);       // B^T (MN-major) x wx (MN-major)
            const uint32_t colS = Cfg::kSepS ? Cfg::kColS : Cfg::kColH;
            // Descriptors are built once: the start-address field is (address >> 4) in
            // the low 14 bits and shared memory ends below 256 KB, so the descriptor
            // of (tile + offset) is the tile's descriptor + offset / 16.
            const uint64_t dC = sdesc_sw128(sc, 16, 1024), dBk = sdesc_sw128(sb, 16, 1024);
            const uint64_t dBm = sdesc_sw128(sb, 16384, 1024);
            const uint64_t dHh = sdesc_sw128(shh, 16384, 1024), dHl = sdesc_sw128(shl, 16384, 1024);
            const uint64_t dXh = sdesc_sw128(sxh, 16384, 1024), dXl = sdesc_sw128(sxl, 16384, 1024);
            const uint64_t dX0 = sdesc_sw128(smem_u32(s.x), 16384, 1024);
            uint32_t pc = 0, nit = 0;
            bool ok = true;
            while (ok) {
                const int w = take_item(s, nit, abort_flag, p.hdr);
                if (w == -2) ok = false;
                if (w < 0) break;
                Item it;
                if (!load_item(p, w, STATE_ONLY, it)) continue;
                Pieces pcs{it.abs0, it.abs0 + it.len, it.tok, Qi};
                int t0, len;
                int64_t ae;
                while (pcs.next(t0, len, ae)) {
                    const int st = pc % kNS, yb = pc % kNY;
                    const uint32_t bsl = pc % Cfg::kNBC, buse = pc / Cfg::kNBC;
                    const uint32_t bo = bsl * (kRows * 128 * 2 >> 4);  // descriptor offset of the buffer
                    if (!wait_bar(&s.full_b[bsl], par(buse), abort_flag, p.hdr)) { ok = false; break; }
                    if (!STATE_ONLY && !wait_bar(&s.full_c[bsl], par(buse), abort_flag, p.hdr)) { ok = false; break; }
                    if (!STATE_ONLY) {
                        // CB = C B^T, once the previous piece's y_intra has read M out of these columns.
                        if (pc > 0 && !wait_bar(&s.m_done, par(pc - 1), abort_flag, p.hdr)) { ok = false; break; }
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {
                            const uint32_t ko = (kk >> 2) * 16384 + (kk & 3) * 32;
                            mma_ss(tbase, dC + bo + (ko >> 4), dBk + bo + (ko >> 4), i_cb, kk > 0);
                        }
                        mma_commit(&s.cb_full);
                        // y_inter = C h^T (h in hi + lo) into accumulator pair yb,
                        // once the epilogue of the piece that last used the pair is done.
                        if (!wait_bar(&s.h_full, par(pc), abort_flag, p.hdr)) { ok = false; break; }
                        if (pc >= (uint32_t)kNY && !wait_bar(&s.y_empty[yb], par(pc / kNY - 1), abort_flag, p.hdr)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
#pragma unroll
                        for (int part = 0; part < 2; ++part) {
                            const uint64_t dH = part ? dHl : dHh;
#pragma unroll
                            for (int kk = 0; kk < 8; ++kk) {
                                const uint32_t ko = (kk >> 2) * 16384 + (kk & 3) * 32;
                                mma_ss(tbase + Cfg::col_ye(yb), dC + bo + (ko >> 4), dH + kk * 128, i_y, (part | kk) != 0);
                            }
                        }
                        mma_commit(&s.empty_c[bsl]);  // C has no further reader in this piece
                    }
                    // state update: S = B^T (w x)  (or h^T += ... in place)
                    if (!wait_bar(&s.xd_full, par(pc), abort_flag, p.hdr)) { ok = false; break; }
                    if (!wait_bar(&s.s_free, par(pc), abort_flag, p.hdr)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int part = 0; part < 2; ++part) {
                        const uint64_t dXd = part ? dXl : dXh;
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            mma_ss(tbase + colS, dBm + bo + kk * 128, dXd + kk * 128, i_s,
                                   Cfg::kSepS ? (uint32_t)((part | kk) != 0) : 1u);
                    }
                    mma_commit(&s.s_full);
                    mma_commit(&s.empty_b[bsl]);  // B has no further reader in this piece
                    if (STATE_ONLY) {
                        mma_commit(&s.empty_x[st]);
                    } else {
                        // y_intra = M x with M (hi, lo) in TMEM over the CB columns:
                        // the 16 columns [16k, 16k+16) hold s in [16k, 16k+16): hi in
                        // the first 8 columns, lo in the next 8 (two bf16 per column).
                        if (!wait_bar(&s.m_full, par(pc), abort_flag, p.hdr)) { ok = false; break; }
                        if (!wait_bar(&s.full_x[st], par(pc / kNS), abort_flag, p.hdr)) { ok = false; break; }
                        tc_fence_after();
                        const uint64_t dX = dX0 + (uint32_t)(st * Cfg::kXBytes >> 4);
#pragma unroll
                        for (int part = 0; part < 2; ++part) {
#pragma unroll
                            for (int kk = 0; kk < 8; ++kk) {
                                const uint32_t acol = kk * 16 + part * 8;
                                mma_ts(tbase + Cfg::col_yi(yb), tbase + acol, dX + kk * 128, i_y, (part | kk) != 0);
                            }
                        }
                        mma_commit(&s.empty_x[st]);
                        mma_commit(&s.m_done);
                        mma_commit(&s.y_full[yb]);
                    }
                    ++pc;
                }
            }
            // Drain: every issued MMA completes before TMEM is freed.
            if (pc > 0) {
                mbar_wait(&s.s_full, par(pc - 1), kWaitNs);
                if (!STATE_ONLY) mbar_wait(&s.y_full[(pc - 1) % kNY], par((pc - 1) / kNY), kWaitNs);
            }
        }
    } else if (warp < 10) {
        // ------------------------------------------------------------ G1: w x, mask
        // Eight warps, two per TMEM lane quadrant q = warp % 4; the pair splits
        // the columns (hf).  Thread r of a pair owns tile row / TMEM lane r.
        const int q = warp & 3;
        const int hf = (warp - 2) >> 2;
        const int r = q * 32 + lane;
        const uint32_t tl = tbase + ((uint32_t)(q * 32) << 16);
        uint32_t pc = 0, nit = 0;
        bool ok = true;
        while (ok) {
            const int w = take_item_warp(s, nit, abort_flag, p.hdr, lane);
            if (w == -2) ok = false;
            if (w < 0) break;
            Item it;
            if (!load_item(p, w, STATE_ONLY, it)) continue;
            if (it.len == 0) continue;
            const int hh = it.head;
            const float Dh = (!STATE_ONLY && p.D) ? p.D[hh] : 0.f;
            Pieces pcs{it.abs0, it.abs0 + it.len, it.tok, Qi};
            int t0, len;
            int64_t ae;
            bool have_piece = pcs.next(t0, len, ae);
            while (have_piece) {
                const int st = pc % kNS;
                int nt0 = 0, nlen = 0;
                int64_t nae = 0;
                const bool has_next = pcs.next(nt0, nlen, nae);
                // ---- this piece's decay values, published by the producer with its x tile
                if (!wait_bar(&s.full_x[st], par(pc / kNS), abort_flag, p.hdr)) { ok = false; break; }
                const int cslot = pc % Cfg::kNC;
                const float *cs2v = s.cs2[cslot];
                const float *dv = s.dtp[cslot];
                const float cs2 = cs2v[r], d = dv[r], cs2_last = s.cslast[cslot];
                // the quadrant's reference row 32q - 1 (used below the diagonal only, q > 0)
                const float cs2_ref = cs2v[(32 * q + 127) & 127];
                // ---- w x (hi, lo) tiles, this warp's half of the columns; the
                // previous state MMA must have read the tiles
                if (pc > 0 && !wait_bar(&s.s_full, par(pc - 1), abort_flag, p.hdr)) { ok = false; break; }
                {
                    const float wr = (r < len) ? fast_exp2(cs2_last - cs2) * d : 0.f;
                    const uint8_t *xs = s.x + st * Cfg::kXBytes;
#pragma unroll 2
                    for (int cc = 0; cc < P / 16; ++cc) {
                        const int cb = hf * (P / 16) + cc;  // 16-byte chunk (8 columns)
                        const uint32_t off = (cb >> 3) * 16384 + sw128_off(r, cb & 7);
                        const uint4 xv = *reinterpret_cast<const uint4 *>(xs + off);
                        const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
                        uint32_t hi[4], lo[4];
                        const uint64_t wr2 = f2(wr, wr);
#pragma unroll
                        for (int e = 0; e < 4; ++e) split_pair(f2_mul(f2_bf16x2(xw[e]), wr2), hi[e], lo[e]);
                        *reinterpret_cast<uint4 *>(s.xd_hi + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                        *reinterpret_cast<uint4 *>(s.xd_lo + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                    }
                }
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s.xd_full);
                if (!STATE_ONLY) {
                    // ---- causal decayed mask M = CB o L o dt' (+ D on the diagonal),
                    // written back over CB in TMEM as bf16 hi/lo, each 16-column
                    // group in place of the CB columns it was computed from.  Below
                    // the diagonal (j < q) exp(cs_r - cs_s) = u_r v_s with both factors
                    // <= 1 around the reference row 32q - 1; the diagonal block is
                    // evaluated directly.
                    if (!wait_bar(&s.cb_full, par(pc), abort_flag, p.hdr)) { ok = false; break; }
                    tc_fence_after();
                    const float u_r = fast_exp2(cs2 - cs2_ref);
                    // 16-column group g = 2j + hf of every 32-column block j: both warps of
                    // the pair get half of the diagonal block and half of the rest.
#pragma unroll 1
                    for (int j = 0; j < 4; ++j) {
                        const uint32_t col = j * 32 + hf * 16;  // hi in [col, col+8), lo in [col+8, col+16)
                        uint32_t hi[8], lo[8];
                        if (j > q) {
#pragma unroll
                            for (int k = 0; k < 8; ++k) hi[k] = lo[k] = 0u;
                        } else if (j < q) {
                            uint32_t v[16];
                            tmem_ld16(tl + col, v);
                            const int sl = j * 32 + lane;
                            const float wl = fast_exp2(cs2_ref - cs2v[sl]) * dv[sl];
                            tmem_ld_wait();
                            const uint64_t u2 = f2(u_r, u_r);
#pragma unroll
                            for (int k = 0; k < 8; ++k) {
                                const uint64_t w2 = f2(__shfl_sync(0xffffffffu, wl, hf * 16 + 2 * k),
                                                       __shfl_sync(0xffffffffu, wl, hf * 16 + 2 * k + 1));
                                const uint64_t cb2 = f2(__uint_as_float(v[2 * k]), __uint_as_float(v[2 * k + 1]));
                                split_pair(f2_mul(f2_mul(cb2, w2), u2), hi[k], lo[k]);
                            }
                        } else {
                            uint32_t v[16];
                            tmem_ld16(tl + col, v);
                            tmem_ld_wait();
                            const uint64_t r2 = f2(cs2, cs2);
#pragma unroll
                            for (int k = 0; k < 8; ++k) {
                                const int s0 = col + 2 * k;
                                const float2 c2 = *reinterpret_cast<const float2 *>(cs2v + s0);
                                const float2 d2 = *reinterpret_cast<const float2 *>(dv + s0);
                                float e0, e1;
                                f2_get(f2_sub(r2, f2(c2.x, c2.y)), e0, e1);
                                const uint64_t cb2 = f2(__uint_as_float(v[2 * k]), __uint_as_float(v[2 * k + 1]));
                                float m0, m1;
                                f2_get(f2_mul(f2_mul(cb2, f2(fast_exp2(e0), fast_exp2(e1))), f2(d2.x, d2.y)), m0, m1);
                                m0 = (s0 < r) ? m0 : ((s0 == r) ? m0 + Dh : 0.f);
                                m1 = (s0 + 1 < r) ? m1 : ((s0 + 1 == r) ? m1 + Dh : 0.f);
                                split_pair(f2(m0, m1), hi[k], lo[k]);
                            }
                        }
                        tmem_st8(tl + col, hi);
                        tmem_st8(tl + col + 8, lo);
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&s.m_full);
                }
                ++pc;
                t0 = nt0;
                len = nlen;
                ae = nae;
                have_piece = has_next;
            }
        }
    } else if (warp < kWarpBC) {
        // ------------------------------------------------------------ G2: state, epilogue, outputs
        // Eight warps, two per quadrant; the pair splits the P columns.
        const int q = warp & 3;
        const int hf = (warp - 10) >> 2;
        const int r = q * 32 + lane;
        const uint32_t tl = tbase + ((uint32_t)(q * 32) << 16);
        constexpr int kHalf = P / 2;              // columns per warp
        const int c0 = hf * kHalf;                // first column of this warp
        const __nv_bfloat16 *__restrict__ zv = static_cast<const __nv_bfloat16 *>(p.z);
        __nv_bfloat16 *__restrict__ yv = static_cast<__nv_bfloat16 *>(p.y);
        uint32_t pc = 0, nit = 0;
        uint32_t n_hin = 0;  // entering states loaded: phases of hin_full and hin_bar
        bool ok = true;
        while (ok) {
            const int w = take_item_warp(s, nit, abort_flag, p.hdr, lane);
            if (w == -2) ok = false;
            if (w < 0) break;
            Item it;
            if (!load_item(p, w, STATE_ONLY, it)) continue;
            const int hh = it.head;
            // ---- entering state: initial slot (first segment) or the chained state;
            // src points at this head's (P, N) block.
            const size_t head_off = (size_t)hh * P * 128;
            const float *src = nullptr;
            if (!STATE_ONLY) {
                if (it.first_seg) {
                    if (p.init_slots) {
                        const int slot = p.init_slots[it.req];
                        if (slot >= p.num_slots) {
                            if (r == 0 && hf == 0) atomicOr(p.hdr + kHdrErr, SSD_DEVERR_INIT_SLOT);
                        } else if (slot >= 0) {
                            src = p.pool + (size_t)slot * slot_elems + head_off;
                        }
                    }
                } else {
                    // the state after the previous segment: chained there by seg_pass_kernel,
                    // or (chained mode) published by the CTA that ran that segment
                    const size_t prev = (size_t)(it.seg - 1 - it.req);
                    if (p.hdr[kHdrMode] == kModeChained &&
                        !__all_sync(0xffffffffu, wait_counter(p.seg_flags + prev * p.H + hh,
                                                              kMathPerRole * p.hdr[kHdrEpoch], abort_flag, p.hdr))) {
                        ok = false;
                        break;
                    }
                    src = p.seg_state + prev * slot_elems + head_off;
                }
            }
            // h^T in TMEM: thread r holds state column n = r (rows p along TMEM columns).
            if (!STATE_ONLY && src) {
                // The state (P rows of 128 floats) into the h^T tiles (hi then lo, one
                // region of P * 512 bytes) by bulk copies of 16 KB issued by one thread
                // (no registers held while they are in flight); then this warp's columns
                // into TMEM and -- once every warp has read its columns -- the hi/lo copy
                // in place.
                constexpr uint32_t kStateBytes = P * 512;
                if (warp == 10 && lane == 0) {
                    mbar_arrive_expect_tx(&s.hin_full, kStateBytes);
                    for (uint32_t off = 0; off < kStateBytes; off += 16384)
                        bulk_g2s(s.h_hi + off, reinterpret_cast<const uint8_t *>(src) + off, 16384, &s.hin_full);
                }
                if (!wait_bar_warp(&s.hin_full, par(n_hin++), abort_flag, p.hdr)) { ok = false; break; }
                const float *raw = reinterpret_cast<const float *>(s.h_hi);
#pragma unroll 1
                for (int cs = c0; cs < c0 + kHalf; cs += 16) {
                    uint32_t v[16];
#pragma unroll
                    for (int k = 0; k < 16; ++k) v[k] = __float_as_uint(raw[(size_t)(cs + k) * 128 + r]);
                    tmem_st16(tl + Cfg::kColH + cs, v);
                }
                tmem_st_wait();
                // the eight warps meet (a bounded wait: a warp that gave up earlier cannot
                // leave the others blocked)
                __syncwarp();
                if (lane == 0) mbar_arrive(&s.hin_bar);
                if (!wait_bar_warp(&s.hin_bar, par(n_hin - 1), abort_flag, p.hdr)) { ok = false; break; }
#pragma unroll 1
                for (int cs = c0; cs < c0 + kHalf; cs += 16) {
                    uint32_t v[16];
                    tmem_ld16(tl + Cfg::kColH + cs, v);
                    tmem_ld_wait();
                    write_h_copy16<P>(s, r, cs, v);
                }
            } else {
#pragma unroll 1
                for (int cs = c0; cs < c0 + kHalf; cs += 16) {
                    uint32_t v[16];
#pragma unroll
                    for (int k = 0; k < 16; ++k) v[k] = src ? __float_as_uint(src[(size_t)(cs + k) * 128 + r]) : 0u;
                    tmem_st16(tl + Cfg::kColH + cs, v);
                    if (!STATE_ONLY) write_h_copy16<P>(s, r, cs, v);
                }
            }
            tmem_st_wait();
            if (!STATE_ONLY) fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (!STATE_ONLY) mbar_arrive(&s.h_full);
                if (Cfg::kSepS) mbar_arrive(&s.s_free);  // S columns are free for the first piece
            }

            float decay_sum2 = 0.f;  // sum of dt' A log2(e) over the segment (STATE_ONLY)
            Pieces pcs{it.abs0, it.abs0 + it.len, it.tok, Qi};
            int t0, len;
            int64_t ae;
            bool have_piece = pcs.next(t0, len, ae);
            while (have_piece) {
                const int st = pc % kNS, yb = pc % kNY;
                int nt0 = 0, nlen = 0;
                int64_t nae = 0;
                const bool has_next = pcs.next(nt0, nlen, nae);
                // ---- this piece's decay values, published by the producer
                const int cslot = pc % Cfg::kNC;
                if (Cfg::kSepY) {
                    if (!wait_bar(&s.full_cs[cslot], par(pc / Cfg::kNC), abort_flag, p.hdr)) { ok = false; break; }
                } else {
                    if (!wait_bar(&s.full_x[st], par(pc / kNS), abort_flag, p.hdr)) { ok = false; break; }
                }
                const float cs2 = s.cs2[cslot][r], cs2_last = s.cslast[cslot];
                if (Cfg::kSepY) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&s.empty_cs[cslot]);
                }
                const float decay = fast_exp2(cs2_last);
                decay_sum2 += cs2_last;
                if (!Cfg::kSepS) {
                    // in-place state update: scale h^T before the state MMA adds B^T (w x)
#pragma unroll 1
                    for (int cs = c0; cs < c0 + kHalf; cs += 16) {
                        uint32_t v[16];
                        tmem_ld16(tl + Cfg::kColH + cs, v);
                        tmem_ld_wait();
#pragma unroll
                        for (int k = 0; k < 16; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * decay);
                        tmem_st16(tl + Cfg::kColH + cs, v);
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&s.s_free);
                }
                // ---- the state after the piece: read out first (it feeds the next piece)
                if (!wait_bar(&s.s_full, par(pc), abort_flag, p.hdr)) { ok = false; break; }
                tc_fence_after();
                const bool seg_end = !has_next;
                const bool req_end = (ae == it.req_end);
                float *dsts[4];
                int nd = 0;
                if (!STATE_ONLY) {
                    if (p.chunk_states && (ae % p.Q == 0 || req_end)) {
                        const int64_t row = (int64_t)p.req_first_chunk[it.req] + (ae - 1) / p.Q - it.req_s / p.Q;
                        dsts[nd++] = p.chunk_states + (size_t)row * slot_elems + head_off;
                    }
                    if (p.block_table && p.block_size > 0 && ae % p.block_size == 0) {
                        const int64_t col = ae / p.block_size - 1;
                        if (col >= p.bt_width) {
                            if (r == 0 && hf == 0) atomicOr(p.hdr + kHdrErr, SSD_DEVERR_BLOCK_TABLE);
                        } else {
                            const int bslot = p.block_table[(size_t)it.req * p.bt_width + col];
                            if (bslot >= p.num_slots) {
                                if (r == 0 && hf == 0) atomicOr(p.hdr + kHdrErr, SSD_DEVERR_BLOCK_SLOT);
                            } else if (bslot >= 0) {
                                dsts[nd++] = p.pool + (size_t)bslot * slot_elems + head_off;
                            }
                        }
                    }
                    if (req_end) {
                        if (p.final_states) dsts[nd++] = p.final_states + (size_t)it.req * slot_elems + head_off;
                        if (p.final_slots) {
                            const int fslot = p.final_slots[it.req];
                            if (fslot >= p.num_slots) {
                                if (r == 0 && hf == 0) atomicOr(p.hdr + kHdrErr, SSD_DEVERR_FINAL_SLOT);
                            } else if (fslot >= 0) {
                                dsts[nd++] = p.pool + (size_t)fslot * slot_elems + head_off;
                            }
                        }
                    }
                } else if (seg_end) {
                    dsts[nd++] = p.seg_state + (size_t)(it.seg - it.req) * slot_elems + head_off;
                    if (r == 0 && hf == 0) p.seg_decay[(size_t)(it.seg - it.req) * p.H + hh] = fast_exp2(decay_sum2);
                }
                // chained mode: the end state of a segment that is not its request's last
                // goes to the next segment through the workspace
                const bool publish = !STATE_ONLY && seg_end && !it.last_seg && p.hdr[kHdrMode] == kModeChained;
                if (publish) dsts[nd++] = p.seg_state + (size_t)(it.seg - it.req) * slot_elems + head_off;
                const bool need_copy = !STATE_ONLY && !seg_end;
                if (Cfg::kSepS || need_copy || nd > 0) {
#pragma unroll 1
                    for (int cs = c0; cs < c0 + kHalf; cs += 32) {  // two 16-column groups per TMEM wait
                        uint32_t v[2][16];
                        tmem_ld16(tl + Cfg::kColH + cs, v[0]);
                        tmem_ld16(tl + Cfg::kColH + cs + 16, v[1]);
                        if (Cfg::kSepS) {
                            uint32_t sv[2][16];
                            tmem_ld16(tl + Cfg::kColS + cs, sv[0]);
                            tmem_ld16(tl + Cfg::kColS + cs + 16, sv[1]);
                            tmem_ld_wait();
#pragma unroll
                            for (int g2 = 0; g2 < 2; ++g2) {
                                const uint64_t dec2 = f2(decay, decay);
#pragma unroll
                                for (int k = 0; k < 16; k += 2) {
                                    float a, b;
                                    f2_get(f2_fma(dec2, f2(__uint_as_float(v[g2][k]), __uint_as_float(v[g2][k + 1])),
                                                  f2(__uint_as_float(sv[g2][k]), __uint_as_float(sv[g2][k + 1]))),
                                           a, b);
                                    v[g2][k] = __float_as_uint(a);
                                    v[g2][k + 1] = __float_as_uint(b);
                                }
                                tmem_st16(tl + Cfg::kColH + cs + 16 * g2, v[g2]);
                            }
                        } else {
                            tmem_ld_wait();
                        }
#pragma unroll
                        for (int g2 = 0; g2 < 2; ++g2) {
                            for (int dd = 0; dd < nd; ++dd) {
                                float *dst = dsts[dd] + (size_t)(cs + 16 * g2) * 128 + r;
#pragma unroll
                                for (int k = 0; k < 16; ++k) dst[(size_t)k * 128] = __uint_as_float(v[g2][k]);
                            }
                            if (need_copy) write_h_copy16<P>(s, r, cs + 16 * g2, v[g2]);
                        }
                    }
                    if (Cfg::kSepS) tmem_st_wait();
                    if (need_copy) fence_async_smem();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        if (need_copy) mbar_arrive(&s.h_full);
                        if (Cfg::kSepS && has_next) mbar_arrive(&s.s_free);  // S read: next state MMA may go
                    }
                }
                if (publish) publish_warp(p.seg_flags + (size_t)(it.seg - it.req) * p.H + hh, lane);
                if (STATE_ONLY) {
                    if (!Cfg::kSepY && lane == 0) mbar_arrive(&s.empty_x[st]);
                } else {
                    // ---- epilogue: y = (y_intra + exp(cs) y_inter) * silu(z), staged
                    // in this stage's x tile, then stored with coalesced 16-byte writes.
                    if (!wait_bar(&s.y_full[yb], par(pc / kNY), abort_flag, p.hdr)) { ok = false; break; }
                    if (z_tile && !wait_bar(&s.full_z[st], par(pc / kNS), abort_flag, p.hdr)) { ok = false; break; }
                    tc_fence_after();
                    const float ecs = fast_exp2(cs2);
                    uint8_t *ys = Cfg::kSepY ? s.ystage : s.x + st * Cfg::kXBytes;
                    const uint8_t *zs = s.z + (Cfg::kZTile ? st * Cfg::kXBytes : 0);
                    const size_t yrow = ((size_t)(t0 + r) * p.H + hh) * P;
#pragma unroll 1
                    for (int cs = c0; cs < c0 + kHalf; cs += 16) {
                        uint32_t vi[16], ve[16];
                        tmem_ld16(tl + Cfg::col_yi(yb) + cs, vi);
                        tmem_ld16(tl + Cfg::col_ye(yb) + cs, ve);
                        tmem_ld_wait();
#pragma unroll
                        for (int c8 = 0; c8 < 2; ++c8) {
                            const int pcol = cs + c8 * 8;
                            const uint32_t off = (pcol >> 6) * 16384 + sw128_off(r, (pcol & 63) >> 3);
                            uint32_t zw[4] = {0u, 0u, 0u, 0u};
                            if (z_tile) {
                                const uint4 zq = *reinterpret_cast<const uint4 *>(zs + off);
                                zw[0] = zq.x; zw[1] = zq.y; zw[2] = zq.z; zw[3] = zq.w;
                            } else if (zv && r < len) {
                                const uint4 zq = *reinterpret_cast<const uint4 *>(zv + yrow + pcol);
                                zw[0] = zq.x; zw[1] = zq.y; zw[2] = zq.z; zw[3] = zq.w;
                            }
                            uint32_t out[4];
                            const uint64_t ecs2 = f2(ecs, ecs);
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int k0 = c8 * 8 + 2 * e;
                                uint64_t y2 = f2_fma(ecs2, f2(__uint_as_float(ve[k0]), __uint_as_float(ve[k0 + 1])),
                                                     f2(__uint_as_float(vi[k0]), __uint_as_float(vi[k0 + 1])));
                                if (zv) y2 = f2_mul(y2, silu2(f2_bf16x2(zw[e])));
                                float y0, y1;
                                f2_get(y2, y0, y1);
                                out[e] = pack_bf16x2(y0, y1);
                            }
                            *reinterpret_cast<uint4 *>(ys + off) = make_uint4(out[0], out[1], out[2], out[3]);
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&s.y_empty[yb]);
                        if (z_tile) mbar_arrive(&s.empty_z[st]);
                    }
                    // coalesced copy of this warp's half of its quadrant's 32 rows:
                    // lane l takes 16-byte chunk (l mod P/16) of row 32q + l / (P/16) + k (512 / P)
                    constexpr int kCh = P / 16;           // 16-byte chunks per half row
                    constexpr int kRowsPerIt = 32 / kCh;  // rows per warp-wide step
#pragma unroll 2
                    for (int it2 = 0; it2 < 32 / kRowsPerIt; ++it2) {
                        const int rr = q * 32 + it2 * kRowsPerIt + lane / kCh;
                        const int ch = hf * kCh + lane % kCh;  // 16-byte chunk within the row
                        if (rr < len) {
                            const uint4 v = *reinterpret_cast<const uint4 *>(ys + (ch >> 3) * 16384 + sw128_off(rr, ch & 7));
                            *reinterpret_cast<uint4 *>(yv + ((size_t)(t0 + rr) * p.H + hh) * P + ch * 8) = v;
                        }
                    }
                    if (!Cfg::kSepY) {
                        fence_async_smem();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&s.empty_x[st]);
                    }
                }
                ++pc;
                t0 = nt0;
                len = nlen;
                ae = nae;
                have_piece = has_next;
            }
        }
        // Never leave a copy in flight: the last entering state's bulk copy has landed.
        if (!STATE_ONLY && warp == 10 && lane == 0 && n_hin > 0) mbar_wait(&s.hin_full, par(n_hin - 1), kWaitNs);
    } else if (warp == kWarpBC) {
        // ------------------------------------------------------------ B and C loader
        if (lane == 0) {
            prefetch_tmap(&maps.b);
            if (!STATE_ONLY) prefetch_tmap(&maps.c);
            // C is released after y_inter, B after the state update: C first.
            constexpr uint32_t tbytes = kRows * 128 * 2;
            Cursor cur{0, 0, Item{}, Pieces{}, false, false};
            int t0 = 0, len = 0;
            int64_t ae = 0;
            uint32_t pc = 0;
            while (cursor_next<false, STATE_ONLY>(cur, s, p, n_work, Qi, abort_flag, t0, len, ae)) {
                const int g = cur.it.head / (p.H / p.G);
                const uint32_t bsl = pc % Cfg::kNBC, buse = pc / Cfg::kNBC;
                uint8_t *const cb = s.c + bsl * tbytes, *const bb = s.b + bsl * tbytes;
                if (!STATE_ONLY) {
                    if (buse >= 1 && !wait_bar(&s.empty_c[bsl], par(buse - 1), abort_flag, p.hdr)) break;
                    mbar_arrive_expect_tx(&s.full_c[bsl], tbytes);
                    tma_load_3d(cb, &maps.c, &s.full_c[bsl], 0, g, t0);
                    tma_load_3d(cb + 16384, &maps.c, &s.full_c[bsl], 64, g, t0);
                }
                if (buse >= 1 && !wait_bar(&s.empty_b[bsl], par(buse - 1), abort_flag, p.hdr)) break;
                mbar_arrive_expect_tx(&s.full_b[bsl], tbytes);
                tma_load_3d(bb, &maps.b, &s.full_b[bsl], 0, g, t0);
                tma_load_3d(bb + 16384, &maps.b, &s.full_b[bsl], 64, g, t0);
                ++pc;
            }
            // Never leave a copy in flight.
            for (uint32_t k = pc > (uint32_t)Cfg::kNBC ? pc - Cfg::kNBC : 0; k < pc; ++k) {
                mbar_wait(&s.full_b[k % Cfg::kNBC], par(k / Cfg::kNBC), kWaitNs);
                if (!STATE_ONLY) mbar_wait(&s.full_c[k % Cfg::kNBC], par(k / Cfg::kNBC), kWaitNs);
            }
        }
    } else {
        // ------------------------------------------------------------ z loader
        if (lane == 0 && z_tile) {
            prefetch_tmap(&maps.z);
            Cursor cur{0, 0, Item{}, Pieces{}, false, false};
            int t0 = 0, len = 0;
            int64_t ae = 0;
            uint32_t pc = 0;
            while (cursor_next<false, STATE_ONLY>(cur, s, p, n_work, Qi, abort_flag, t0, len, ae)) {
                const int st = pc % kNS;
                if (pc >= (uint32_t)kNS && !wait_bar(&s.empty_z[st], par(pc / kNS - 1), abort_flag, p.hdr)) break;
                mbar_arrive_expect_tx(&s.full_z[st], Cfg::kXBytes);
                tma_load_3d(s.z + st * Cfg::kXBytes, &maps.z, &s.full_z[st], 0, cur.it.head, t0);
                ++pc;
            }
            if (pc > 0) mbar_wait(&s.full_z[(pc - 1) % kNS], par((pc - 1) / kNS), kWaitNs);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
}

// Per (request, head, run of kSegPassChunk state elements): chains the segment
// end states of a long request, element by element (the chains are independent),
//   h <- initial state;  for every segment k but the last:
//   h <- decay_k h + S_k  and store it in slot k (= entering state of segment k+1),
// and writes an empty request's final state (its initial state).  The chain
// loads kSegPassBatch segments' states and decays before it updates and stores
// them, so a batch costs one memory round trip instead of one per segment.
constexpr int kSegPassBatch = 16;
constexpr int kSegPassThreads = 256;
constexpr int kSegPassChunk = kSegPassThreads * 4;  // one float4 per thread

template <int P>
__device__ void seg_pass_one(const FwdParams &p, int i, int hh, int chunk) {
    const int first = p.req_first_seg[i], cnt = p.req_first_seg[i + 1] - first;
    const size_t pn = (size_t)P * 128, slot_elems = (size_t)p.H * pn;
    const float *init = nullptr;
    if (p.init_slots) {
        const int slot = p.init_slots[i];
        if (slot >= 0 && slot < p.num_slots) init = p.pool + (size_t)slot * slot_elems + hh * pn;
    }
    const size_t e = (size_t)chunk * kSegPassChunk + threadIdx.x * 4;  // this thread's 4 elements
    if (p.segs[first].len == 0) {
        // An empty request: its final state is its initial state.
        const bool reporter = threadIdx.x == 0 && chunk == 0;
        if (reporter && p.init_slots && p.init_slots[i] >= p.num_slots) atomicOr(p.hdr + kHdrErr, SSD_DEVERR_INIT_SLOT);
        float *fd = p.final_states ? p.final_states + (size_t)i * slot_elems + hh * pn : nullptr;
        float *fs = nullptr;
        if (p.final_slots) {
            const int fslot = p.final_slots[i];
            if (fslot >= p.num_slots) {
                if (reporter) atomicOr(p.hdr + kHdrErr, SSD_DEVERR_FINAL_SLOT);
            } else if (fslot >= 0) {
                fs = p.pool + (size_t)fslot * slot_elems + hh * pn;
            }
        }
        const float4 v = init ? *reinterpret_cast<const float4 *>(init + e) : make_float4(0.f, 0.f, 0.f, 0.f);
        if (fd) *reinterpret_cast<float4 *>(fd + e) = v;
        if (fs) *reinterpret_cast<float4 *>(fs + e) = v;
        return;
    }
    if (cnt <= 1 || p.hdr[kHdrMode] == kModeChained) return;  // chained mode: the scan carries the states
    const int nk = cnt - 1;
    {
        float4 h = init ? *reinterpret_cast<const float4 *>(init + e) : make_float4(0.f, 0.f, 0.f, 0.f);
        for (int k0 = 0; k0 < nk; k0 += kSegPassBatch) {
            float4 sv[kSegPassBatch];
            float dk[kSegPassBatch];
#pragma unroll
            for (int j = 0; j < kSegPassBatch; ++j) {
                sv[j] = make_float4(0.f, 0.f, 0.f, 0.f);
                dk[j] = 0.f;
                if (k0 + j < nk) {
                    const size_t sg = (size_t)(first + k0 + j - i);  // compact index
                    dk[j] = p.seg_decay[sg * p.H + hh];
                    sv[j] = *reinterpret_cast<const float4 *>(p.seg_state + sg * slot_elems + hh * pn + e);
                }
            }
#pragma unroll
            for (int j = 0; j < kSegPassBatch; ++j) {
                if (k0 + j < nk) {
                    h = make_float4(fmaf(dk[j], h.x, sv[j].x), fmaf(dk[j], h.y, sv[j].y), fmaf(dk[j], h.z, sv[j].z),
                                    fmaf(dk[j], h.w, sv[j].w));
                    *reinterpret_cast<float4 *>(p.seg_state + (size_t)(first + k0 + j - i) * slot_elems + hh * pn +
                                                e) = h;
                }
            }
        }
    }
}

// A grid of at most a few CTAs per SM strides over the (request, head) pairs.
// Batches with no multi-segment and no empty request leave at once.
template <int P>
__global__ void __launch_bounds__(kSegPassThreads) seg_pass_kernel(const FwdParams p) {
    pdl_wait();  // the segment states from zero are written
    if (p.hdr[kHdrSegs] == 0) return;  // the plan rejected the batch
    if (p.hdr[kHdrEmpty] == 0 && (p.hdr[kHdrNonFinal] == 0 || p.hdr[kHdrMode] == kModeChained)) return;
    constexpr int kChunks = P * 128 / kSegPassChunk;
    const int64_t work = (int64_t)p.R * p.H * kChunks;
    for (int64_t w = blockIdx.x; w < work; w += gridDim.x) {
        const int64_t rh = w / kChunks;
        seg_pass_one<P>(p, (int)(rh / p.H), (int)(rh % p.H), (int)(w % kChunks));
    }
}

// The driver's tensor-map encoder, looked up once per process (thread-safe).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// 3-D bf16 map over a row-major (d2, d1, d0) tensor; box = 64 x 1 x 128 with the 128-byte swizzle.
bool make_map(CUtensorMap *m, const void *g, uint64_t d0, uint64_t d1, uint64_t d2) {
    auto fn = encode_fn();
    if (!fn) return false;
    const uint64_t dims[3] = {d0, d1, d2 > 0 ? d2 : 1};
    const uint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
    const uint32_t box[3] = {64, 1, (uint32_t)kRows};
    const uint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(g), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int P>
cudaError_t launch_p(const FwdParams &p, int Qi, int64_t max_items, bool pair, cudaStream_t stream) {
    const int64_t seg_ctas = (int64_t)p.R * p.H;
    if (seg_ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    TcMaps maps;
    if (!make_map(&maps.x, p.x, P, p.H, p.T) || !make_map(&maps.b, p.B, 128, p.G, p.T) ||
        !make_map(&maps.c, p.C, 128, p.G, p.T) || !make_map(&maps.z, p.z ? p.z : p.x, P, p.H, p.T))
        return cudaErrorInvalidValue;
    const int smem = (int)sizeof(TcSmem<P>);
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    // The shared-memory attribute is per device: set once on each device this
    // process uses, under a lock (host threads may launch concurrently).
    static std::mutex mu;
    static bool attr_done[64] = {};
    {
        std::lock_guard<std::mutex> lock(mu);
        const bool known = dev >= 0 && dev < 64;
        if (!known || !attr_done[dev]) {
            cudaError_t e = cudaFuncSetAttribute(ssd_chunk_tc_kernel<P, false>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e != cudaSuccess) return e;
            e = cudaFuncSetAttribute(ssd_chunk_tc_kernel<P, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     smem);
            if (e != cudaSuccess) return e;
            if (known) attr_done[dev] = true;
        }
    }
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(sms, max_items));
    // the segment states from zero: one contraction per segment where supported,
    // else this kernel's piece-by-piece state-only mode
    cudaError_t e = cudaSuccess;
    if (seg_state_supported(p)) {
        e = launch_seg_state(p, max_items, stream);
    } else {
        e = launch_after_prev(ssd_chunk_tc_kernel<P, true>, dim3(grid), dim3(kThreads), smem, stream, p, maps, Qi);
    }
    if (e != cudaSuccess) return e;
    constexpr int kPassChunks = P * 128 / kSegPassChunk;
    static_assert(P * 128 % kSegPassChunk == 0, "state elements must split into whole chunks");
    const int pass_grid =
        (int)std::max<int64_t>(1, std::min<int64_t>(seg_ctas * kPassChunks, 8LL * std::max(sms, 1)));
    e = launch_after_prev(seg_pass_kernel<P>, dim3(pass_grid), dim3(kSegPassThreads), 0, stream, p);
    if (e != cudaSuccess) return e;
    if (pair) return launch_pair_scan(p, Qi, max_items, stream);
    return launch_after_prev(ssd_chunk_tc_kernel<P, false>, dim3(grid), dim3(kThreads), smem, stream, p, maps, Qi);
}

}  // namespace

bool chunk_tc_supported(const FwdParams &p, int dtype) {
    return dtype == SSD_DTYPE_BF16 && (p.P == 64 || p.P == 128) && p.N == 128;
}

int chunk_tc_tile(const FwdParams &p) {
    int qi = kRows;
    if (p.chunk_states && p.Q < qi) qi = p.Q;
    if (p.block_table && p.block_size > 0) {
        const int low = p.block_size & -p.block_size;  // largest power of two dividing block_size
        if (low < qi) qi = low;
    }
    return qi;
}

cudaError_t launch_chunk_tc(const FwdParams &p, int64_t max_segs, cudaStream_t stream) {
    const int Qi = chunk_tc_tile(p);
    const int64_t max_items = max_segs * p.H;
    return p.P == 64 ? launch_p<64>(p, Qi, max_items, pair_supported(p), stream)
                     : launch_p<128>(p, Qi, max_items, false, stream);
}

}  // namespace ssd
