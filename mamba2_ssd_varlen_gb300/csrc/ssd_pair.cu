// ssd_pair.cu -- the fused chunked SSD scan for headdim 64, two heads of one
// group per CTA, on Blackwell tensor cores (bf16 in, fp32 state).
//
// The same chunk decomposition as the one-head kernel (ssd_chunk_tc.cu): per
// piece of at most 128 tokens, cut at absolute multiples of the tile Qi,
//   CB      = C B^T                                   (bmm_chunk, tcgen05)
//   M[t,s]  = CB[t,s] exp(cs_t - cs_s) dt'_s, s <= t, + D on the diagonal
//   Y       = C h_prev^T, then each row scaled by exp(cs_t) in place, then
//   Y      += M x                                     (y_inter, then y_intra)
//   y       = Y * silu(z)
//   h^T     = exp(cs_last) h_prev^T  (in place)  then  h^T += B^T (w x)
// with cs measured from the piece's first valid token, so a carried or initial
// state decays from exactly that token (the initial-state decay fix of
// "[Bugfix] Mamba2 SSD varlen bug fix initstates decay", instinctive
// explanation items 1-4).  M, the carried h and w x enter the MMAs as bf16
// hi + lo pairs (about 16 significant bits); CB, x, B, C are exact bf16.
//
// Why two heads: the heads of a group share B and C, so one B/C tile load
// serves both; and each SM then runs two independent piece chains (mask ->
// y_intra -> epilogue, and state MMA -> read-out -> next y_inter), which hide
// each other's latencies.  The one-head kernel runs one such chain per SM.
//
// Roles (640 threads, 20 warps):
//   warp 0       producer: draws the work items (segment, head pair) from the
//                ticket counter, loads both heads' x tiles by TMA and computes
//                dt' and the cumulative decay of both heads (their dt values are
//                adjacent in memory: one 32-bit load per token);
//   warp 1       B and C tiles by TMA (one buffer, shared by the two heads);
//   warps 2, 3   MMA issuer of head slot 0 / 1 (warp 2 owns TMEM);
//   warps 4-11   G1 of slot 0 (4-7) / slot 1 (8-11), one warp per TMEM lane
//                quadrant: the w x split tiles, then the causal mask;
//   warps 12-19  G2 of slot 0 (12-15) / slot 1 (16-19): the state decay, the
//                y_inter row scale, the state read-out (exports, h^T copy for
//                the next piece, the z tile load) and the epilogue.
// TMEM: M0 [0,128) M1 [128,256) Y0 [256,320) Y1 [320,384) H0 [384,448)
// H1 [448,512).  Shared memory: B, C, per slot x, w x (hi, lo) and the h^T copy
// (hi, lo); once a piece's state MMA has read w x, its hi tile stages y for the
// coalesced store and its lo tile receives the z tile: 232,448 bytes in all.
// Every wait is a bounded mbarrier wait; on a timeout the CTA records
// SSD_DEVERR_TIMEOUT, drains what it issued and exits.
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

constexpr int kP = 64;
constexpr int kRows = 128;
constexpr int kTile = kRows * kP * 2;  // 16384 bytes: 128 rows of 64 bf16
constexpr int kThreads = 640;
constexpr int kWarpProd = 0, kWarpBC = 1, kWarpMma = 2, kWarpG1 = 4, kWarpG2 = 12;
constexpr int kItemRing = 8;
constexpr int kItemTakers = 2 + 8 + 8 + 1;  // MMA, G1, G2 warps and the B/C loader
#ifdef SSD_TIMEOUT_TEST
// Test build only (never the library's default build): waits give up after
// 20 ms, and when header word kHdrTestHook is set, block 0's producer publishes
// no work item, so that block's other roles time out on the item ring before
// any copy or MMA is issued while the other CTAs take all the work.
constexpr uint64_t kWaitNs = 20000000ull;
#else
constexpr uint64_t kWaitNs = 1000000000ull;  // bounded waits: 1 s, then abort
#endif
// Rows of the w x tile each G1 warp (TMEM lane quadrant 0..3) computes: the
// quadrant q mask has one diagonal block and q blocks below it, so the lower
// quadrants take more w x rows.
constexpr int kWxRows0 = 48, kWxRows1 = 36, kWxRows2 = 26, kWxRows3 = 18;
static_assert(kWxRows0 + kWxRows1 + kWxRows2 + kWxRows3 == kRows, "w x rows");

__host__ __device__ constexpr uint32_t colM(int k) { return 128u * (uint32_t)k; }
__host__ __device__ constexpr uint32_t colY(int k) { return 256u + 64u * (uint32_t)k; }
__host__ __device__ constexpr uint32_t colH(int k) { return 384u + 64u * (uint32_t)k; }

struct __align__(1024) PairSmem {
    uint8_t b[2 * kTile];    // B tile: t rows, n 0-63 | n 64-127 sub-tiles
    uint8_t c[2 * kTile];    // C tile
    uint8_t x[2][kTile];     // x tile of each slot
    uint8_t wx_hi[2][kTile]; // w x (hi) of each slot; then y staged for the store
    uint8_t wx_lo[2][kTile]; // w x (lo) of each slot; then the z tile
    uint8_t h_hi[2][kTile];  // h^T copy (n rows, p columns), hi and lo
    uint8_t h_lo[2][kTile];
    float cs2[2][kRows];     // per slot: cumulative decay of the piece (log2 units)
    float dtp[2][kRows];     // per slot: dt' (zero beyond the piece's length)
    float cslast[2];
    uint64_t x_full[2], x_empty[2], cb_full[2], m_full[2], m_done[2], wx_full[2], h_copy[2], h_scaled[2];
    uint64_t ye_done[2], y_scaled[2], y_done[2], y_empty[2], s_done[2], stage_free[2], z_full[2], drain[2];
    uint64_t bc_full, bc_empty;
    uint64_t hin_bar[2];   // per slot: G2's four warps meet while building an entering state
    uint64_t hin_full[2];  // per slot: the entering state's bulk copy has landed
    int32_t item_ring[kItemRing];
    uint64_t item_full[kItemRing], item_empty[kItemRing];
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(sizeof(PairSmem) <= 232448, "pair kernel tiles exceed the 227 KB shared-memory limit");
#define SSD_PAIR_ALIGNED(m) static_assert(offsetof(PairSmem, m) % 1024 == 0, "tile " #m " misaligned")
SSD_PAIR_ALIGNED(b); SSD_PAIR_ALIGNED(c); SSD_PAIR_ALIGNED(x); SSD_PAIR_ALIGNED(wx_hi); SSD_PAIR_ALIGNED(wx_lo);
SSD_PAIR_ALIGNED(h_hi); SSD_PAIR_ALIGNED(h_lo);
#undef SSD_PAIR_ALIGNED

struct PairMaps {
    CUtensorMap x, b, c, z;
};

// A work item: one segment (a run of at most seg_len tokens of one request)
// and one pair of heads (2 pair, 2 pair + 1) of the same group.
struct Item {
    int seg, pair, req;
    int tok, len;
    int64_t abs0;            // absolute position of the segment's first token
    int64_t req_s, req_end;  // request's num_computed and absolute end
    bool first_seg, last_seg;
};

__device__ __forceinline__ bool load_item(const FwdParams &p, int w, Item &it) {
    const int pairs = p.H >> 1;
    const int pos = w / pairs;
    it.pair = w % pairs;
    if (pos >= p.hdr[kHdrSegs]) return false;
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

extern __shared__ __align__(1024) uint8_t pair_smem[];

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
    record_timeout(hdr, (int)(smem_u32(bar) - smem_u32(pair_smem)));
    return false;
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

// A wait by every lane of a warp, with one outcome for the whole warp (each lane
// acquires the barrier itself; if any gave up, every lane takes the abort path,
// so the warp never diverges around a __syncwarp).
__device__ __forceinline__ bool wait_bar_warp(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                              int32_t *hdr) {
    return __all_sync(0xffffffffu, wait_bar(bar, parity, abort_flag, hdr));
}

// ---- work items -----------------------------------------------------------
// The producer draws items from the ticket counter (neighbouring CTAs take
// neighbouring head pairs of a segment, whose B and C tiles then come from L2)
// and publishes them through a ring in shared memory; every other role takes
// them in the same order.  Only items with tokens are published (an empty
// request's final state is written by seg_pass_kernel), so every published item
// holds a piece and a ring of 8 covers the producer's two-piece look-ahead.
__device__ __forceinline__ int publish_item(PairSmem &s, const FwdParams &p, uint32_t n_work, uint32_t &n,
                                            volatile int *abort_flag) {
    int item = -1;
    while (true) {
        const uint32_t w = (uint32_t)atomicAdd(p.hdr + kHdrTicket, 1);
        if (w >= n_work) break;
        Item it;
        if (load_item(p, (int)w, it) && it.len > 0) {
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

__device__ __forceinline__ int take_item(PairSmem &s, uint32_t &n, volatile int *abort_flag, int32_t *hdr) {
    const int slot = n % kItemRing;
    if (!wait_bar(&s.item_full[slot], par(n / kItemRing), abort_flag, hdr)) return -2;
    const int item = s.item_ring[slot];
    mbar_arrive(&s.item_empty[slot]);
    ++n;
    return item;
}

__device__ __forceinline__ int take_item_warp(PairSmem &s, uint32_t &n, volatile int *abort_flag, int32_t *hdr,
                                              int lane) {
    int item = 0;
    if (lane == 0) item = take_item(s, n, abort_flag, hdr);
    return __shfl_sync(0xffffffffu, item, 0);
}

// The CTA's pieces in order across its items (one lane draws or takes the items).
struct Cursor {
    uint32_t n;
    Item it;
    Pieces pcs;
    bool in_item, done;
};
template <bool PUBLISH>
__device__ __forceinline__ bool cursor_next(Cursor &c, PairSmem &s, const FwdParams &p, uint32_t n_work, int Qi,
                                            volatile int *abort_flag, int &t0, int &len, int64_t &ae) {
    while (!c.done) {
        if (c.in_item && c.pcs.next(t0, len, ae)) return true;
        c.in_item = false;
        const int w = PUBLISH ? publish_item(s, p, n_work, c.n, abort_flag) : take_item(s, c.n, abort_flag, p.hdr);
        if (w < 0) {
            c.done = true;
            break;
        }
        if (!load_item(p, w, c.it)) continue;
        c.pcs = Pieces{c.it.abs0, c.it.abs0 + c.it.len, c.it.tok, Qi};
        c.in_item = true;
    }
    return false;
}

// 16 columns (p0 .. p0+15) of state row n -> bf16 hi/lo copies of h^T row n.
__device__ __forceinline__ void write_h_copy16(uint8_t *hh, uint8_t *hl, int n, int pcol0, const uint32_t (&v)[16]) {
#pragma unroll
    for (int c8 = 0; c8 < 2; ++c8) {
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
            split_pair(f2(__uint_as_float(v[c8 * 8 + 2 * e]), __uint_as_float(v[c8 * 8 + 2 * e + 1])), hi[e], lo[e]);
        const uint32_t off = sw128_off(n, (pcol0 >> 3) + c8);
        *reinterpret_cast<uint4 *>(hh + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4 *>(hl + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
}

// Barrier phases: every per-slot barrier completes once per piece of the CTA's
// running piece count pc (both slots walk the same pieces), the item ring once
// per use of a slot.  Each barrier's next phase needs an arrival that comes
// after every waiter of the current one, so no waiter falls two phases behind.
//
// Per piece and slot the MMA warp issues CB (once its previous y_intra has
// read M out of the same columns), y_inter into Y (once G2 has the h^T copy
// and has read Y's previous contents), the state update onto H (once G1 has
// w x and G2 has scaled H by the piece's decay) and y_intra onto Y (once G1
// has the mask and G2 has scaled Y's rows).  G2 works through its steps in the
// order decay H, scale Y, read out H, epilogue; none waits on a later one.

__global__ void __launch_bounds__(kThreads, 1)
ssd_pair_kernel(const FwdParams p, const __grid_constant__ PairMaps maps, int Qi) {
    // The tiles need 1024-byte alignment (swizzle atoms); the dynamic shared
    // window starts there on this architecture.  Refuse to run otherwise.
    if ((smem_u32(pair_smem) & 1023u) != 0) {
        pdl_wait();
        if (threadIdx.x == 0) atomicOr(p.hdr + kHdrErr, SSD_DEVERR_INTERNAL);
        return;
    }
    PairSmem &s = *reinterpret_cast<PairSmem *>(pair_smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int *abort_flag = &s.abort_flag;
    const size_t slot_elems = (size_t)p.H * kP * 128;
    const bool has_z = p.z != nullptr;

    if (threadIdx.x == 0) {
        for (int k = 0; k < 2; ++k) {
            mbar_init(&s.x_full[k], 2);  // TMA bytes + the producer warp's decay values
            mbar_init(&s.x_empty[k], 1);
            mbar_init(&s.cb_full[k], 1);
            mbar_init(&s.m_full[k], 4);
            mbar_init(&s.m_done[k], 1);
            mbar_init(&s.wx_full[k], 4);
            mbar_init(&s.h_copy[k], 4);
            mbar_init(&s.h_scaled[k], 4);
            mbar_init(&s.ye_done[k], 1);
            mbar_init(&s.y_scaled[k], 4);
            mbar_init(&s.y_done[k], 1);
            mbar_init(&s.y_empty[k], 4);
            mbar_init(&s.s_done[k], 1);
            mbar_init(&s.stage_free[k], 4);
            mbar_init(&s.z_full[k], 1);
            mbar_init(&s.drain[k], 1);
            mbar_init(&s.hin_bar[k], 4);
            mbar_init(&s.hin_full[k], 1);
        }
        mbar_init(&s.bc_full, 1);
        mbar_init(&s.bc_empty, 2);  // each slot's state MMA is the last reader of B and C
        for (int i = 0; i < kItemRing; ++i) {
            mbar_init(&s.item_full[i], 1);
            mbar_init(&s.item_empty[i], kItemTakers);
        }
        s.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc(&s.tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_wait();  // the segment-state passes have finished
    const uint32_t tbase = s.tmem_base;
    const uint32_t n_work = (uint32_t)p.hdr[kHdrSegs] * (uint32_t)(p.H >> 1);

    if (warp == kWarpProd) {
        // ------------------------------------------------------------ producer
        // Per piece: both heads' dt (one 32-bit word per token, loaded into
        // registers two pieces ahead) -> dt' and the inclusive cumulative decay
        // dt' A (log2 units) of each head; then per slot, once its x stage is
        // free, the x tile by TMA and the decay values beside it.
        const uint32_t *__restrict__ dt32 = static_cast<const uint32_t *>(p.dt);
        const int pairs = p.H >> 1;
        if (lane == 0) prefetch_tmap(&maps.x);
        struct Ahead {
            bool have;
            int t0, len, pair;
            uint32_t d[4];
        };
        Cursor cur{0, Item{}, Pieces{}, false, false};
        auto next_piece = [&](Ahead &a) {
            int t0 = 0, len = 0, pair = 0;
            int64_t ae = 0;
            bool have = false;
            if (lane == 0) {
                have = cursor_next<true>(cur, s, p, n_work, Qi, abort_flag, t0, len, ae);
                pair = cur.it.pair;
            }
            a.have = __shfl_sync(0xffffffffu, have, 0);
            a.t0 = __shfl_sync(0xffffffffu, t0, 0);
            a.len = __shfl_sync(0xffffffffu, len, 0);
            a.pair = __shfl_sync(0xffffffffu, pair, 0);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                a.d[k] = 0;
                if (a.have && lane * 4 + k < a.len) a.d[k] = dt32[(size_t)(a.t0 + lane * 4 + k) * pairs + a.pair];
            }
        };
        Ahead a0, a1, a2;
#ifdef SSD_TIMEOUT_TEST
        if (blockIdx.x == 0 && p.hdr[kHdrTestHook] != 0) {
            a0.have = false;  // withhold every item: nothing published, nothing loaded
        } else
#endif
        {
            next_piece(a0);
            next_piece(a1);
        }
        uint32_t pc = 0, pub[2] = {0, 0};
        bool ok = true;
        while (ok && a0.have) {
            next_piece(a2);  // its dt loads stay in flight for two pieces
            float dl[2][4], cl[2][4], run[2] = {0.f, 0.f};
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int head = 2 * a0.pair + k;
                const float dtb = p.dt_bias[head], Ah2 = p.A[head] * kLog2e;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float v = k ? bf16hi_to_f32(a0.d[e]) : bf16lo_to_f32(a0.d[e]);
                    dl[k][e] = lane * 4 + e < a0.len ? softplus_fast(v + dtb) : 0.f;
                    run[k] += dl[k][e] * Ah2;
                    cl[k][e] = run[k];
                }
            }
            float incl[2] = {run[0], run[1]};
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const float v = __shfl_up_sync(0xffffffffu, incl[k], o);
                    if (lane >= o) incl[k] += v;
                }
            }
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                bool good = true;
                if (lane == 0 && pc >= 1) good = wait_bar(&s.x_empty[k], par(pc - 1), abort_flag, p.hdr);
                if (!__shfl_sync(0xffffffffu, good, 0)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(&s.x_full[k], kTile);
                    tma_load_3d(s.x[k], &maps.x, &s.x_full[k], 0, 2 * a0.pair + k, a0.t0);
                }
                const float excl = incl[k] - run[k];
                *reinterpret_cast<float4 *>(&s.cs2[k][lane * 4]) =
                    make_float4(cl[k][0] + excl, cl[k][1] + excl, cl[k][2] + excl, cl[k][3] + excl);
                *reinterpret_cast<float4 *>(&s.dtp[k][lane * 4]) = make_float4(dl[k][0], dl[k][1], dl[k][2], dl[k][3]);
                if (lane == 31) s.cslast[k] = incl[k];
                __syncwarp();
                if (lane == 0) mbar_arrive(&s.x_full[k]);
                ++pub[k];
            }
            a0 = a1;
            a1 = a2;
            ++pc;
        }
        // Never leave a copy in flight: wait for the last published loads.
        if (lane == 0)
            for (int k = 0; k < 2; ++k)
                if (pub[k] > 0) mbar_wait(&s.x_full[k], par(pub[k] - 1), kWaitNs);
    } else if (warp == kWarpBC) {
        // ------------------------------------------------------------ B and C loader
        if (lane == 0) {
            prefetch_tmap(&maps.b);
            prefetch_tmap(&maps.c);
            Cursor cur{0, Item{}, Pieces{}, false, false};
            int t0 = 0, len = 0;
            int64_t ae = 0;
            uint32_t pc = 0;
            while (cursor_next<false>(cur, s, p, n_work, Qi, abort_flag, t0, len, ae)) {
                const int g = (2 * cur.it.pair) / (p.H / p.G);
                if (pc >= 1 && !wait_bar(&s.bc_empty, par(pc - 1), abort_flag, p.hdr)) break;
                mbar_arrive_expect_tx(&s.bc_full, 4 * kTile);
                tma_load_3d(s.b, &maps.b, &s.bc_full, 0, g, t0);
                tma_load_3d(s.b + kTile, &maps.b, &s.bc_full, 64, g, t0);
                tma_load_3d(s.c, &maps.c, &s.bc_full, 0, g, t0);
                tma_load_3d(s.c + kTile, &maps.c, &s.bc_full, 64, g, t0);
                ++pc;
            }
            if (pc > 0) mbar_wait(&s.bc_full, par(pc - 1), kWaitNs);
        }
    } else if (warp < kWarpG1) {
        // ------------------------------------------------------------ MMA issuer of slot k
        const int k = warp - kWarpMma;
        if (lane == 0) {
            const uint32_t sb = smem_u32(s.b), sc = smem_u32(s.c);
            constexpr uint32_t i_cb = idesc_bf16_f32(128, 128, false, false);  // C (K-major) x B^T (K-major)
            constexpr uint32_t i_y = idesc_bf16_f32(128, kP, false, true);     // K-major A x MN-major B
            constexpr uint32_t i_s = idesc_bf16_f32(128, kP, true, true);      // B^T (MN-major) x w x (MN-major)
            // Descriptors are built once: the start-address field is (address >> 4) in
            // the low 14 bits and shared memory ends below 256 KB, so the descriptor
            // of (tile + offset) is the tile's descriptor + offset / 16.
            const uint64_t dC = sdesc_sw128(sc, 16, 1024), dBk = sdesc_sw128(sb, 16, 1024);
            const uint64_t dBm = sdesc_sw128(sb, kTile, 1024);
            const uint64_t dHh = sdesc_sw128(smem_u32(s.h_hi[k]), kTile, 1024);
            const uint64_t dHl = sdesc_sw128(smem_u32(s.h_lo[k]), kTile, 1024);
            const uint64_t dXh = sdesc_sw128(smem_u32(s.wx_hi[k]), kTile, 1024);
            const uint64_t dXl = sdesc_sw128(smem_u32(s.wx_lo[k]), kTile, 1024);
            const uint64_t dX = sdesc_sw128(smem_u32(s.x[k]), kTile, 1024);
            const uint32_t tM = tbase + colM(k), tY = tbase + colY(k), tH = tbase + colH(k);
            uint32_t pc = 0, nit = 0;
            bool ok = true;
            while (ok) {
                const int w = take_item(s, nit, abort_flag, p.hdr);
                if (w < 0) break;
                Item it;
                if (!load_item(p, w, it)) continue;
                Pieces pcs{it.abs0, it.abs0 + it.len, it.tok, Qi};
                int t0, len;
                int64_t ae;
                while (pcs.next(t0, len, ae)) {
                    // CB = C B^T into M's columns, once the previous y_intra has read them
                    if (!wait_bar(&s.bc_full, par(pc), abort_flag, p.hdr)) { ok = false; break; }
                    if (pc > 0 && !wait_bar(&s.m_done[k], par(pc - 1), abort_flag, p.hdr)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t ko = (kk >> 2) * kTile + (kk & 3) * 32;
                        mma_ss(tM, dC + (ko >> 4), dBk + (ko >> 4), i_cb, kk > 0);
                    }
                    mma_commit(&s.cb_full[k]);
                    // Y = C h^T (h in hi + lo), once the h^T copy is written and the
                    // previous epilogue has read Y
                    if (!wait_bar(&s.h_copy[k], par(pc), abort_flag, p.hdr)) { ok = false; break; }
                    if (pc > 0 && !wait_bar(&s.y_empty[k], par(pc - 1), abort_flag, p.hdr)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int part = 0; part < 2; ++part) {
                        const uint64_t dH = part ? dHl : dHh;
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {
                            const uint32_t ko = (kk >> 2) * kTile + (kk & 3) * 32;
                            mma_ss(tY, dC + (ko >> 4), dH + kk * 128, i_y, (part | kk) != 0);
                        }
                    }
                    mma_commit(&s.ye_done[k]);
                    // h^T += B^T (w x), once G1 has w x and G2 has decayed h^T
                    if (!wait_bar(&s.wx_full[k], par(pc), abort_flag, p.hdr)) { ok = false; break; }
                    if (!wait_bar(&s.h_scaled[k], par(pc), abort_flag, p.hdr)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int part = 0; part < 2; ++part) {
                        const uint64_t dXd = part ? dXl : dXh;
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) mma_ss(tH, dBm + kk * 128, dXd + kk * 128, i_s, 1u);
                    }
                    mma_commit(&s.s_done[k]);
                    mma_commit(&s.bc_empty);  // B and C have no further reader in this slot
                    // Y += M x with M (hi, lo) in TMEM over the CB columns: the 16
                    // columns [16j, 16j+16) hold s in [16j, 16j+16): hi in the first 8
                    // columns, lo in the next 8 (two bf16 per column).
                    if (!wait_bar(&s.m_full[k], par(pc), abort_flag, p.hdr)) { ok = false; break; }
                    if (!wait_bar(&s.y_scaled[k], par(pc), abort_flag, p.hdr)) { ok = false; break; }
                    if (!wait_bar(&s.x_full[k], par(pc), abort_flag, p.hdr)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int part = 0; part < 2; ++part) {
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) mma_ts(tY, tM + kk * 16 + part * 8, dX + kk * 128, i_y, 1u);
                    }
                    mma_commit(&s.y_done[k]);
                    mma_commit(&s.x_empty[k]);
                    mma_commit(&s.m_done[k]);
                    ++pc;
                }
            }
            // Drain: every issued MMA completes before TMEM is freed.
            mma_commit(&s.drain[k]);
            mbar_wait(&s.drain[k], 0, kWaitNs);
        }
    } else if (warp < kWarpG2) {
        // ------------------------------------------------------------ G1: w x, mask
        // Four warps per slot, one per TMEM lane quadrant q; thread r owns tile
        // row / TMEM lane r.
        const int k = (warp - kWarpG1) >> 2;
        const int q = warp & 3;
        const int r = q * 32 + lane;
        const uint32_t tl = tbase + ((uint32_t)(q * 32) << 16) + colM(k);
        uint8_t *const xs = s.x[k];
        uint8_t *const wxh = s.wx_hi[k];
        uint8_t *const wxl = s.wx_lo[k];
        uint32_t pc = 0, nit = 0;
        bool ok = true;
        while (ok) {
            const int w = take_item_warp(s, nit, abort_flag, p.hdr, lane);
            if (w < 0) break;
            Item it;
            if (!load_item(p, w, it)) continue;
            const int hh = 2 * it.pair + k;
            const float Dh = p.D ? p.D[hh] : 0.f;
            Pieces pcs{it.abs0, it.abs0 + it.len, it.tok, Qi};
            int t0, len;
            int64_t ae;
            while (pcs.next(t0, len, ae)) {
                // ---- this piece's decay values, published with its x tile
                if (!wait_bar_warp(&s.x_full[k], par(pc), abort_flag, p.hdr)) { ok = false; break; }
                const float *cs2v = s.cs2[k];
                const float *dv = s.dtp[k];
                const float cs2 = cs2v[r], cs2_last = s.cslast[k];
                // the quadrant's reference row 32q - 1 (used below the diagonal only, q > 0)
                const float cs2_ref = cs2v[(32 * q + 127) & 127];
                // ---- w x (hi, lo) of row r, once the last epilogue has released
                // the tiles (it staged y and z there, after the last state MMA)
                if (pc > 0 && !wait_bar_warp(&s.stage_free[k], par(pc - 1), abort_flag, p.hdr)) { ok = false; break; }
                {
                    // The rows are shared out unevenly -- the quadrants with fewer mask
                    // blocks below the diagonal take more -- so that the four warps finish
                    // w x and the mask together.  Lane l takes (row, 16-byte chunk) items
                    // l, l + 32, ... of the warp's rows.
                    const int row0 = q == 0 ? 0 : q == 1 ? kWxRows0 : q == 2 ? kWxRows0 + kWxRows1
                                                                              : kWxRows0 + kWxRows1 + kWxRows2;
                    const int nitems = 8 * (q == 0 ? kWxRows0 : q == 1 ? kWxRows1 : q == 2 ? kWxRows2 : kWxRows3);
#pragma unroll 2
                    for (int i = lane; i < nitems; i += 32) {
                        const int row = row0 + (i >> 3), cb = i & 7;
                        const float wr = row < len ? fast_exp2(cs2_last - cs2v[row]) * dv[row] : 0.f;
                        const uint64_t wr2 = f2(wr, wr);
                        const uint32_t off = sw128_off(row, cb);
                        const uint4 xv = *reinterpret_cast<const uint4 *>(xs + off);
                        const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
                        uint32_t hi[4], lo[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) split_pair(f2_mul(f2_bf16x2(xw[e]), wr2), hi[e], lo[e]);
                        *reinterpret_cast<uint4 *>(wxh + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                        *reinterpret_cast<uint4 *>(wxl + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                    }
                }
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s.wx_full[k]);
                // ---- causal decayed mask M = CB o L o dt' (+ D on the diagonal),
                // written back over CB as bf16 hi/lo, each 16-column group in place
                // of the CB columns it was computed from.  Below the diagonal
                // (block j < q) exp(cs_r - cs_s) = u_r v_s with both factors <= 1
                // around the reference row 32q - 1; the diagonal block is evaluated
                // directly; blocks above it are zero.
                if (!wait_bar_warp(&s.cb_full[k], par(pc), abort_flag, p.hdr)) { ok = false; break; }
                tc_fence_after();
                const float u_r = fast_exp2(cs2 - cs2_ref);
                const uint64_t u2 = f2(u_r, u_r);
#pragma unroll 1
                for (int j = 0; j < 4; ++j) {
                    const uint32_t col = j * 32;
                    if (j > q) {
                        uint32_t z8[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) z8[e] = 0u;
                        tmem_st8(tl + col, z8);
                        tmem_st8(tl + col + 8, z8);
                        tmem_st8(tl + col + 16, z8);
                        tmem_st8(tl + col + 24, z8);
                    } else if (j < q) {
                        uint32_t v[2][16];
                        tmem_ld16(tl + col, v[0]);
                        tmem_ld16(tl + col + 16, v[1]);
                        const int sl = j * 32 + lane;
                        const float wl = fast_exp2(cs2_ref - cs2v[sl]) * dv[sl];
                        tmem_ld_wait();
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf) {
                            uint32_t hi[8], lo[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const uint64_t w2 = f2(__shfl_sync(0xffffffffu, wl, hf * 16 + 2 * e),
                                                       __shfl_sync(0xffffffffu, wl, hf * 16 + 2 * e + 1));
                                const uint64_t cb2 =
                                    f2(__uint_as_float(v[hf][2 * e]), __uint_as_float(v[hf][2 * e + 1]));
                                split_pair(f2_mul(f2_mul(cb2, w2), u2), hi[e], lo[e]);
                            }
                            tmem_st8(tl + col + hf * 16, hi);
                            tmem_st8(tl + col + hf * 16 + 8, lo);
                        }
                    } else {
                        uint32_t v[2][16];
                        tmem_ld16(tl + col, v[0]);
                        tmem_ld16(tl + col + 16, v[1]);
                        tmem_ld_wait();
                        const uint64_t r2 = f2(cs2, cs2);
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf) {
                            uint32_t hi[8], lo[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const int s0 = col + hf * 16 + 2 * e;
                                const float2 c2 = *reinterpret_cast<const float2 *>(cs2v + s0);
                                const float2 d2 = *reinterpret_cast<const float2 *>(dv + s0);
                                float e0, e1;
                                f2_get(f2_sub(r2, f2(c2.x, c2.y)), e0, e1);
                                const uint64_t cb2 =
                                    f2(__uint_as_float(v[hf][2 * e]), __uint_as_float(v[hf][2 * e + 1]));
                                float m0, m1;
                                f2_get(f2_mul(f2_mul(cb2, f2(fast_exp2(e0), fast_exp2(e1))), f2(d2.x, d2.y)), m0, m1);
                                m0 = (s0 < r) ? m0 : ((s0 == r) ? m0 + Dh : 0.f);
                                m1 = (s0 + 1 < r) ? m1 : ((s0 + 1 == r) ? m1 + Dh : 0.f);
                                split_pair(f2(m0, m1), hi[e], lo[e]);
                            }
                            tmem_st8(tl + col + hf * 16, hi);
                            tmem_st8(tl + col + hf * 16 + 8, lo);
                        }
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s.m_full[k]);
                ++pc;
            }
        }
    } else {
        // ------------------------------------------------------------ G2: state, Y scale, read-out, epilogue
        // Four warps per slot, one per quadrant q; thread r owns TMEM lane r:
        // state column n = r of H (rows p along the columns), token row t = r of Y.
        const int k = (warp - kWarpG2) >> 2;
        const int q = warp & 3;
        const int r = q * 32 + lane;
        const uint32_t tl = tbase + ((uint32_t)(q * 32) << 16);
        const uint32_t tH = tl + colH(k), tY = tl + colY(k);
        uint8_t *const hh_t = s.h_hi[k];
        uint8_t *const hl_t = s.h_lo[k];
        uint8_t *const ys = s.wx_hi[k];  // y staging (after the state MMA)
        uint8_t *const zs = s.wx_lo[k];  // z tile (after the state MMA)
        __nv_bfloat16 *__restrict__ yv = static_cast<__nv_bfloat16 *>(p.y);
        uint32_t pc = 0, nit = 0, zissued = 0;
        uint32_t n_hin = 0;  // entering states loaded: phases of hin_full[k] and hin_bar[k]
        bool ok = true;
        while (ok) {
            const int w = take_item_warp(s, nit, abort_flag, p.hdr, lane);
            if (w < 0) break;
            Item it;
            if (!load_item(p, w, it)) continue;
            const int hh = 2 * it.pair + k;
            // ---- entering state: initial slot (first segment) or the chained state
            const size_t head_off = (size_t)hh * kP * 128;
            const float *src = nullptr;
            if (it.first_seg) {
                if (p.init_slots) {
                    const int slot = p.init_slots[it.req];
                    if (slot >= p.num_slots) {
                        if (r == 0) atomicOr(p.hdr + kHdrErr, SSD_DEVERR_INIT_SLOT);
                    } else if (slot >= 0) {
                        src = p.pool + (size_t)slot * slot_elems + head_off;
                    }
                }
            } else {
                // the state after the previous segment: chained there by seg_pass_kernel,
                // or (chained mode) published by the CTA that ran that segment
                const size_t prev = (size_t)(it.seg - 1 - it.req);
                if (p.hdr[kHdrMode] == kModeChained &&
                    !__all_sync(0xffffffffu, wait_counter(p.seg_flags + prev * p.H + hh, 4 * p.hdr[kHdrEpoch],
                                                          abort_flag, p.hdr))) {
                    ok = false;
                    break;
                }
                src = p.seg_state + prev * slot_elems + head_off;
            }
            // H in TMEM (thread r: state column n = r) and its bf16 hi/lo copy for
            // the first y_inter.  The previous item's last state MMA and y_inter
            // have completed (waited for below), so both are free.
            if (src) {
                // the state (p rows of 128 floats, 32 KB) into the h^T tiles by two bulk
                // copies (rows 0-31 to the hi tile, 32-63 to the lo tile: no registers held
                // while it is in flight); then all of it into H, and -- once every thread
                // has read its column -- the hi/lo copy in place
                if (q == 0 && lane == 0) {
                    mbar_arrive_expect_tx(&s.hin_full[k], 2 * kTile);
                    bulk_g2s(hh_t, src, kTile, &s.hin_full[k]);
                    bulk_g2s(hl_t, src + 32 * 128, kTile, &s.hin_full[k]);
                }
                const uint32_t ph = par(n_hin++);
                if (!wait_bar_warp(&s.hin_full[k], ph, abort_flag, p.hdr)) { ok = false; break; }
#pragma unroll 1
                for (int cs = 0; cs < kP; cs += 16) {
                    const float *raw = reinterpret_cast<const float *>(cs < 32 ? hh_t : hl_t) + (size_t)(cs & 31) * 128;
                    uint32_t v[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(raw[(size_t)e * 128 + r]);
                    tmem_st16(tH + cs, v);
                }
                tmem_st_wait();
                // the slot's four warps meet (a bounded wait: a warp that gave up earlier
                // cannot leave the others blocked)
                __syncwarp();
                if (lane == 0) mbar_arrive(&s.hin_bar[k]);
                if (!wait_bar_warp(&s.hin_bar[k], ph, abort_flag, p.hdr)) { ok = false; break; }
#pragma unroll 1
                for (int cs = 0; cs < kP; cs += 16) {
                    uint32_t v[16];
                    tmem_ld16(tH + cs, v);
                    tmem_ld_wait();
                    write_h_copy16(hh_t, hl_t, r, cs, v);
                }
            } else {
#pragma unroll 1
                for (int cs = 0; cs < kP; cs += 16) {
                    uint32_t v[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) v[e] = 0u;
                    tmem_st16(tH + cs, v);
                    write_h_copy16(hh_t, hl_t, r, cs, v);
                }
            }
            tmem_st_wait();
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.h_copy[k]);

            Pieces pcs{it.abs0, it.abs0 + it.len, it.tok, Qi};
            int t0, len;
            int64_t ae;
            bool have_piece = pcs.next(t0, len, ae);
            while (have_piece) {
                int nt0 = 0, nlen = 0;
                int64_t nae = 0;
                const bool has_next = pcs.next(nt0, nlen, nae);
                // ---- decay H by the piece's total decay before the state MMA adds to it
                if (!wait_bar_warp(&s.x_full[k], par(pc), abort_flag, p.hdr)) { ok = false; break; }
                const float decay = fast_exp2(s.cslast[k]);
                const float ecs = fast_exp2(s.cs2[k][r]);
#pragma unroll 1
                for (int cs = 0; cs < kP; cs += 32) {
                    uint32_t v[2][16];
                    tmem_ld16(tH + cs, v[0]);
                    tmem_ld16(tH + cs + 16, v[1]);
                    tmem_ld_wait();
#pragma unroll
                    for (int g = 0; g < 2; ++g) {
#pragma unroll
                        for (int e = 0; e < 16; ++e) v[g][e] = __float_as_uint(__uint_as_float(v[g][e]) * decay);
                        tmem_st16(tH + cs + 16 * g, v[g]);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s.h_scaled[k]);
                // ---- scale Y = C h_prev^T row t by exp(cs_t) before y_intra adds to it
                if (!wait_bar_warp(&s.ye_done[k], par(pc), abort_flag, p.hdr)) { ok = false; break; }
                tc_fence_after();
#pragma unroll 1
                for (int cs = 0; cs < kP; cs += 32) {
                    uint32_t v[2][16];
                    tmem_ld16(tY + cs, v[0]);
                    tmem_ld16(tY + cs + 16, v[1]);
                    tmem_ld_wait();
#pragma unroll
                    for (int g = 0; g < 2; ++g) {
#pragma unroll
                        for (int e = 0; e < 16; ++e) v[g][e] = __float_as_uint(__uint_as_float(v[g][e]) * ecs);
                        tmem_st16(tY + cs + 16 * g, v[g]);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s.y_scaled[k]);
                // ---- the state after the piece: exports, and the h^T copy for the next piece
                if (!wait_bar_warp(&s.s_done[k], par(pc), abort_flag, p.hdr)) { ok = false; break; }
                tc_fence_after();
                // w x has been read: the lo tile takes this piece's z
                if (has_z && q == 0 && lane == 0) {
                    mbar_arrive_expect_tx(&s.z_full[k], kTile);
                    tma_load_3d(zs, &maps.z, &s.z_full[k], 0, hh, t0);
                    ++zissued;
                }
                const bool req_end = (ae == it.req_end);
                float *dsts[5];  // chunk export, block checkpoint, two finals (or the published state)
                int nd = 0;
                if (p.chunk_states && (ae % p.Q == 0 || req_end)) {
                    const int64_t row = (int64_t)p.req_first_chunk[it.req] + (ae - 1) / p.Q - it.req_s / p.Q;
                    dsts[nd++] = p.chunk_states + (size_t)row * slot_elems + head_off;
                }
                if (p.block_table && p.block_size > 0 && ae % p.block_size == 0) {
                    const int64_t col = ae / p.block_size - 1;
                    if (col >= p.bt_width) {
                        if (r == 0) atomicOr(p.hdr + kHdrErr, SSD_DEVERR_BLOCK_TABLE);
                    } else {
                        const int bslot = p.block_table[(size_t)it.req * p.bt_width + col];
                        if (bslot >= p.num_slots) {
                            if (r == 0) atomicOr(p.hdr + kHdrErr, SSD_DEVERR_BLOCK_SLOT);
                        } else if (bslot >= 0) {
                            dsts[nd++] = p.pool + (size_t)bslot * slot_elems + head_off;
                        }
                    }
                }
                float *fdst[2];
                int nf = 0;
                if (req_end) {
                    if (p.final_states) fdst[nf++] = p.final_states + (size_t)it.req * slot_elems + head_off;
                    if (p.final_slots) {
                        const int fslot = p.final_slots[it.req];
                        if (fslot >= p.num_slots) {
                            if (r == 0) atomicOr(p.hdr + kHdrErr, SSD_DEVERR_FINAL_SLOT);
                        } else if (fslot >= 0) {
                            fdst[nf++] = p.pool + (size_t)fslot * slot_elems + head_off;
                        }
                    }
                }
                for (int f = 0; f < nf; ++f) dsts[nd++] = fdst[f];
                // chained mode: the end state of a segment that is not its request's last
                // goes to the next segment through the workspace
                const bool publish = !has_next && !it.last_seg && p.hdr[kHdrMode] == kModeChained;
                if (publish) dsts[nd++] = p.seg_state + (size_t)(it.seg - it.req) * slot_elems + head_off;
                const bool need_copy = has_next;
                if (need_copy || nd > 0) {
#pragma unroll 1
                    for (int cs = 0; cs < kP; cs += 32) {
                        uint32_t v[2][16];
                        tmem_ld16(tH + cs, v[0]);
                        tmem_ld16(tH + cs + 16, v[1]);
                        tmem_ld_wait();
#pragma unroll
                        for (int g = 0; g < 2; ++g) {
                            for (int dd = 0; dd < nd; ++dd) {
                                float *dst = dsts[dd] + (size_t)(cs + 16 * g) * 128 + r;
#pragma unroll
                                for (int e = 0; e < 16; ++e) dst[(size_t)e * 128] = __uint_as_float(v[g][e]);
                            }
                            if (need_copy) write_h_copy16(hh_t, hl_t, r, cs + 16 * g, v[g]);
                        }
                    }
                }
                if (need_copy) {
                    fence_async_smem();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&s.h_copy[k]);
                }
                if (publish) publish_warp(p.seg_flags + (size_t)(it.seg - it.req) * p.H + hh, lane);
                // ---- epilogue: y = Y * silu(z), staged in the w x hi tile, then
                // stored with coalesced 16-byte writes
                if (!wait_bar_warp(&s.y_done[k], par(pc), abort_flag, p.hdr)) { ok = false; break; }
                if (has_z && !wait_bar_warp(&s.z_full[k], par(pc), abort_flag, p.hdr)) { ok = false; break; }
                tc_fence_after();
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t vy[32];
                    tmem_ld32(tY + 32 * half, vy);
                    tmem_ld_wait();
                    if (half == 1) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&s.y_empty[k]);  // Y read: the next y_inter may go
                    }
#pragma unroll
                    for (int c8 = 0; c8 < 4; ++c8) {
                        const uint32_t off = sw128_off(r, half * 4 + c8);
                        uint32_t zw[4] = {0u, 0u, 0u, 0u};
                        if (has_z) {
                            const uint4 zq = *reinterpret_cast<const uint4 *>(zs + off);
                            zw[0] = zq.x; zw[1] = zq.y; zw[2] = zq.z; zw[3] = zq.w;
                        }
                        uint32_t out[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int k0 = c8 * 8 + 2 * e;
                            uint64_t y2 = f2(__uint_as_float(vy[k0]), __uint_as_float(vy[k0 + 1]));
                            if (has_z) y2 = f2_mul(y2, silu2(f2_bf16x2(zw[e])));
                            float y0, y1;
                            f2_get(y2, y0, y1);
                            out[e] = pack_bf16x2(y0, y1);
                        }
                        *reinterpret_cast<uint4 *>(ys + off) = make_uint4(out[0], out[1], out[2], out[3]);
                    }
                }
                // coalesced copy of the quadrant's 32 rows: lane l takes 16-byte chunk
                // l % 8 of row 32q + 4 i + l / 8 (all eight loads first, then the stores)
                __syncwarp();
                {
                    uint4 v[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        v[i] = *reinterpret_cast<const uint4 *>(ys + sw128_off(q * 32 + i * 4 + (lane >> 3), lane & 7));
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int rr = q * 32 + i * 4 + (lane >> 3);
                        if (rr < len)
                            *reinterpret_cast<uint4 *>(yv + ((size_t)(t0 + rr) * p.H + hh) * kP + (lane & 7) * 8) = v[i];
                    }
                }
                // the tiles go back to G1 (and, for a later piece, to the z load)
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s.stage_free[k]);
                ++pc;
                t0 = nt0;
                len = nlen;
                ae = nae;
                have_piece = has_next;
            }
            // Before the next item rewrites H and the h^T copy: the last state MMA
            // (waited for above) and the last y_inter (waited for in the Y scale)
            // have completed.
        }
        // Never leave a copy in flight: the last z load has landed (waited for in its
        // epilogue unless a wait gave up first).
        if (zissued > 0) mbar_wait(&s.z_full[k], par(zissued - 1), kWaitNs);
        if (q == 0 && lane == 0 && n_hin > 0) mbar_wait(&s.hin_full[k], par(n_hin - 1), kWaitNs);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 pair_encode_fn() {
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
bool pair_map(CUtensorMap *m, const void *g, uint64_t d0, uint64_t d1, uint64_t d2) {
    auto fn = pair_encode_fn();
    if (!fn) return false;
    const uint64_t dims[3] = {d0, d1, d2 > 0 ? d2 : 1};
    const uint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
    const uint32_t box[3] = {64, 1, (uint32_t)kRows};
    const uint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(g), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool pair_supported(const FwdParams &p) { return p.P == kP && p.N == 128 && (p.H / p.G) % 2 == 0; }

cudaError_t launch_pair_scan(const FwdParams &p, int Qi, int64_t max_items, cudaStream_t stream) {
    PairMaps maps;
    if (!pair_map(&maps.x, p.x, kP, p.H, p.T) || !pair_map(&maps.b, p.B, 128, p.G, p.T) ||
        !pair_map(&maps.c, p.C, 128, p.G, p.T) || !pair_map(&maps.z, p.z ? p.z : p.x, kP, p.H, p.T))
        return cudaErrorInvalidValue;
    const int smem = (int)sizeof(PairSmem);
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
            const cudaError_t e =
                cudaFuncSetAttribute(ssd_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e != cudaSuccess) return e;
            if (known) attr_done[dev] = true;
        }
    }
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(sms, max_items / 2));
    return launch_after_prev(ssd_pair_kernel, dim3(grid), dim3(kThreads), smem, stream, p, maps, Qi);
}

}  // namespace ssd
