// ssd_segstate.cu -- the state pre-pass for headdim 64: the end state from zero
// of every segment that is not the last of its request, and its total decay.
//
// Unrolling h_t = exp(dt'_t A) h_{t-1} + dt'_t x_t (outer) B_t from h = 0 over a
// segment of L tokens gives
//     S = (w o x)^T B,   w_t = exp(sum_{s=t+1}^{L-1} dt'_s A) dt'_t,
//     decay = exp(sum_{s=0}^{L-1} dt'_s A),
// i.e. one contraction over the segment's tokens (K = L), with no state read out
// between pieces: the MMA accumulates piece after piece into TMEM.  Every weight
// is at most dt'_t (the exponent is a sum of non-positive terms, so nothing
// overflows), and it is built from suffix sums taken from the segment's end,
// so the weights of the last tokens -- the ones that matter -- stay exact in
// fp32 however long the segment.  w o x enters the MMA as a bf16 hi + lo pair
// (about 16 significant bits); B is exact bf16.
//
// This replaces, for P = 64, the piece-by-piece state-only mode of
// ssd_chunk_tc.cu (the same numbers: seg_state[k - i] and seg_decay of segment
// k of request i), which seg_pass_kernel then chains.
//
// Work items: (segment, pair of heads of one group) for every non-final
// segment, strided over a persistent grid.  The two heads share the B tile of
// each piece, and stack into one M = 128 contraction:
//     D[(h, p), n] = sum_t (w_h o x_h)[t, p] B[t, n],
// A = (w o x)^T written by threads into TMEM (lane = 64 h + p, two tokens per
// column), B = the B tile in shared memory, D = the two states in TMEM.
// Roles (14 warps):
//   warp 0       TMA: the two x tiles and the B tile of each 128-token piece,
//                three stages deep;
//   warp 1       MMA issuer and TMEM owner: D += A B per piece; D is
//                double-buffered across items, A across pieces;
//   warps 2-9    A (hi, lo) of each piece: two warps per TMEM lane quadrant,
//                64 tokens each;
//   warps 10-13  the weights w of the next item (512 tokens each: per-row
//                suffix scans, then a carry exchanged through shared memory),
//                and the read-out of each finished item's D.
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
constexpr int kTile = kRows * kP * 2;      // 16384: 128 rows of 64 bf16
constexpr int kMaxSeg = 2048;              // tokens of a segment, at most
constexpr int kWarps = 14;
constexpr int kThreads = kWarps * 32;
constexpr int kWarpTma = 0, kWarpMma = 1, kWarpA = 2, kWarpW = 10;
constexpr int kAW = 8;                     // A-tile warps
constexpr int kWW = 4;                     // weight / read-out warps
constexpr int kWTok = kMaxSeg / kWW;       // 512 tokens of a segment per weight warp
constexpr int kSt = 3;                     // x and B stages (the loads take microseconds to land)
constexpr uint32_t kColS = 0, kColA = 256; // TMEM: D0 | D1 | A0 | A1, 128 columns each
constexpr uint64_t kWaitNs = 1000000000ull;  // bounded waits: 1 s, then abort

struct __align__(1024) SegSmem {
    uint8_t x[kSt][2][kTile];      // x tiles of the two heads
    uint8_t b[kSt][2 * kTile];     // B tiles: n 0-63 | n 64-127 sub-tiles
    float w[2][2][kMaxSeg];        // per item (double-buffered), per head: the token weights
    float cs_total[2][2];          // per item, per head: log2 of the segment's total decay
    float wsum[2][kWW][2];         // per item: each weight warp's sum of dt' A (log2 units)
    uint64_t x_full[kSt], x_empty[kSt], b_full[kSt], b_empty[kSt], a_full[2], a_empty[2];
    uint64_t w_full[2], w_empty[2], wsum_full[2], s_full[2], s_empty[2], drain;
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(sizeof(SegSmem) <= 232448, "segment-state tiles exceed the shared-memory limit");
static_assert(offsetof(SegSmem, b) % 1024 == 0, "tiles must start on 1024-byte swizzle atoms");

struct SegMaps {
    CUtensorMap x, b;
};

extern __shared__ __align__(1024) uint8_t seg_smem[];

__device__ __noinline__ void seg_record_timeout(int32_t *hdr, int site) {
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
    seg_record_timeout(hdr, (int)(smem_u32(bar) - smem_u32(seg_smem)));
    return false;
}
__device__ __forceinline__ bool wait_bar_warp(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                              int32_t *hdr) {
    return __all_sync(0xffffffffu, wait_bar(bar, parity, abort_flag, hdr));
}

// A work item: a non-final segment and a pair of heads (2j, 2j + 1) of one group.
// Every role walks the same items: w = blockIdx.x, blockIdx.x + gridDim.x, ...
// over (segment, pair), skipping the segments that end their request.
struct Item {
    int seg, head0, req, tok, len;
};
__device__ __forceinline__ bool next_item(const FwdParams &p, uint32_t &w, uint32_t n_work, Item &it) {
    const uint32_t pairs = (uint32_t)(p.H >> 1);
    while (w < n_work) {
        const uint32_t cur = w;
        w += gridDim.x;
        const int seg = (int)(cur / pairs);
        if (seg == p.req_first_seg[p.segs[seg].req + 1] - 1) continue;  // the last segment of its request
        const Seg sg = p.segs[seg];
        it.seg = seg;
        it.head0 = 2 * (int)(cur % pairs);
        it.req = sg.req;
        it.tok = sg.tok;
        it.len = sg.len;
        return true;
    }
    return false;
}
__device__ __forceinline__ int pieces_of(int len) { return (len + kRows - 1) / kRows; }

__global__ void __launch_bounds__(kThreads, 1) seg_state_kernel(const FwdParams p, const __grid_constant__ SegMaps maps) {
    pdl_wait();  // the plan (or the previous forward) has finished
    // The first kernel of a forward rewinds the scan's work ticket and counts the
    // forward (the chained mode's publication counters grow by one round per forward).
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        p.hdr[kHdrTicket] = 0;
        p.hdr[kHdrEpoch] += 1;
    }
    // Nothing to do for batches whose requests each fit one segment, or whose
    // segment states the scan chains itself.
    if (p.hdr[kHdrNonFinal] == 0 || p.hdr[kHdrMode] == kModeChained) return;
    if ((smem_u32(seg_smem) & 1023u) != 0) {
        if (threadIdx.x == 0) atomicOr(p.hdr + kHdrErr, SSD_DEVERR_INTERNAL);
        return;
    }
    SegSmem &s = *reinterpret_cast<SegSmem *>(seg_smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int *abort_flag = &s.abort_flag;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kSt; ++i) {
            mbar_init(&s.x_full[i], 1);
            mbar_init(&s.x_empty[i], kAW);
            mbar_init(&s.b_full[i], 1);
            mbar_init(&s.b_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s.a_full[i], kAW);
            mbar_init(&s.a_empty[i], 1);
            mbar_init(&s.w_full[i], kWW);
            mbar_init(&s.w_empty[i], kAW);
            mbar_init(&s.wsum_full[i], kWW);
            mbar_init(&s.s_full[i], 1);
            mbar_init(&s.s_empty[i], kWW);
        }
        mbar_init(&s.drain, 1);
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
    const uint32_t tbase = s.tmem_base;
    const uint32_t n_work = (uint32_t)p.hdr[kHdrSegs] * (uint32_t)(p.H >> 1);
    const size_t slot_elems = (size_t)p.H * kP * 128;

    if (warp == kWarpTma) {
        // ------------------------------------------------------------ x and B tiles
        if (lane == 0) {
            prefetch_tmap(&maps.x);
            prefetch_tmap(&maps.b);
            uint32_t w = blockIdx.x, pc = 0;
            Item it;
            bool ok = true;
            while (ok && next_item(p, w, n_work, it)) {
                const int g = it.head0 / (p.H / p.G);
                for (int c = 0; c < pieces_of(it.len); ++c, ++pc) {
                    const int st = pc % kSt;
                    const int t0 = it.tok + c * kRows;
                    if (pc >= kSt && !wait_bar(&s.x_empty[st], par(pc / kSt - 1), abort_flag, p.hdr)) { ok = false; break; }
                    mbar_arrive_expect_tx(&s.x_full[st], 2 * kTile);
                    tma_load_3d(s.x[st][0], &maps.x, &s.x_full[st], 0, it.head0, t0);
                    tma_load_3d(s.x[st][1], &maps.x, &s.x_full[st], 0, it.head0 + 1, t0);
                    if (pc >= kSt && !wait_bar(&s.b_empty[st], par(pc / kSt - 1), abort_flag, p.hdr)) { ok = false; break; }
                    mbar_arrive_expect_tx(&s.b_full[st], 2 * kTile);
                    tma_load_3d(s.b[st], &maps.b, &s.b_full[st], 0, g, t0);
                    tma_load_3d(s.b[st] + kTile, &maps.b, &s.b_full[st], 64, g, t0);
                }
            }
            // Never leave a copy in flight.
            for (uint32_t k = pc > kSt ? pc - kSt : 0; k < pc; ++k) {
                mbar_wait(&s.x_full[k % kSt], par(k / kSt), kWaitNs);
                mbar_wait(&s.b_full[k % kSt], par(k / kSt), kWaitNs);
            }
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------ D += A B
        if (lane == 0) {
            constexpr uint32_t i_s = idesc_bf16_f32(128, 128, false, true);  // A (TMEM, K-major) x B (MN-major)
            // descriptor built once; + offset / 16 addresses a tile further on
            const uint64_t dB = sdesc_sw128(smem_u32(s.b[0]), kTile, 1024);
            uint32_t w = blockIdx.x, pc = 0, nitem = 0;
            Item it;
            bool ok = true;
            while (ok && next_item(p, w, n_work, it)) {
                const int sb = nitem & 1;
                const uint32_t tS = tbase + kColS + 128u * sb;
                // the read-out of the item two back has left this D buffer
                if (nitem >= 2 && !wait_bar(&s.s_empty[sb], par(nitem / 2 - 1), abort_flag, p.hdr)) { ok = false; break; }
                const int np = pieces_of(it.len);
                for (int c = 0; c < np; ++c, ++pc) {
                    const int st = pc % kSt, ab = pc & 1;
                    if (!wait_bar(&s.b_full[st], par(pc / kSt), abort_flag, p.hdr)) { ok = false; break; }
                    if (!wait_bar(&s.a_full[ab], par(pc / 2), abort_flag, p.hdr)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t bo = (uint32_t)(st * 2 * kTile) >> 4;
                    const uint32_t tA = tbase + kColA + 128u * ab;
#pragma unroll
                    for (int part = 0; part < 2; ++part) {
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            mma_ts(tS, tA + kk * 16 + part * 8, dB + bo + kk * 128, i_s, (c | part | kk) != 0);
                    }
                    mma_commit(&s.b_empty[st]);
                    mma_commit(&s.a_empty[ab]);
                    if (c == np - 1) mma_commit(&s.s_full[sb]);
                }
                ++nitem;
            }
            mma_commit(&s.drain);
            mbar_wait(&s.drain, 0, kWaitNs);
        }
    } else if (warp < kWarpW) {
        // ------------------------------------------------------------ A = (w o x)^T, hi | lo
        // Warp (quadrant q, half j) fills TMEM lanes 32 q .. 32 q + 31 (head h = q / 2 of
        // the pair, p = 32 (q % 2) + lane offset) for tokens 64 j .. 64 j + 63 of a piece:
        // per 16-token block kk, 8 hi then 8 lo columns (two tokens per column, the
        // earlier in the low half).  Per block and 16-lane half, one transposed
        // ldmatrix takes the x values straight into the 16x256b store fragment:
        // matrices 0 and 1 are the tokens {0,1,4,5,8,9,12,13} and {2,3,6,7,10,11,14,15}
        // of the block at p0 .. p0 + 7, matrices 2 and 3 the same at p0 + 8 .. p0 + 15,
        // so thread T (g = T / 4, c = T % 4) receives the token pairs 2 c and 2 c + 1
        // of lanes p0 + g and p0 + g + 8 -- the fragment's four registers.
        const int q = warp & 3;
        const int half = (warp - kWarpA) >> 2;
        const int hh = q >> 1;
        const int c4 = lane & 3;
        // this thread's ldmatrix row: matrix mi = lane / 8, row r = lane % 8
        const int mi = lane >> 3, r8 = lane & 7;
        const int row_tok = (r8 >> 1) * 4 + (r8 & 1) + ((mi & 1) ? 2 : 0);  // token within the block
        const uint32_t row_chunk = (uint32_t)((q & 1) * 4 + ((mi >> 1) ? 1 : 0));  // 16-byte chunk of p0 (+ 8)
        const uint32_t tl = (uint32_t)(q * 32) << 16;
        uint32_t w = blockIdx.x, pc = 0, nitem = 0;
        Item it;
        bool ok = true;
        while (ok && next_item(p, w, n_work, it)) {
            const int wb = nitem & 1;
            if (!wait_bar_warp(&s.w_full[wb], par(nitem / 2), abort_flag, p.hdr)) { ok = false; break; }
            const int np = pieces_of(it.len);
            for (int c = 0; c < np; ++c, ++pc) {
                const int st = pc % kSt, ab = pc & 1;
                if (!wait_bar_warp(&s.x_full[st], par(pc / kSt), abort_flag, p.hdr)) { ok = false; break; }
                if (pc >= 2 && !wait_bar_warp(&s.a_empty[ab], par(pc / 2 - 1), abort_flag, p.hdr)) { ok = false; break; }
                tc_fence_after();
                const uint32_t xs = smem_u32(s.x[st][hh]);
                // weights of this half's 64 tokens (zero past the segment's end)
                const float *wv = s.w[wb][hh] + c * kRows + half * 64;
                const uint32_t ta = tbase + tl + kColA + 128u * ab + (uint32_t)half * 64;
#pragma unroll
                for (int blk = 0; blk < 4; ++blk) {
                    const float4 w4 = *reinterpret_cast<const float4 *>(wv + blk * 16 + 4 * c4);
                    const uint64_t wa = f2(w4.x, w4.y), wb2 = f2(w4.z, w4.w);
                    const int t = half * 64 + blk * 16 + row_tok;
#pragma unroll
                    for (int sh = 0; sh < 2; ++sh) {
                        uint32_t xv[4];
                        ldmatrix_x4_trans(xs + (uint32_t)t * 128u + (((row_chunk + 2u * sh) ^ (uint32_t)(t & 7)) << 4), xv);
                        uint32_t v[8];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            split_pair(f2_mul(f2_bf16x2(xv[e]), (e & 1) ? wb2 : wa), v[e], v[4 + e]);
                        tmem_st16x256_x2(ta + ((uint32_t)(16 * sh) << 16) + blk * 16, v);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&s.x_empty[st]);
                    mbar_arrive(&s.a_full[ab]);
                }
            }
            if (!ok) break;
            // this item's weights are no longer needed
            if (lane == 0) mbar_arrive(&s.w_empty[wb]);
            ++nitem;
        }
    } else {
        // ------------------------------------------------------------ weights, read-out
        // Weight warp v takes tokens 512 v .. 512 v + 511 of the segment; lane l holds
        // tokens t = 512 v + 32 u + l (u = 0..15) of both heads.  a_t = dt'_t A log2(e);
        // w_t = 2^(-r_t) dt'_t with r_t = the sum of a_s over s > t: a suffix scan
        // across the lanes of each row u, the rows after u, and the later warps'
        // totals (exchanged through shared memory).  The total is the segment's decay.
        const int v = warp - kWarpW;
        const int q = warp & 3;  // read-out: TMEM lane quadrant
        const uint32_t *__restrict__ dt32 = static_cast<const uint32_t *>(p.dt);
        uint32_t w = blockIdx.x, nitem = 0;
        Item it, prev;
        bool ok = true;
        // read-out of item m: D (lane 64 h + p, columns n) -> seg_state[seg - req][head][p][n].
        // Each 32 x 32 block goes through shared memory (the item's weight buffer, free
        // once its last MMA has completed: 1024 floats per warp, 16-byte chunks XOR-
        // swizzled by row) so that every global store writes whole 128-byte lines.
        auto read_out = [&](const Item &pv, uint32_t m) -> bool {
            const int sb = m & 1;
            if (!wait_bar_warp(&s.s_full[sb], par(m / 2), abort_flag, p.hdr)) return false;
            tc_fence_after();
            const int h = q >> 1;
            const size_t k = (size_t)(pv.seg - pv.req);
            float *dst = p.seg_state + k * slot_elems + ((size_t)(pv.head0 + h) * kP + (q & 1) * 32) * 128;
            const uint32_t tS = tbase + ((uint32_t)(q * 32) << 16) + kColS + 128u * sb;
            float *tr = &s.w[sb][0][0] + v * 1024;
            const int rr = lane >> 3, kk = lane & 7;  // store phase: row 4 i + rr, chunk kk
#pragma unroll 1
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t r[32];
                tmem_ld32(tS + cc * 32, r);
                tmem_ld_wait();
                if (cc == 3) {
                    // D is free for the item two ahead
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&s.s_empty[sb]);
                }
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    *reinterpret_cast<uint4 *>(tr + lane * 32 + ((j ^ (lane & 7)) << 2)) =
                        make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int row = 4 * i + rr;
                    const float4 val = *reinterpret_cast<const float4 *>(tr + row * 32 + ((kk ^ (row & 7)) << 2));
                    *reinterpret_cast<float4 *>(dst + (size_t)row * 128 + cc * 32 + 4 * kk) = val;
                }
                __syncwarp();
            }
            if ((q & 1) == 0 && lane == 0) p.seg_decay[k * p.H + pv.head0 + h] = fast_exp2(s.cs_total[sb][h]);
            return true;
        };
        while (ok && next_item(p, w, n_work, it)) {
            const int wb = nitem & 1;
            if (nitem >= 2 && !wait_bar_warp(&s.w_empty[wb], par(nitem / 2 - 1), abort_flag, p.hdr)) { ok = false; break; }
            float dtb[2], Ah2[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                dtb[h] = p.dt_bias[it.head0 + h];
                Ah2[h] = p.A[it.head0 + h] * kLog2e;
            }
            // dt of both heads of a token is one 32-bit word (head0 is even, H is even)
            uint32_t dv[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int t = v * kWTok + 32 * u + lane;
                dv[u] = t < it.len ? dt32[((size_t)(it.tok + t) * p.H + it.head0) >> 1] : 0u;
            }
            // d = dt'; suf = a = d A log2(e), then its inclusive suffix sums within each row
            float d[2][16], suf[2][16];
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int t = v * kWTok + 32 * u + lane;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float raw = __uint_as_float(h ? (dv[u] & 0xffff0000u) : (dv[u] << 16));
                    d[h][u] = t < it.len ? softplus_fast(raw + dtb[h]) : 0.f;
                    suf[h][u] = d[h][u] * Ah2[h];
                }
            }
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
                for (int u = 0; u < 16; ++u) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const float y = __shfl_down_sync(0xffffffffu, suf[h][u], o);
                        if (lane + o < 32) suf[h][u] += y;
                    }
                }
            }
            // exclusive suffix sums over the warp's tokens: the rows after u (their totals
            // are lane 0's inclusive sums, added from the last row) plus the lanes after l
            float tot[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float run = 0.f;
#pragma unroll
                for (int u = 15; u >= 0; --u) {
                    const float row = __shfl_sync(0xffffffffu, suf[h][u], 0);
                    suf[h][u] = run + (suf[h][u] - d[h][u] * Ah2[h]);
                    run += row;
                }
                tot[h] = run;
            }
            if (lane == 0) {
                s.wsum[wb][v][0] = tot[0];
                s.wsum[wb][v][1] = tot[1];
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.wsum_full[wb]);
            if (!wait_bar_warp(&s.wsum_full[wb], par(nitem / 2), abort_flag, p.hdr)) { ok = false; break; }
            float later[2] = {0.f, 0.f};
#pragma unroll
            for (int h = 0; h < 2; ++h)
                for (int v2 = kWW - 1; v2 > v; --v2) later[h] += s.wsum[wb][v2][h];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float *wv = s.w[wb][h] + v * kWTok + lane;
#pragma unroll
                for (int u = 0; u < 16; ++u) wv[32 * u] = fast_exp2(later[h] + suf[h][u]) * d[h][u];
            }
            if (v == 0 && lane == 0) {
                s.cs_total[wb][0] = later[0] + tot[0];
                s.cs_total[wb][1] = later[1] + tot[1];
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.w_full[wb]);
            // the previous item's state, while this item's pieces run
            if (nitem >= 1 && !read_out(prev, nitem - 1)) { ok = false; break; }
            prev = it;
            ++nitem;
        }
        if (ok && nitem >= 1) read_out(prev, nitem - 1);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 seg_encode_fn() {
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
bool seg_map(CUtensorMap *m, const void *g, uint64_t d0, uint64_t d1, uint64_t d2) {
    auto fn = seg_encode_fn();
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

bool seg_state_supported(const FwdParams &p) {
    return p.P == kP && p.N == 128 && p.seg_len <= kMaxSeg && p.G > 0 && p.H % p.G == 0 && (p.H / p.G) % 2 == 0;
}

cudaError_t launch_seg_state(const FwdParams &p, int64_t max_items, cudaStream_t stream) {
    SegMaps maps;
    if (!seg_map(&maps.x, p.x, kP, p.H, p.T) || !seg_map(&maps.b, p.B, 128, p.G, p.T)) return cudaErrorInvalidValue;
    const int smem = (int)sizeof(SegSmem);
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    static std::mutex mu;
    static bool attr_done[64] = {};
    {
        std::lock_guard<std::mutex> lock(mu);
        const bool known = dev >= 0 && dev < 64;
        if (!known || !attr_done[dev]) {
            const cudaError_t e =
                cudaFuncSetAttribute(seg_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e != cudaSuccess) return e;
            if (known) attr_done[dev] = true;
        }
    }
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(sms, max_items));
    return launch_after_prev(seg_state_kernel, dim3(grid), dim3(kThreads), smem, stream, p, maps);
}

}  // namespace ssd
