// ssd_gdn_tc.cu -- the gated delta rule (GDN) chunked prefill on the tcgen05
// tensor cores, for key and value head dims K = V = 128 ("Automatic prefix
// caching for GDN hybrid models (mamba_cache_mode=all) with MTP speculative
// decoding", Purpose, Kernels/layers: the chunk kernel with intermediate-state
// export and the block-aligned checkpoint scatter).
//
// The rule per value head (published gated delta rule; S a K x V matrix):
//     S <- e^{g_t} S;  u = beta_t (v_t - S^T k_t);  S <- S + k_t u^T;  o_t = scale S^T q_t
// with k, q optionally l2-normalised (row factors rk, rq).  Per chunk of L = 64
// tokens from the state S0, with G the in-chunk prefix sums of g, gamma = e^G:
//     A[s,r] = beta_s rk_s rk_r e^{G_s - G_r} k_s.k_r   (r < s)
//     T = (I + A)^-1                                    (unit lower triangular)
//     R = diag(beta) (V - diag(gamma rk) K S0),   U = T R
//     O = diag(scale gamma rq) Q S0 + P U,   P[t,s] = scale rq_t rk_s e^{G_t - G_s} q_t.k_s  (s <= t)
//     S = gamma_L S0 + K^T diag(rk e^{G_L - G}) U
// The state-independent part of a chunk (its tiles, gates, l2 factors, A, P
// and T) is prepared one chunk ahead of the state chain, whose products all run
// on the tensor cores with their accumulators in TMEM:
//     [K;Q] [K]^T -> [KK^T ; QK^T]   (M = 128: the 64 k rows over the 64 q rows)
//     S0^T K^T    -> (K S0)^T        (S0 as bf16 hi + lo; value columns on the TMEM lanes)
//     [K;Q] S0    -> [K S0 ; Q S0]   (only the Q S0 rows are used: the output)
//     U^T = R^T T^T                  (R^T hi/lo formed in TMEM over (K S0)^T, T hi/lo:
//                                     hi.hi + hi.lo + lo.hi)
//     S  += K^T U'                   (U' = diag(rk e^{G_L - G}) U as hi + lo; S pre-scaled by gamma_L)
//     O  += P U                      (onto the Q S0 rows scaled by scale gamma rq; P hi/lo in TMEM)
// q, k, v enter exactly (bf16); every fp32 operand is split into a bf16 high part
// and a bf16 remainder, about 16 significant bits.  T comes from A in fp32 by
// 32 x 32 blocks (substitution for the diagonal blocks, products for the other).
//
// One CTA per (request, value head); roles:
//   warp 0      TMA: the K and Q tiles of each chunk (two buffers), the V tile;
//   warp 1      MMA issuer and TMEM owner;
//   warps 2, 3  the output rows (TMEM lane quadrants 2 and 3): the Q S0 rows
//               scaled, then O -> bf16;
//   warps 4-7   the state chain: S read-out (state outputs, S0 hi/lo, gamma_L S),
//               R^T (one value column per thread), U and U' hi/lo;
//   warps 8-11  the next chunk: gates and their prefix sums, l2 factors, A
//               (to shared memory) and P (hi/lo in place in TMEM), then T by 32 x 32
//               blocks: the two diagonal blocks by right-looking substitutions in
//               parallel, the off-diagonal one by two small products.
// Every wait is a bounded mbarrier wait; on a timeout the CTA records
// SSD_DEVERR_TIMEOUT in the call's device error word, drains and exits.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstddef>
#include <cstring>
#include <mutex>

#include "sm100.cuh"
#include "pdl.cuh"
#include "ssd_internal.cuh"
#include "tc_util.cuh"

namespace ssd {
namespace {
using namespace sm100;
using namespace tc;

constexpr int kL = 64;    // chunk length
constexpr int kK = 128;   // key head dim
constexpr int kV = 128;   // value head dim
constexpr int kThreads = 12 * 32;
constexpr int kWarpTma = 0, kWarpMma = 1, kWarpOut = 2, kWarpChain = 4, kWarpPrep = 8;
constexpr int kLdA = kL + 4;  // fp32 row stride of A (float4 rows, conflict-free)
constexpr uint64_t kWaitNs = 1000000000ull;
// TMEM columns: S (128) | [K S0 ; Q S0] then O (128) | [KK^T ; QK^T] / P, two buffers (2 x 64) | U^T (64)
// | (K S0)^T, then R^T hi/lo in place (64)
constexpr uint32_t kColS = 0, kColKQ = 128, kColAP = 256, kColU = 384, kColKT = 448;

struct GdnTcParams {
    int64_t T;
    int32_t R, Hk, Hv, bs, btw, num_slots, l2norm;
    float scale;
    const int32_t *cu;
    ssd_gdn_io io;
};

struct GdnTcMaps {
    CUtensorMap q, k, v;
};

// Per chunk: gate prefix sums (log2 units), write strengths, l2 factors (zero past the
// chunk's tokens), and what the state chain takes from them: gamma rk (R), scale gamma
// rq (the Q S0 rows), rk e^{G_L - G} (U') and gamma_L.
struct GdnVec {
    float gl2[kL], beta[kL], rk[kL], rq[kL];
    float grk[kL], osc[kL], wu[kL];
    float wb[kL];  // rk_r e^{G_b - G_r}, b = the last row of r's 16-row block (the masks' column factor)
    float gL, pad[3];
};

struct __align__(1024) GdnTcSmem {
    uint8_t kq[2][32768];  // per chunk: k-half h at h*16384: 64 K rows (8 KB) then 64 Q rows (8 KB)
    uint8_t s0[65536];     // S0 hi | lo [v-half][128 k rows][64 v]; then U' hi | lo [128 v rows][64 t]
    uint8_t r[32768];      // U hi | lo [128 v rows][64 s]
    uint8_t v[16384];      // V tile [v-half][64 t rows][64 v]
    uint8_t t[16384];      // T^T hi | lo [64 s rows][64 t]
    float a[kL * kLdA];    // A^T (row c = column c of A), fp32; rows 32..63, columns 0..31: T22^T
    float t11[32 * 33], m1[32 * 33], t21[32 * 33];  // blocks of T = (I + A)^-1, column-major
    GdnVec vec[2];
    uint64_t kq_full[2], kq_empty[2], ap_full[2], p_ready[2], vec_ready[2], vec2_ready[2], vec_free[2];
    uint64_t v_full, v_empty, a_ready, inv1, inv2, inv3, t_ready, t_free, s0_copy, kt_full, kqs0_full, r_ready, o_scaled,
        u_full, u_copy, s_ready, o_full, o_free, drain;
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(sizeof(GdnTcSmem) <= 232448, "GDN tiles exceed the shared-memory limit");

extern __shared__ __align__(1024) uint8_t gdn_tc_smem[];

__device__ __noinline__ void gdn_record_timeout(int32_t *err) { atomicOr(err, SSD_DEVERR_TIMEOUT); }

__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, volatile int *abort_flag, int32_t *err) {
    if (*abort_flag) return false;
    if (mbar_wait(bar, parity, kWaitNs)) return true;
    *abort_flag = 1;
    gdn_record_timeout(err);
    return false;
}
__device__ __forceinline__ bool wait_bar_warp(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                              int32_t *err) {
    return __all_sync(0xffffffffu, wait_bar(bar, parity, abort_flag, err));
}

// The chunks of a request: cut at absolute multiples of kL (positions from s0).
struct Chunks {
    int64_t a, len, s0, pos;
    __device__ __forceinline__ bool next(int64_t &t0, int &n, int64_t &abs_end) {
        if (pos >= len) return false;
        const int64_t abs0 = s0 + pos;
        n = (int)min((abs0 / kL + 1) * kL - abs0, len - pos);
        t0 = a + pos;
        abs_end = abs0 + n;
        pos += n;
        return true;
    }
};

// Where the state after a chunk ending at absolute position abs_end goes (export
// row, block checkpoint), or the final destinations; at most four.
struct Dests {
    float *d[4];
    int n;
};

__global__ void __launch_bounds__(kThreads, 1) gdn_tc_kernel(const __grid_constant__ GdnTcParams p,
                                                             const __grid_constant__ GdnTcMaps maps) {
    pdl_wait();  // a dependent launch: the stream's previous kernel has finished
    const ssd_gdn_io &io = p.io;
    int32_t *err = io.device_err;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int i = (int)(blockIdx.x / p.Hv), hv = (int)(blockIdx.x % p.Hv);
    const int kh = hv / (p.Hv / p.Hk);
    const size_t state_elems = (size_t)kK * kV;

    if (blockIdx.x == 0 && tid == 0 && (p.cu[0] != 0 || (int64_t)p.cu[p.R] != p.T)) atomicOr(err, SSD_DEVERR_CU_SEQLENS);
    const int64_t a = p.cu[i], b = p.cu[i + 1];
    if (a < 0 || b < a || b > p.T) {
        if (tid == 0) atomicOr(err, SSD_DEVERR_CU_SEQLENS);
        return;
    }
    int64_t s0 = io.num_computed ? io.num_computed[i] : 0;
    if (s0 < 0 || s0 + (b - a) > 0x7fffffffLL) {
        if (tid == 0) atomicOr(err, SSD_DEVERR_NUM_COMPUTED);
        s0 = 0;
    }
    const float *init = nullptr;
    if (io.init_slots && io.state_pool) {
        const int sl = io.init_slots[i];
        if (sl >= p.num_slots) {
            if (tid == 0) atomicOr(err, SSD_DEVERR_INIT_SLOT);
        } else if (sl >= 0) {
            init = io.state_pool + ((size_t)sl * p.Hv + hv) * state_elems;
        }
    }
    // final destinations (every CTA of the request checks the slot; thread 0 reports)
    Dests fin{{nullptr, nullptr, nullptr, nullptr}, 0};
    if (io.final_states) fin.d[fin.n++] = io.final_states + ((size_t)i * p.Hv + hv) * state_elems;
    if (io.final_slots && io.state_pool) {
        const int fs = io.final_slots[i];
        if (fs >= p.num_slots) {
            if (tid == 0) atomicOr(err, SSD_DEVERR_FINAL_SLOT);
        } else if (fs >= 0) {
            fin.d[fin.n++] = io.state_pool + ((size_t)fs * p.Hv + hv) * state_elems;
        }
    }
    if (b == a) {
        // An empty request: its final state is its initial state.
        for (size_t e = (size_t)tid * 4; e < state_elems; e += kThreads * 4) {
            const float4 val = init ? *reinterpret_cast<const float4 *>(init + e) : make_float4(0.f, 0.f, 0.f, 0.f);
            for (int f = 0; f < fin.n; ++f) *reinterpret_cast<float4 *>(fin.d[f] + e) = val;
        }
        return;
    }
    const int nch = (int)((s0 + (b - a) - 1) / kL - s0 / kL + 1);

    if ((smem_u32(gdn_tc_smem) & 1023u) != 0) {
        if (tid == 0) atomicOr(err, SSD_DEVERR_INTERNAL);
        return;
    }
    GdnTcSmem &s = *reinterpret_cast<GdnTcSmem *>(gdn_tc_smem);
    volatile int *abort_flag = &s.abort_flag;
    if (tid == 0) {
        for (int k = 0; k < 2; ++k) {
            mbar_init(&s.kq_full[k], 1);
            mbar_init(&s.kq_empty[k], 1);
            mbar_init(&s.ap_full[k], 1);
            mbar_init(&s.p_ready[k], 4);
            mbar_init(&s.vec_ready[k], 4);
            mbar_init(&s.vec2_ready[k], 4);
            mbar_init(&s.vec_free[k], 6);
        }
        mbar_init(&s.v_full, 1);
        mbar_init(&s.v_empty, 4);
        mbar_init(&s.a_ready, 2);
        mbar_init(&s.inv1, 2);
        mbar_init(&s.inv2, 4);
        mbar_init(&s.inv3, 4);
        mbar_init(&s.t_ready, 2);
        mbar_init(&s.t_free, 1);
        mbar_init(&s.s0_copy, 4);
        mbar_init(&s.kt_full, 1);
        mbar_init(&s.kqs0_full, 1);
        mbar_init(&s.r_ready, 4);
        mbar_init(&s.o_scaled, 2);
        mbar_init(&s.u_full, 1);
        mbar_init(&s.u_copy, 4);
        mbar_init(&s.s_ready, 1);
        mbar_init(&s.o_full, 1);
        mbar_init(&s.o_free, 2);
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

    if (warp == kWarpTma) {
        // ------------------------------------------------------------ K, Q and V tiles
        if (lane == 0) {
            prefetch_tmap(&maps.q);
            prefetch_tmap(&maps.k);
            prefetch_tmap(&maps.v);
            Chunks ch{a, b - a, s0, 0};
            int64_t t0, ae;
            int n;
            uint32_t c = 0, nkq = 0, nv = 0;
            bool ok = true;
            while (ok && ch.next(t0, n, ae)) {
                const int bb = c & 1;
                if (c >= 2 && !wait_bar(&s.kq_empty[bb], par((c >> 1) - 1), abort_flag, err)) { ok = false; break; }
                mbar_arrive_expect_tx(&s.kq_full[bb], 32768);
                ++nkq;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    tma_load_3d(s.kq[bb] + h * 16384, &maps.k, &s.kq_full[bb], 64 * h, kh, (int)t0);
                    tma_load_3d(s.kq[bb] + h * 16384 + 8192, &maps.q, &s.kq_full[bb], 64 * h, kh, (int)t0);
                }
                if (c >= 1 && !wait_bar(&s.v_empty, par(c - 1), abort_flag, err)) { ok = false; break; }
                mbar_arrive_expect_tx(&s.v_full, 16384);
                ++nv;
#pragma unroll
                for (int h = 0; h < 2; ++h) tma_load_3d(s.v + h * 8192, &maps.v, &s.v_full, 64 * h, hv, (int)t0);
                ++c;
            }
            // never leave a copy in flight
            for (uint32_t k = nkq > 2 ? nkq - 2 : 0; k < nkq; ++k) mbar_wait(&s.kq_full[k & 1], par(k >> 1), kWaitNs);
            if (nv > 0) mbar_wait(&s.v_full, par(nv - 1), kWaitNs);
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t i_kq = idesc_bf16_f32(128, 64, false, false);   // [K;Q] x K^T
            constexpr uint32_t i_ks = idesc_bf16_f32(128, 128, false, true);   // [K;Q] x S0 (MN-major)
            constexpr uint32_t i_kt = idesc_bf16_f32(128, 64, true, false);    // S0^T (MN) x K^T (K-major)
            constexpr uint32_t i_u = idesc_bf16_f32(128, 64, false, true);     // R^T (TMEM) x T^T (MN)
            constexpr uint32_t i_s = idesc_bf16_f32(128, 128, true, false);    // K^T (MN) x U' (K-major)
            constexpr uint32_t i_o = idesc_bf16_f32(128, 128, false, false);   // P (TMEM) x U (K-major)
            // descriptors built once; + offset / 16 addresses further into a tile
            uint64_t dKQ[2], dKt[2];
            for (int bb = 0; bb < 2; ++bb) {
                dKQ[bb] = sdesc_sw128(smem_u32(s.kq[bb]), 16, 1024);     // K-major, k-halves 16 KB apart
                dKt[bb] = sdesc_sw128(smem_u32(s.kq[bb]), 16384, 1024);  // K^T: MN-major, k-halves 16 KB apart
            }
            const uint64_t dS0 = sdesc_sw128(smem_u32(s.s0), 16384, 1024);  // MN-major, v-halves 16 KB apart
            const uint64_t dUp = sdesc_sw128(smem_u32(s.s0), 16, 1024);     // U': K-major, 128 v rows
            const uint64_t dU = sdesc_sw128(smem_u32(s.r), 16, 1024);       // U: K-major, 128 v rows
            const uint64_t dT = sdesc_sw128(smem_u32(s.t), 16, 1024);       // T^T: MN-major, one 64-wide atom
            const uint32_t tS = tbase + kColS, tKQ = tbase + kColKQ, tU = tbase + kColU, tKT = tbase + kColKT;
            bool ok = true;
            auto issue_kq = [&](uint32_t c) -> bool {
                const int bb = c & 1;
                if (!wait_bar(&s.kq_full[bb], par(c >> 1), abort_flag, err)) return false;
                tc_fence_after();
                const uint32_t tAP = tbase + kColAP + 64u * bb;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t ko = (uint32_t)((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
                    mma_ss(tAP, dKQ[bb] + ko, dKQ[bb] + ko, i_kq, kk > 0);
                }
                mma_commit(&s.ap_full[bb]);
                return true;
            };
            ok = issue_kq(0);
            for (uint32_t c = 0; ok && c < (uint32_t)nch; ++c) {
                const int bb = c & 1;
                // (K S0)^T = S0^T K^T (v lanes: R^T is then formed by all four chain warps),
                // once S0 hi/lo is written
                if (!wait_bar(&s.s0_copy, par(c), abort_flag, err)) { ok = false; break; }
                tc_fence_after();
#pragma unroll
                for (int part = 0; part < 2; ++part) {
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t ko = (uint32_t)((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
                        mma_ss(tKT, dS0 + ((uint32_t)(part * 32768 + kk * 2048) >> 4), dKQ[bb] + ko, i_kt,
                               (part | kk) != 0);
                    }
                }
                mma_commit(&s.kt_full);
                // [K S0 ; Q S0] for the Q S0 rows of the output, once the last output rows were
                // read (it runs while the chain forms R^T)
                if (c >= 1 && !wait_bar(&s.o_free, par(c - 1), abort_flag, err)) { ok = false; break; }
                tc_fence_after();
#pragma unroll
                for (int part = 0; part < 2; ++part) {
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t ko = (uint32_t)((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
                        mma_ss(tKQ, dKQ[bb] + ko, dS0 + ((uint32_t)(part * 32768 + kk * 2048) >> 4), i_ks,
                               (part | kk) != 0);
                    }
                }
                mma_commit(&s.kqs0_full);
                // U^T = R^T T^T with R^T (hi/lo) read from TMEM: hi.hi + hi.lo + lo.hi
                if (!wait_bar(&s.r_ready, par(c), abort_flag, err)) { ok = false; break; }
                if (!wait_bar(&s.t_ready, par(c), abort_flag, err)) { ok = false; break; }
                tc_fence_after();
#pragma unroll
                for (int pass = 0; pass < 3; ++pass) {
                    const uint32_t ra = pass == 2 ? 8u : 0u, to = pass == 1 ? 8192u : 0u;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_ts(tU, tKT + kk * 16 + ra, dT + ((to + kk * 2048) >> 4), i_u, (pass | kk) != 0);
                }
                mma_commit(&s.u_full);
                mma_commit(&s.t_free);
                // the next chunk's [KK^T ; QK^T] for its preparation
                if (c + 1 < (uint32_t)nch && !issue_kq(c + 1)) { ok = false; break; }
                // S += K^T U' (hi, lo), then O += P U onto the scaled Q S0 rows
                if (!wait_bar(&s.u_copy, par(c), abort_flag, err)) { ok = false; break; }
                tc_fence_after();
#pragma unroll
                for (int part = 0; part < 2; ++part) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_ss(tS, dKt[bb] + ((uint32_t)(kk * 2048) >> 4),
                               dUp + ((uint32_t)(part * 16384 + kk * 32) >> 4), i_s, 1u);
                }
                mma_commit(&s.s_ready);
                if (!wait_bar(&s.p_ready[bb], par(c >> 1), abort_flag, err)) { ok = false; break; }
                if (!wait_bar(&s.o_scaled, par(c), abort_flag, err)) { ok = false; break; }
                tc_fence_after();
                const uint32_t tAP = tbase + kColAP + 64u * bb;
#pragma unroll
                for (int pass = 0; pass < 3; ++pass) {
                    const uint32_t pa = pass == 2 ? 8u : 0u, uo = pass == 1 ? 16384u : 0u;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_ts(tKQ, tAP + kk * 16 + pa, dU + ((uo + kk * 32) >> 4), i_o, 1u);
                }
                mma_commit(&s.o_full);
                mma_commit(&s.kq_empty[bb]);
            }
            mma_commit(&s.drain);
            mbar_wait(&s.drain, 0, kWaitNs);
        }
    } else if (warp >= kWarpChain && warp < kWarpPrep) {
        // ------------------------------------------------------------ the state chain
        const int q = warp & 3;
        const int r = q * 32 + lane;  // TMEM lane: state row k / output row / value column v
        const uint32_t tl = (uint32_t)(q * 32) << 16;
        const uint32_t tS = tbase + tl + kColS, tU = tbase + tl + kColU, tKT = tbase + tl + kColKT;
        // export row of this request's first chunk: the chunks of the requests before it
        int64_t fc = 0;
        if (io.chunk_states) {
            for (int rr = 0; rr < i; ++rr) {
                const int64_t lr = (int64_t)p.cu[rr + 1] - p.cu[rr];
                int64_t sr = io.num_computed ? io.num_computed[rr] : 0;
                if (sr < 0 || sr + lr > 0x7fffffffLL) sr = 0;
                if (lr > 0) fc += (sr + lr - 1) / kL - sr / kL + 1;
            }
        }
        auto chunk_dests = [&](int j, int64_t abs_end) {
            Dests d{{nullptr, nullptr, nullptr, nullptr}, 0};
            if (io.chunk_states) d.d[d.n++] = io.chunk_states + ((size_t)(fc + j) * p.Hv + hv) * state_elems;
            if (io.block_table && p.bs > 0 && abs_end % p.bs == 0) {
                const int64_t colb = abs_end / p.bs - 1;
                if (colb >= p.btw) {
                    if (r == 0) atomicOr(err, SSD_DEVERR_BLOCK_TABLE);
                } else {
                    const int slot = io.block_table[(size_t)i * p.btw + colb];
                    if (slot >= p.num_slots || !io.state_pool) {
                        if (r == 0 && slot >= 0) atomicOr(err, SSD_DEVERR_BLOCK_SLOT);
                    } else if (slot >= 0) {
                        d.d[d.n++] = io.state_pool + ((size_t)slot * p.Hv + hv) * state_elems;
                    }
                }
            }
            return d;
        };
        auto store_row = [&](const Dests &d, int cc, const uint32_t (&vals)[32]) {
            for (int f = 0; f < d.n; ++f) {
                float *dst = d.d[f] + (size_t)r * kV + cc * 32;
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    *reinterpret_cast<uint4 *>(dst + 4 * e) =
                        make_uint4(vals[4 * e], vals[4 * e + 1], vals[4 * e + 2], vals[4 * e + 3]);
            }
        };
        Chunks ch{a, b - a, s0, 0};
        int64_t t0 = 0, ae = 0, prev_ae = 0;
        int n = 0;
        bool ok = true;
        for (uint32_t c = 0; ok && ch.next(t0, n, ae); ++c) {
            const int bb = c & 1;
            const GdnVec &vc = s.vec[bb];
            // ---- S: state outputs of the previous chunk, S0 hi/lo (for the K S0 / Q S0
            // product) and gamma_L S in place, in one pass
            if (c >= 1 && !wait_bar_warp(&s.s_ready, par(c - 1), abort_flag, err)) { ok = false; break; }
            if (!wait_bar_warp(&s.vec2_ready[bb], par(c >> 1), abort_flag, err)) { ok = false; break; }
            tc_fence_after();
            {
                const Dests d = c >= 1 ? chunk_dests((int)c - 1, prev_ae) : Dests{{nullptr, nullptr, nullptr, nullptr}, 0};
#pragma unroll 1
                for (int c2 = 0; c2 < 2; ++c2) {
                    uint32_t v[2][32];
                    if (c == 0) {
#pragma unroll
                        for (int h = 0; h < 2; ++h)
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                v[h][e] = init ? __float_as_uint(init[(size_t)r * kV + c2 * 64 + h * 32 + e]) : 0u;
                    } else {
                        tmem_ld32(tS + c2 * 64, v[0]);
                        tmem_ld32(tS + c2 * 64 + 32, v[1]);
                        tmem_ld_wait();
                        store_row(d, 2 * c2, v[0]);
                        store_row(d, 2 * c2 + 1, v[1]);
                    }
                    // S0 hi/lo: row k = r, v = 64 c2 .. 64 c2 + 63 (v-half c2)
                    uint8_t *hb = s.s0 + c2 * 16384, *lb = hb + 32768;
#pragma unroll
                    for (int ch8 = 0; ch8 < 8; ++ch8) {
                        uint32_t hi[4], lo[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            split_pair(f2(__uint_as_float(v[ch8 >> 2][8 * (ch8 & 3) + 2 * e]),
                                          __uint_as_float(v[ch8 >> 2][8 * (ch8 & 3) + 2 * e + 1])),
                                       hi[e], lo[e]);
                        const uint32_t off = sw128_off((uint32_t)r, (uint32_t)ch8);
                        *reinterpret_cast<uint4 *>(hb + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                        *reinterpret_cast<uint4 *>(lb + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                    }
                    // gamma_L S back to TMEM in the same pass (the state product adds to it)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[h][e] = __float_as_uint(__uint_as_float(v[h][e]) * vc.gL);
                        tmem_st32(tS + c2 * 64 + h * 32, v[h]);
                    }
                }
            }
            tmem_st_wait();
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.s0_copy);
            // ---- R^T[v][t] = beta_t (V[t][v] - gamma_t rk_t (K S0)^T[v][t]) by all four warps
            // (thread = value column v = r), written over (K S0)^T as bf16 hi/lo -- per
            // 16-token block 8 hi then 8 lo columns -- the A operand of the U product
            if (!wait_bar_warp(&s.kt_full, par(c), abort_flag, err)) { ok = false; break; }
            if (!wait_bar_warp(&s.v_full, par(c), abort_flag, err)) { ok = false; break; }
            tc_fence_after();
            {
                const uint8_t *vt = s.v + (r >> 6) * 8192;  // this column's v-half of the V tile
                const uint32_t vch = (uint32_t)((r & 63) >> 3), vsub = (uint32_t)(r & 7) * 2;
#pragma unroll 1
                for (int kk = 0; kk < 4; ++kk) {
                    uint32_t v[16];
                    tmem_ld16(tKT + kk * 16, v);
                    tmem_ld_wait();
                    uint32_t hi[8], lo[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int t = kk * 16 + 2 * e;
                        const uint32_t x0 = *reinterpret_cast<const uint16_t *>(vt + t * 128 + ((vch ^ (uint32_t)(t & 7)) << 4) + vsub);
                        const uint32_t x1 =
                            *reinterpret_cast<const uint16_t *>(vt + (t + 1) * 128 + ((vch ^ (uint32_t)((t + 1) & 7)) << 4) + vsub);
                        const float r0 = vc.beta[t] * (__uint_as_float(x0 << 16) - vc.grk[t] * __uint_as_float(v[2 * e]));
                        const float r1 =
                            vc.beta[t + 1] * (__uint_as_float(x1 << 16) - vc.grk[t + 1] * __uint_as_float(v[2 * e + 1]));
                        split_pair(f2(r0, r1), hi[e], lo[e]);
                    }
                    tmem_st8(tKT + kk * 16, hi);
                    tmem_st8(tKT + kk * 16 + 8, lo);
                }
                tmem_st_wait();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&s.v_empty);
                mbar_arrive(&s.r_ready);
            }
            // ---- U and U' = diag(rk e^{G_L - G}) U as hi/lo, row v = r: [v][s] (U' over S0
            // hi/lo: both products that read S0 were issued before U)
            if (!wait_bar_warp(&s.u_full, par(c), abort_flag, err)) { ok = false; break; }
            tc_fence_after();
            {
                uint32_t v[2][32];
                tmem_ld32(tU, v[0]);
                tmem_ld32(tU + 32, v[1]);
                tmem_ld_wait();
#pragma unroll
                for (int ch8 = 0; ch8 < 8; ++ch8) {
                    uint32_t hi[4], lo[4], hw[4], lw[4];
                    const float4 wa = *reinterpret_cast<const float4 *>(&vc.wu[8 * ch8]);
                    const float4 wb = *reinterpret_cast<const float4 *>(&vc.wu[8 * ch8 + 4]);
                    const float wv[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float u0 = __uint_as_float(v[ch8 >> 2][8 * (ch8 & 3) + 2 * e]);
                        const float u1 = __uint_as_float(v[ch8 >> 2][8 * (ch8 & 3) + 2 * e + 1]);
                        split_pair(f2(u0, u1), hi[e], lo[e]);
                        split_pair(f2(wv[2 * e] * u0, wv[2 * e + 1] * u1), hw[e], lw[e]);
                    }
                    const uint32_t off = sw128_off((uint32_t)r, (uint32_t)ch8);
                    *reinterpret_cast<uint4 *>(s.r + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                    *reinterpret_cast<uint4 *>(s.r + 16384 + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                    *reinterpret_cast<uint4 *>(s.s0 + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                    *reinterpret_cast<uint4 *>(s.s0 + 16384 + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                }
            }
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.u_copy);
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.vec_free[bb]);
            prev_ae = ae;
        }
        // ---- the state after the last chunk: its outputs and the final states
        if (ok && wait_bar_warp(&s.s_ready, par((uint32_t)nch - 1), abort_flag, err)) {
            tc_fence_after();
            const Dests d = chunk_dests(nch - 1, prev_ae);
#pragma unroll 1
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t v[32];
                tmem_ld32(tS + cc * 32, v);
                tmem_ld_wait();
                store_row(d, cc, v);
                store_row(fin, cc, v);
            }
        }
    } else if (warp == kWarpOut || warp == kWarpOut + 1) {
        // ------------------------------------------------------------ output rows
        // Rows 64..127 of the [K S0 ; Q S0] accumulator (warps 2, 3: TMEM lane quadrants
        // 2, 3): the Q S0 rows scaled by scale gamma rq, then, once P U has been added,
        // O -> bf16; off the state chain, whose warps go on to the next chunk.
        const int q = warp & 3;
        const int t = (q - 2) * 32 + lane;  // token row of the chunk
        const uint32_t tKQ = tbase + ((uint32_t)(q * 32) << 16) + kColKQ;
        __nv_bfloat16 *__restrict__ og = static_cast<__nv_bfloat16 *>(io.o);
        Chunks ch{a, b - a, s0, 0};
        int64_t t0, ae;
        int n;
        bool ok = true;
        for (uint32_t c = 0; ok && ch.next(t0, n, ae); ++c) {
            const int bb = c & 1;
            // the Q S0 rows scaled by scale gamma rq before the P U product adds to them
            if (!wait_bar_warp(&s.vec2_ready[bb], par(c >> 1), abort_flag, err)) { ok = false; break; }
            if (!wait_bar_warp(&s.kqs0_full, par(c), abort_flag, err)) { ok = false; break; }
            tc_fence_after();
            {
                const float wq = s.vec[bb].osc[t];
#pragma unroll 1
                for (int c2 = 0; c2 < 2; ++c2) {
                    uint32_t v[2][32];
                    tmem_ld32(tKQ + c2 * 64, v[0]);
                    tmem_ld32(tKQ + c2 * 64 + 32, v[1]);
                    tmem_ld_wait();
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[h][e] = __float_as_uint(__uint_as_float(v[h][e]) * wq);
                        tmem_st32(tKQ + c2 * 64 + h * 32, v[h]);
                    }
                }
                tmem_st_wait();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&s.o_scaled);
                mbar_arrive(&s.vec_free[bb]);
            }
            if (!wait_bar_warp(&s.o_full, par(c), abort_flag, err)) { ok = false; break; }
            tc_fence_after();
            __nv_bfloat16 *orow = og + ((size_t)(t0 + t) * p.Hv + hv) * kV;
#pragma unroll 1
            for (int c2 = 0; c2 < 2; ++c2) {
                uint32_t v[2][32];
                tmem_ld32(tKQ + c2 * 64, v[0]);
                tmem_ld32(tKQ + c2 * 64 + 32, v[1]);
                tmem_ld_wait();
                if (c2 == 1) {
                    // the accumulator is free for the next chunk's K S0 / Q S0 product
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&s.o_free);
                }
                if (t < n) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        uint32_t pk[4];
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj)
                            pk[jj] = pack_bf16x2(__uint_as_float(v[e >> 2][8 * (e & 3) + 2 * jj]),
                                                 __uint_as_float(v[e >> 2][8 * (e & 3) + 2 * jj + 1]));
                        *reinterpret_cast<uint4 *>(orow + c2 * 64 + 8 * e) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    }
                }
            }
        }
    } else if (warp >= kWarpPrep) {
        // ------------------------------------------------------------ the next chunk's A, P and T
        const int q = warp & 3;
        const uint32_t tl = (uint32_t)(q * 32) << 16;
        const float *__restrict__ gg = io.g;
        const float *__restrict__ gb = io.beta;
        Chunks ch{a, b - a, s0, 0}, ahead{a, b - a, s0, 0};
        int64_t t0, ae, ta0 = 0, tae;
        int n, na = 0;
        // warp q = 0 loads each chunk's gates a chunk ahead (lane l: tokens 2l, 2l + 1)
        float g_nx[2] = {0.f, 0.f}, b_nx[2] = {0.f, 0.f};
        auto load_gates = [&]() {
            if (q == 0 && ahead.next(ta0, na, tae)) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int t = 2 * lane + e;
                    g_nx[e] = t < na ? gg[(size_t)(ta0 + t) * p.Hv + hv] : 0.f;
                    b_nx[e] = t < na ? gb[(size_t)(ta0 + t) * p.Hv + hv] : 0.f;
                }
            }
        };
        load_gates();
        bool ok = true;
        for (uint32_t c = 0; ok && ch.next(t0, n, ae); ++c) {
            const int bb = c & 1;
            GdnVec &vc = s.vec[bb];
            const float gx[2] = {g_nx[0], g_nx[1]}, bx[2] = {b_nx[0], b_nx[1]};
            load_gates();  // the next chunk's, in flight while this one is prepared
            if (c >= 2 && !wait_bar_warp(&s.vec_free[bb], par((c >> 1) - 1), abort_flag, err)) { ok = false; break; }
            if (!wait_bar_warp(&s.kq_full[bb], par(c >> 1), abort_flag, err)) { ok = false; break; }
            // gates: inclusive prefix sums of g log2(e) over the chunk (zero past its tokens)
            if (q == 0) {
                const float x0 = gx[0] * kLog2e, x1 = gx[1] * kLog2e;
                vc.beta[2 * lane] = bx[0];
                vc.beta[2 * lane + 1] = bx[1];
                float incl = x0 + x1;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += y;
                }
                vc.gl2[2 * lane] = incl - x1;
                vc.gl2[2 * lane + 1] = incl;
            }
            // l2 factors: warps q = 0, 1 the k rows 32 q + lane, q = 2, 3 the q rows 32 (q - 2) + lane
            const int tq = (q & 1) * 32 + lane;
            {
                float f = 0.f;
                if (tq < n) {
                    f = 1.f;
                    if (p.l2norm) {
                        float ss0 = 0.f, ss1 = 0.f;
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const uint8_t *row = s.kq[bb] + h * 16384 + (q >= 2 ? 8192 : 0) + tq * 128;
#pragma unroll
                            for (int c16 = 0; c16 < 8; ++c16) {
                                const uint4 raw = *reinterpret_cast<const uint4 *>(row + c16 * 16);
                                const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    const float lo = bf16lo_to_f32(w4[e]), hi = bf16hi_to_f32(w4[e]);
                                    ss0 = fmaf(lo, lo, ss0);
                                    ss1 = fmaf(hi, hi, ss1);
                                }
                            }
                        }
                        f = rsqrtf(ss0 + ss1 + 1e-6f);
                    }
                }
                if (q < 2) vc.rk[tq] = f;
                else vc.rq[tq] = f;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.vec_ready[bb]);
            if (!wait_bar_warp(&s.vec_ready[bb], par(c >> 1), abort_flag, err)) { ok = false; break; }
            // what the state chain takes: gamma rk and rk e^{G_L - G} (q = 0, 1), scale gamma rq
            // (q = 2, 3), gamma_L
            {
                const float gLl = vc.gl2[kL - 1], gt = vc.gl2[tq];
                if (q < 2) {
                    vc.grk[tq] = fast_exp2(gt) * vc.rk[tq];
                    vc.wu[tq] = vc.rk[tq] * fast_exp2(fminf(gLl - gt, 0.f));
                    vc.wb[tq] = vc.rk[tq] * fast_exp2(fminf(vc.gl2[tq | 15] - gt, 0.f));
                } else {
                    vc.osc[tq] = p.scale * vc.rq[tq] * fast_exp2(gt);
                }
                if (q == 0 && lane == 0) vc.gL = fast_exp2(gLl);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.vec2_ready[bb]);
            if (!wait_bar_warp(&s.vec2_ready[bb], par(c >> 1), abort_flag, err)) { ok = false; break; }
            // ---- A (to shared memory, transposed) and P rows (hi/lo in place in TMEM).  Below
            // the diagonal 16-row block the decay splits around the column block's last row
            // b: e^{G_s - G_r} = e^{G_s - G_b} e^{G_b - G_r}, both factors <= 1, the second
            // (times rk_r) precomputed per column; the diagonal block is evaluated directly.
            if (!wait_bar_warp(&s.ap_full[bb], par(c >> 1), abort_flag, err)) { ok = false; break; }
            tc_fence_after();
            const uint32_t tAP = tbase + tl + kColAP + 64u * bb;
            // one 16-column block of TMEM per round (a short loop body: the code stays small)
            if (q < 2) {
                const int sr = tq, bs = sr >> 4;
                const float ws = vc.beta[sr] * vc.rk[sr], gs = vc.gl2[sr];
#pragma unroll 1
                for (int cb = 0; cb < 4; ++cb) {
                    uint32_t v[16];
                    tmem_ld16(tAP + cb * 16, v);
                    tmem_ld_wait();
                    float av[16];
                    if (cb < bs) {
                        const float f = ws * fast_exp2(fminf(gs - vc.gl2[16 * cb + 15], 0.f));
#pragma unroll
                        for (int e = 0; e < 16; ++e) av[e] = f * vc.wb[cb * 16 + e] * __uint_as_float(v[e]);
                    } else if (cb == bs) {
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const int rc = cb * 16 + e;
                            av[e] = rc < sr ? ws * vc.rk[rc] * fast_exp2(fminf(gs - vc.gl2[rc], 0.f)) * __uint_as_float(v[e])
                                            : 0.f;
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 16; ++e) av[e] = 0.f;
                    }
                    // A^T[rc][sr] = A[sr][rc]: for each rc the lanes store consecutive words
#pragma unroll
                    for (int e = 0; e < 16; ++e) s.a[(cb * 16 + e) * kLdA + sr] = av[e];
                }
            } else {
                const int t = tq, bt = t >> 4;
                const float wt = p.scale * vc.rq[t], gt = vc.gl2[t];
                // in place per block: the 16 fp32 columns read become 8 hi + 8 lo columns
#pragma unroll 1
                for (int kk = 0; kk < 4; ++kk) {
                    uint32_t v[16];
                    tmem_ld16(tAP + kk * 16, v);
                    tmem_ld_wait();
                    float pv[16];
                    if (kk < bt) {
                        const float f = wt * fast_exp2(fminf(gt - vc.gl2[16 * kk + 15], 0.f));
#pragma unroll
                        for (int e = 0; e < 16; ++e) pv[e] = f * vc.wb[kk * 16 + e] * __uint_as_float(v[e]);
                    } else if (kk == bt) {
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const int sc = kk * 16 + e;
                            pv[e] = sc <= t ? wt * vc.rk[sc] * fast_exp2(fminf(gt - vc.gl2[sc], 0.f)) * __uint_as_float(v[e])
                                            : 0.f;
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 16; ++e) pv[e] = 0.f;
                    }
                    uint32_t hi[8], lo[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) split_pair(f2(pv[2 * e], pv[2 * e + 1]), hi[e], lo[e]);
                    tmem_st8(tAP + kk * 16, hi);
                    tmem_st8(tAP + kk * 16 + 8, lo);
                }
                tmem_st_wait();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.p_ready[bb]);
            // ---- T = (I + A)^-1 by 32 x 32 blocks:
            //   T11 = (I + A11)^-1, T22 = (I + A22)^-1   (warps q = 0 and 1, in parallel: one
            //        column per thread by a right-looking substitution over 32 rows)
            //   M1  = A21 T11,  T21 = -T22 M1           (all four warps: 8 rows x 1 column each)
            // T11, M1, T21 are kept column by column (stride 33, lane-indexed reads); T22
            // as rows of T22^T in the A^T rows 32..63, columns 0..31 (that block, A12^T, is
            // zero and never read).  T^T (row j = column j of T) is then written as hi/lo,
            // once the last U product has read T.
            const int j = lane;
            if (q < 2) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&s.a_ready);
                if (!wait_bar_warp(&s.a_ready, par(c), abort_flag, err)) { ok = false; break; }
                const int o = 32 * q;  // the diagonal block's first row / column
                float x[32];
#pragma unroll
                for (int rr = 0; rr < 32; ++rr) x[rr] = rr == j ? 1.f : 0.f;
#pragma unroll
                for (int cc = 0; cc < 31; ++cc) {
                    const float xc = x[cc];
                    const float *arow = s.a + (o + cc) * kLdA + o;
#pragma unroll
                    for (int rr = (cc + 1) & ~3; rr < 32; rr += 4) {
                        const float4 a4 = *reinterpret_cast<const float4 *>(arow + rr);
                        // entries rr <= cc of A^T row cc are zero (A is strictly lower)
                        x[rr] = fmaf(-a4.x, xc, x[rr]);
                        x[rr + 1] = fmaf(-a4.y, xc, x[rr + 1]);
                        x[rr + 2] = fmaf(-a4.z, xc, x[rr + 2]);
                        x[rr + 3] = fmaf(-a4.w, xc, x[rr + 3]);
                    }
                }
                if (q == 0) {
#pragma unroll
                    for (int rr = 0; rr < 32; ++rr) s.t11[j * 33 + rr] = x[rr];
                } else {
#pragma unroll
                    for (int rr = 0; rr < 32; rr += 4)
                        *reinterpret_cast<float4 *>(s.a + (32 + j) * kLdA + rr) = make_float4(x[rr], x[rr + 1], x[rr + 2], x[rr + 3]);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&s.inv1);
            }
            if (!wait_bar_warp(&s.inv1, par(c), abort_flag, err)) { ok = false; break; }
            const int r0 = 8 * q;  // this warp's 8 rows of M1 and T21
            {
                // M1[r][j] = sum_c A[32 + r][c] T11[c][j] = sum_c A^T[c][32 + r] T11[c][j]
                float m[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
                for (int cc = 0; cc < 32; ++cc) {
                    const float tv = s.t11[j * 33 + cc];
                    const float4 a0 = *reinterpret_cast<const float4 *>(s.a + cc * kLdA + 32 + r0);
                    const float4 a1 = *reinterpret_cast<const float4 *>(s.a + cc * kLdA + 36 + r0);
                    m[0] = fmaf(a0.x, tv, m[0]);
                    m[1] = fmaf(a0.y, tv, m[1]);
                    m[2] = fmaf(a0.z, tv, m[2]);
                    m[3] = fmaf(a0.w, tv, m[3]);
                    m[4] = fmaf(a1.x, tv, m[4]);
                    m[5] = fmaf(a1.y, tv, m[5]);
                    m[6] = fmaf(a1.z, tv, m[6]);
                    m[7] = fmaf(a1.w, tv, m[7]);
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) s.m1[j * 33 + r0 + e] = m[e];
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.inv2);
            if (!wait_bar_warp(&s.inv2, par(c), abort_flag, err)) { ok = false; break; }
            {
                // T21[r][j] = -sum_k T22[r][k] M1[k][j]; T22[r][k] = (T22^T row k)[r]
                float m[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
                for (int kk = 0; kk < 32; ++kk) {
                    const float mv = s.m1[j * 33 + kk];
                    const float4 t0v = *reinterpret_cast<const float4 *>(s.a + (32 + kk) * kLdA + r0);
                    const float4 t1v = *reinterpret_cast<const float4 *>(s.a + (32 + kk) * kLdA + r0 + 4);
                    m[0] = fmaf(-t0v.x, mv, m[0]);
                    m[1] = fmaf(-t0v.y, mv, m[1]);
                    m[2] = fmaf(-t0v.z, mv, m[2]);
                    m[3] = fmaf(-t0v.w, mv, m[3]);
                    m[4] = fmaf(-t1v.x, mv, m[4]);
                    m[5] = fmaf(-t1v.y, mv, m[5]);
                    m[6] = fmaf(-t1v.z, mv, m[6]);
                    m[7] = fmaf(-t1v.w, mv, m[7]);
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) s.t21[j * 33 + r0 + e] = m[e];
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.inv3);
            if (q >= 2) continue;
            if (!wait_bar_warp(&s.inv3, par(c), abort_flag, err)) { ok = false; break; }
            if (c >= 1 && !wait_bar_warp(&s.t_free, par(c - 1), abort_flag, err)) { ok = false; break; }
            {
                // row sj of T^T = column sj of T: rows 0..31 then 32..63
                const int sj = 32 * q + j;
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) {
                    float col[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int t = 8 * c8 + e;
                        if (q == 0) col[e] = t < 32 ? s.t11[j * 33 + t] : s.t21[j * 33 + (t - 32)];
                        else col[e] = t < 32 ? 0.f : s.a[(32 + j) * kLdA + (t - 32)];
                    }
                    uint32_t hi[4], lo[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) split_pair(f2(col[2 * e], col[2 * e + 1]), hi[e], lo[e]);
                    const uint32_t off = sw128_off((uint32_t)sj, (uint32_t)c8);
                    *reinterpret_cast<uint4 *>(s.t + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                    *reinterpret_cast<uint4 *>(s.t + 8192 + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                }
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.t_ready);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 gdn_encode_fn() {
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

// 3-D bf16 map over a row-major (d2, d1, d0 = 128) tensor; box = 64 x 1 x 64 rows, 128-byte swizzle.
bool gdn_map(CUtensorMap *m, const void *g, uint64_t d1, uint64_t d2) {
    auto fn = gdn_encode_fn();
    if (!fn) return false;
    const uint64_t dims[3] = {128, d1, d2 > 0 ? d2 : 1};
    const uint64_t strides[2] = {128 * 2, 128 * d1 * 2};
    const uint32_t box[3] = {64, 1, (uint32_t)kL};
    const uint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(g), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool gdn_tc_supported(const ssd_gdn_dims *d) {
    return d->dtype == SSD_DTYPE_BF16 && d->K == kK && d->V == kV && d->chunk_size == kL;
}

// The tcgen05 GDN prefill: one CTA per (request, value head).  The caller has
// validated the arguments (dims, pointers, alignment, slot tables).
int launch_gdn_tc(const ssd_gdn_dims *d, const int32_t *cu_seqlens, const ssd_gdn_io *io, cudaStream_t stream) {
    GdnTcParams p{};
    p.T = d->T;
    p.R = d->R;
    p.Hk = d->Hk;
    p.Hv = d->Hv;
    p.bs = io->block_table ? d->block_size : 0;
    p.btw = d->block_table_width;
    p.num_slots = d->num_slots;
    p.l2norm = d->l2norm ? 1 : 0;
    p.scale = d->scale != 0.f ? d->scale : 1.f / sqrtf((float)d->K);
    p.cu = cu_seqlens;
    p.io = *io;
    // with no tokens (every request empty) no tile is loaded and the maps stay zero
    GdnTcMaps maps;
    memset(&maps, 0, sizeof(maps));
    if (d->T > 0 && (!gdn_map(&maps.q, io->q, d->Hk, (uint64_t)d->T) || !gdn_map(&maps.k, io->k, d->Hk, (uint64_t)d->T) ||
                     !gdn_map(&maps.v, io->v, d->Hv, (uint64_t)d->T)))
        return SSD_ERR_CUDA;
    const int smem = (int)sizeof(GdnTcSmem);
    int dev = 0;
    cudaGetDevice(&dev);
    static std::mutex mu;
    static bool attr_done[64] = {};
    {
        std::lock_guard<std::mutex> lock(mu);
        const bool known = dev >= 0 && dev < 64;
        if (!known || !attr_done[dev]) {
            if (cudaFuncSetAttribute(gdn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
                return SSD_ERR_CUDA;
            if (known) attr_done[dev] = true;
        }
    }
    const int64_t ctas = (int64_t)d->R * d->Hv;
    if (ctas > 0x7fffffffLL) return SSD_ERR_DIMS;
    return launch_after_prev(gdn_tc_kernel, dim3((unsigned)ctas), dim3(kThreads), smem, stream, p, maps) == cudaSuccess
               ? SSD_OK
               : SSD_ERR_CUDA;
}

}  // namespace ssd
