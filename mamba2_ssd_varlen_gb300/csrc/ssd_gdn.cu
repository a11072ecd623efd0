// ssd_gdn.cu -- gated delta rule (GDN) varlen prefill by chunks, with per-chunk
// state export, block checkpoints and dual read/write state slots ("Automatic
// prefix caching for GDN hybrid models (mamba_cache_mode=all) with MTP
// speculative decoding", Purpose, Kernels/layers: the chunk kernel's
// intermediate-state export and the block-aligned checkpoint scatter).
//
// The rule (published gated delta rule; S a K x V matrix per value head):
//     S <- e^{g_t} S;  u = beta_t (v_t - S^T k_t);  S <- S + k_t u^T;  o_t = scale S^T q_t
// Per chunk of L <= 64 tokens starting from state S0, with in-chunk prefix sums
// G of g and gamma = e^G (the WY form of the chunked rule):
//     A[s,r] = beta_s e^{G_s - G_r} k_s.k_r  (r < s)       strictly lower
//     (I + A) U = diag(beta) (V - diag(gamma) K S0)         a unit-lower solve
//     O = scale diag(gamma) Q S0 + P U,  P[t,s] = scale e^{G_t - G_s} q_t.k_s (s <= t)
//     S = gamma_L S0 + (diag(e^{G_L - G}) K)^T U
// The matrix products run on the tensor cores (mma.sync m16n8k16, bf16 operands,
// fp32 accumulation).  q, k, v are bf16 and enter exactly; the fp32 operands
// (S0, P, U) are split into a bf16 high part and a bf16 remainder, and the
// products that involve them are summed from hi*hi + hi*lo (+ lo*hi), which keeps
// about 16 mantissa bits.  The unit-lower solve runs on the CUDA cores in fp32,
// by 16-row blocks: each warp inverts one diagonal block, then every warp
// substitutes block by block for its own value columns.
//
// A CTA owns one (request, value head, 32-column slice of V) and walks the
// request's chunks in order, the state slice in registers (warp w holds rows
// 32w..32w+31 in the accumulator layout of the state product).  A and P do not
// depend on the column slice; the slices of one head recompute them rather than
// exchange them.
#include "ssd_internal.cuh"

namespace ssd {
namespace {

constexpr int kL = 64;        // chunk length
constexpr int kK = 128;       // key head dim
constexpr int kBV = 32;       // value columns per CTA
constexpr int kThreads = 128; // four warps
constexpr int kLdK = kK + 8;  // bf16 row stride of the K / Q tiles (272 bytes)
constexpr int kLdA = kL + 4;  // fp32 row stride of A
constexpr int kLdU = kL + 4;  // fp32 row stride of R^T / U^T (eight columns x four rows: 32 banks)
constexpr int kLdP = kL + 8;  // bf16 row stride of P and of U^T (144 bytes)
constexpr int kLdS = kBV + 8; // bf16 row stride of S0 [k][v] (80 bytes)
constexpr int kLdT = 20;      // fp32 row stride of the inverted diagonal blocks
constexpr float kLog2e = 1.4426950408889634f;

struct GdnParams {
    int64_t T;
    int32_t R, Hk, Hv, V, nvb, bs, btw, num_slots, l2norm;
    float scale;
    const int32_t *cu;
    ssd_gdn_io io;
};

struct GdnSmem {
    __nv_bfloat16 k[kL * kLdK];   // K tile [s][k]
    __nv_bfloat16 q[kL * kLdK];   // Q tile [t][k]
    float a[kL * kLdA];           // A [s][r]; after the solve: U' hi/lo [v][s] (bf16)
    __nv_bfloat16 ph[kL * kLdP];  // P hi [t][s]
    __nv_bfloat16 pl[kL * kLdP];  // P lo
    float ut[kBV * kLdU];         // R^T, solved in place into U^T [v][s]
    float tb[kL * kLdT];          // (I + A_bb)^-1 of the four 16 x 16 diagonal blocks, rows 16b..
    __nv_bfloat16 uh[kBV * kLdP]; // U^T hi [v][s]
    __nv_bfloat16 ul[kBV * kLdP]; // U^T lo
    __nv_bfloat16 sh[kK * kLdS];  // S0 hi [k][v]
    __nv_bfloat16 sl[kK * kLdS];  // S0 lo
    float gl2[kL];                // G * log2 e, inclusive prefix sums
    float beta[kL];
    float rk[kL], rq[kL];         // per-row l2 scale factors of k and q (1 without l2norm)
    float wu[kL];                 // rk e^{G_L - G}: the row weights of U' in the state product
};

__device__ __forceinline__ uint32_t smem_addr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void *p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(smem_addr(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void *p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(smem_addr(p)));
}
// d += a (16x16, row) * b (16x8, col), bf16 in, fp32 accumulate
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// Packed fp32 pairs (one 64-bit register pair) for the f32x2 instructions.
__device__ __forceinline__ uint64_t pair(float a, float b) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(a), "f"(b));
    return d;
}
__device__ __forceinline__ float pair_sum(uint64_t d) {
    float a, b;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(d));
    return a + b;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// fp32 pair -> (bf16x2 high parts, bf16x2 remainders)
__device__ __forceinline__ void split2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

__global__ void __launch_bounds__(kThreads, 2) gdn_chunk_kernel(const __grid_constant__ GdnParams p) {
    extern __shared__ __align__(16) uint8_t gdn_smem_raw[];
    GdnSmem &s = *reinterpret_cast<GdnSmem *>(gdn_smem_raw);
    __nv_bfloat16 *u2h = reinterpret_cast<__nv_bfloat16 *>(s.a);  // U'^T hi [v][s], after the solve
    __nv_bfloat16 *u2l = u2h + kBV * kLdP;
    const ssd_gdn_io &io = p.io;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gq = lane >> 2, cq = lane & 3;  // accumulator row group and column pair
    const int64_t cta = blockIdx.x;
    const int vb = (int)(cta % p.nvb);
    const int h = (int)((cta / p.nvb) % p.Hv);
    const int i = (int)(cta / ((int64_t)p.nvb * p.Hv));
    const int kh = h / (p.Hv / p.Hk);
    const int V = p.V, v0 = vb * kBV;
    const size_t state_elems = (size_t)kK * V;
    int32_t *err = io.device_err;

    if (cta == 0 && tid == 0 && (p.cu[0] != 0 || (int64_t)p.cu[p.R] != p.T)) atomicOr(err, SSD_DEVERR_CU_SEQLENS);
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
    // export row of this request's first chunk: chunks of the requests before it
    int64_t fc = 0;
    if (io.chunk_states) {
        for (int r = 0; r < i; ++r) {
            const int64_t lr = (int64_t)p.cu[r + 1] - p.cu[r];
            int64_t sr = io.num_computed ? io.num_computed[r] : 0;
            if (sr < 0 || sr + lr > 0x7fffffffLL) sr = 0;
            if (lr > 0) fc += (sr + lr - 1) / kL - sr / kL + 1;
        }
    }

    // ---- initial state slice -> registers (warp w: rows 32w.., 2 m-tiles x 4 n-tiles)
    float st[2][4][4];
    {
        const float *init = nullptr;
        if (io.init_slots && io.state_pool) {
            const int sl = io.init_slots[i];
            if (sl >= p.num_slots) {
                if (tid == 0) atomicOr(err, SSD_DEVERR_INIT_SLOT);
            } else if (sl >= 0) {
                init = io.state_pool + ((size_t)sl * p.Hv + h) * state_elems;
            }
        }
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int kr = 32 * warp + 16 * mt + gq + 8 * hh, vc = v0 + 8 * nt + 2 * cq;
                    float2 val = make_float2(0.f, 0.f);
                    if (init) val = *reinterpret_cast<const float2 *>(init + (size_t)kr * V + vc);
                    st[mt][nt][2 * hh] = val.x;
                    st[mt][nt][2 * hh + 1] = val.y;
                }
    }
    // S0 hi/lo for the products of the next chunk
    auto publish_state = [&]() {
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int kr = 32 * warp + 16 * mt + gq + 8 * hh, vc = 8 * nt + 2 * cq;
                    uint32_t hi, lo;
                    split2(st[mt][nt][2 * hh], st[mt][nt][2 * hh + 1], hi, lo);
                    *reinterpret_cast<uint32_t *>(s.sh + kr * kLdS + vc) = hi;
                    *reinterpret_cast<uint32_t *>(s.sl + kr * kLdS + vc) = lo;
                }
    };
    auto write_state = [&](float *dst) {
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int kr = 32 * warp + 16 * mt + gq + 8 * hh, vc = v0 + 8 * nt + 2 * cq;
                    *reinterpret_cast<float2 *>(dst + (size_t)kr * V + vc) =
                        make_float2(st[mt][nt][2 * hh], st[mt][nt][2 * hh + 1]);
                }
    };
    publish_state();

    const __nv_bfloat16 *qg = static_cast<const __nv_bfloat16 *>(io.q);
    const __nv_bfloat16 *kg = static_cast<const __nv_bfloat16 *>(io.k);
    const __nv_bfloat16 *vg = static_cast<const __nv_bfloat16 *>(io.v);
    __nv_bfloat16 *og = static_cast<__nv_bfloat16 *>(io.o);
    const int m0 = 16 * warp;  // the chunk rows this warp owns in the row-blocked products

    int64_t pos = 0;
    for (int j = 0; pos < b - a; ++j) {
        const int64_t abs0 = s0 + pos;
        const int n = (int)min((abs0 / kL + 1) * kL - abs0, b - a - pos);  // tokens of this chunk
        const int64_t t0 = a + pos;

        // ---- stage K and Q rows (zeros past the chunk), gates, and this thread's V values
        for (int idx = tid; idx < kL * (kK / 8); idx += kThreads) {
            const int r = idx / (kK / 8), c = (idx % (kK / 8)) * 8;
            __nv_bfloat16 *dk = s.k + r * kLdK + c, *dq = s.q + r * kLdK + c;
            if (r < n) {
                const size_t off = ((size_t)(t0 + r) * p.Hk + kh) * kK + c;
                cp_async16(dk, kg + off);
                cp_async16(dq, qg + off);
            } else {
                *reinterpret_cast<uint4 *>(dk) = make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4 *>(dq) = make_uint4(0, 0, 0, 0);
            }
        }
        if (tid < kL) {
            const bool in = tid < n;
            s.gl2[tid] = in ? io.g[(size_t)(t0 + tid) * p.Hv + h] * kLog2e : 0.f;
            s.beta[tid] = in ? io.beta[(size_t)(t0 + tid) * p.Hv + h] : 0.f;
        }
        uint32_t vraw[4][2];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int row = m0 + gq + 8 * hh;
                vraw[nt][hh] = row < n ? *reinterpret_cast<const uint32_t *>(
                                             vg + ((size_t)(t0 + row) * p.Hv + h) * V + v0 + 8 * nt + 2 * cq)
                                       : 0u;
            }
        cp_async_wait_all();
        __syncthreads();

        // ---- prefix sums of the gates (warp 0, two rows per lane); l2 factors (all warps)
        if (warp == 0) {
            const float x0 = s.gl2[2 * lane], x1 = s.gl2[2 * lane + 1];
            float incl = x0 + x1;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const float excl = incl - (x0 + x1);
            s.gl2[2 * lane] = excl + x0;
            s.gl2[2 * lane + 1] = incl;
        }
        {  // one row per lane: lanes 0-15 the k rows m0.., lanes 16-31 the q rows
            const int r = m0 + (lane & 15);
            const __nv_bfloat16 *row = (lane < 16 ? s.k : s.q) + r * kLdK;
            float f = 1.f;
            if (p.l2norm) {
                float ss0 = 0.f, ss1 = 0.f;
#pragma unroll
                for (int c = 0; c < kK; c += 8) {
                    const uint4 raw = *reinterpret_cast<const uint4 *>(row + c);
                    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float lo = __uint_as_float(w[e] << 16), hi = __uint_as_float(w[e] & 0xFFFF0000u);
                        ss0 = fmaf(lo, lo, ss0);
                        ss1 = fmaf(hi, hi, ss1);
                    }
                }
                f = rsqrtf(ss0 + ss1 + 1e-6f);
            }
            if (lane < 16) s.rk[r] = f;
            else s.rq[r] = f;
        }
        __syncthreads();

        // ---- A and P (rows m0..m0+15, columns up to the diagonal block)
        {
            float acc_a[8][4], acc_p[8][4];
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc_a[nt][e] = acc_p[nt][e] = 0.f;
#pragma unroll
            for (int kk = 0; kk < kK / 16; ++kk) {
                uint32_t fk[4], fq[4];
                ldsm_x4(fk, s.k + (m0 + (lane & 15)) * kLdK + kk * 16 + (lane >> 4) * 8);
                ldsm_x4(fq, s.q + (m0 + (lane & 15)) * kLdK + kk * 16 + (lane >> 4) * 8);
#pragma unroll
                for (int np = 0; np < 4; ++np) {
                    if (np > warp) break;
                    uint32_t fb[4];
                    ldsm_x4(fb, s.k + (16 * np + (lane & 7) + ((lane >> 4) << 3)) * kLdK + kk * 16 +
                                    ((lane >> 3) & 1) * 8);
                    mma_bf16(acc_a[2 * np], fk, fb[0], fb[1]);
                    mma_bf16(acc_a[2 * np + 1], fk, fb[2], fb[3]);
                    mma_bf16(acc_p[2 * np], fq, fb[0], fb[1]);
                    mma_bf16(acc_p[2 * np + 1], fq, fb[2], fb[3]);
                }
            }
            float wa_row[2], wp_row[2], g_row[2];  // this thread's two rows
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int row = m0 + gq + 8 * hh;
                wa_row[hh] = s.beta[row] * s.rk[row];
                wp_row[hh] = p.scale * s.rq[row];
                g_row[hh] = s.gl2[row];
            }
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                if (nt > 2 * warp + 1) break;
                const int col = 8 * nt + 2 * cq;
                const float2 gc = *reinterpret_cast<const float2 *>(s.gl2 + col);
                const float2 kc = *reinterpret_cast<const float2 *>(s.rk + col);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int row = m0 + gq + 8 * hh;
                    float pa[2], pp[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int c = col + e;
                        const float base = (e ? kc.y : kc.x) * exp2f(fminf(g_row[hh] - (e ? gc.y : gc.x), 0.f));
                        pa[e] = c < row ? wa_row[hh] * base * acc_a[nt][2 * hh + e] : 0.f;
                        pp[e] = c <= row ? wp_row[hh] * base * acc_p[nt][2 * hh + e] : 0.f;
                    }
                    *reinterpret_cast<float2 *>(s.a + row * kLdA + col) = make_float2(pa[0], pa[1]);
                    uint32_t hi, lo;
                    split2(pp[0], pp[1], hi, lo);
                    *reinterpret_cast<uint32_t *>(s.ph + row * kLdP + col) = hi;
                    *reinterpret_cast<uint32_t *>(s.pl + row * kLdP + col) = lo;
                }
            }
            // (I + A_bb)^-1 of this warp's diagonal block (its own rows and columns of A):
            // lane j < 16 solves for column j by forward substitution
            __syncwarp();
            if (lane < 16) {
                float x[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) {
                    const float *arow = s.a + (m0 + r) * kLdA + m0;
                    float acc = r == lane ? 1.f : 0.f;
#pragma unroll
                    for (int c = 0; c < r; ++c) acc = fmaf(-arow[c], x[c], acc);
                    x[r] = acc;
                }
#pragma unroll
                for (int r = 0; r < 16; ++r) s.tb[(m0 + r) * kLdT + lane] = x[r];
            }
        }

        // ---- K S0 -> R = diag(beta)(V - diag(gamma rk) K S0) into R^T; Q S0 kept for O
        float acc_o[4][4];
        {
            float acc_r[4][4];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc_r[nt][e] = acc_o[nt][e] = 0.f;
#pragma unroll
            for (int kk = 0; kk < kK / 16; ++kk) {
                uint32_t fk[4], fq[4];
                ldsm_x4(fk, s.k + (m0 + (lane & 15)) * kLdK + kk * 16 + (lane >> 4) * 8);
                ldsm_x4(fq, s.q + (m0 + (lane & 15)) * kLdK + kk * 16 + (lane >> 4) * 8);
#pragma unroll
                for (int np = 0; np < 2; ++np) {
                    uint32_t bh[4], bl[4];
                    const int mat = lane >> 3;
                    const int off = (kk * 16 + (lane & 7) + ((mat & 1) << 3)) * kLdS + 16 * np + ((mat >> 1) << 3);
                    ldsm_x4_t(bh, s.sh + off);
                    ldsm_x4_t(bl, s.sl + off);
                    mma_bf16(acc_r[2 * np], fk, bh[0], bh[1]);
                    mma_bf16(acc_r[2 * np], fk, bl[0], bl[1]);
                    mma_bf16(acc_r[2 * np + 1], fk, bh[2], bh[3]);
                    mma_bf16(acc_r[2 * np + 1], fk, bl[2], bl[3]);
                    mma_bf16(acc_o[2 * np], fq, bh[0], bh[1]);
                    mma_bf16(acc_o[2 * np], fq, bl[0], bl[1]);
                    mma_bf16(acc_o[2 * np + 1], fq, bh[2], bh[3]);
                    mma_bf16(acc_o[2 * np + 1], fq, bl[2], bl[3]);
                }
            }
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int row = m0 + gq + 8 * hh, col = 8 * nt + 2 * cq;
                    const float2 vv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&vraw[nt][hh]));
                    const float w = exp2f(s.gl2[row]) * s.rk[row], bt = s.beta[row];
                    s.ut[col * kLdU + row] = bt * (vv.x - w * acc_r[nt][2 * hh]);
                    s.ut[(col + 1) * kLdU + row] = bt * (vv.y - w * acc_r[nt][2 * hh + 1]);
                }
        }
        __syncthreads();

        // ---- unit-lower solve (I + A) U = R by 16-row blocks b = 0..3:
        //   U_b = (I + A_bb)^-1 (R_b - A_{b,<b} U_{<b})
        // warp w owns value columns 8w..8w+7, four lanes per column, lane quarter q the
        // rows q, q+4, q+8, q+12 of each block (neighbouring rows in one access: no
        // bank conflicts); the columns are independent, so only the warp syncs.
        if (warp == 0) {
            const float gll = s.gl2[n - 1];
            s.wu[lane] = s.rk[lane] * exp2f(fminf(gll - s.gl2[lane], 0.f));
            s.wu[lane + 32] = s.rk[lane + 32] * exp2f(fminf(gll - s.gl2[lane + 32], 0.f));
        }
        {
            const int vcol = 8 * warp + (lane >> 2), qr = lane & 3;
            float *ucol = s.ut + vcol * kLdU;
#pragma unroll
            for (int bk = 0; bk < kL / 16; ++bk) {
                float rr[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int sr = 16 * bk + 4 * e + qr;
                    const float *arow = s.a + sr * kLdA;
                    // A r-pairs times U r-pairs, two terms per packed instruction
                    uint64_t acc0 = pair(ucol[sr], 0.f), acc1 = pair(0.f, 0.f);
#pragma unroll
                    for (int r = 0; r < 16 * bk; r += 4) {
                        const float4 a4 = *reinterpret_cast<const float4 *>(arow + r);
                        const float2 u01 = *reinterpret_cast<const float2 *>(ucol + r);
                        const float2 u23 = *reinterpret_cast<const float2 *>(ucol + r + 2);
                        acc0 = fma2(pair(-a4.x, -a4.y), pair(u01.x, u01.y), acc0);
                        acc1 = fma2(pair(-a4.z, -a4.w), pair(u23.x, u23.y), acc1);
                    }
                    rr[e] = pair_sum(acc0) + pair_sum(acc1);
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) ucol[16 * bk + 4 * e + qr] = rr[e];
                __syncwarp();
                float uu[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float *trow = s.tb + (16 * bk + 4 * e + qr) * kLdT;
                    uint64_t acc0 = pair(0.f, 0.f), acc1 = pair(0.f, 0.f);
#pragma unroll
                    for (int c = 0; c < 16; c += 4) {
                        const float4 t4 = *reinterpret_cast<const float4 *>(trow + c);
                        const float2 u01 = *reinterpret_cast<const float2 *>(ucol + 16 * bk + c);
                        const float2 u23 = *reinterpret_cast<const float2 *>(ucol + 16 * bk + c + 2);
                        acc0 = fma2(pair(t4.x, t4.y), pair(u01.x, u01.y), acc0);
                        acc1 = fma2(pair(t4.z, t4.w), pair(u23.x, u23.y), acc1);
                    }
                    uu[e] = pair_sum(acc0) + pair_sum(acc1);
                }
                __syncwarp();
#pragma unroll
                for (int e = 0; e < 4; ++e) ucol[16 * bk + 4 * e + qr] = uu[e];
                __syncwarp();
            }
        }
        __syncthreads();  // U complete; A no longer read (its space takes U')

        // ---- U and U' = diag(rk e^{G_L - G}) U as bf16 hi/lo, [v][s]
        {
            for (int idx = tid; idx < kBV * (kL / 2); idx += kThreads) {
                const int vc = idx / (kL / 2), r = (idx % (kL / 2)) * 2;
                const float u0 = s.ut[vc * kLdU + r], u1 = s.ut[vc * kLdU + r + 1];
                uint32_t hi, lo;
                split2(u0, u1, hi, lo);
                *reinterpret_cast<uint32_t *>(s.uh + vc * kLdP + r) = hi;
                *reinterpret_cast<uint32_t *>(s.ul + vc * kLdP + r) = lo;
                split2(s.wu[r] * u0, s.wu[r + 1] * u1, hi, lo);
                *reinterpret_cast<uint32_t *>(u2h + vc * kLdP + r) = hi;
                *reinterpret_cast<uint32_t *>(u2l + vc * kLdP + r) = lo;
            }
        }
        __syncthreads();

        // ---- O = P U + scale gamma rq (Q S0), rows m0..m0+15
        {
            float acc[4][4];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
#pragma unroll
            for (int kk = 0; kk < kL / 16; ++kk) {
                if (kk > warp) break;
                uint32_t fh[4], fl[4];
                ldsm_x4(fh, s.ph + (m0 + (lane & 15)) * kLdP + kk * 16 + (lane >> 4) * 8);
                ldsm_x4(fl, s.pl + (m0 + (lane & 15)) * kLdP + kk * 16 + (lane >> 4) * 8);
#pragma unroll
                for (int np = 0; np < 2; ++np) {
                    uint32_t bh[4], bl[4];
                    const int off = (16 * np + (lane & 7) + ((lane >> 4) << 3)) * kLdP + kk * 16 + ((lane >> 3) & 1) * 8;
                    ldsm_x4(bh, s.uh + off);
                    ldsm_x4(bl, s.ul + off);
                    mma_bf16(acc[2 * np], fh, bh[0], bh[1]);
                    mma_bf16(acc[2 * np], fh, bl[0], bl[1]);
                    mma_bf16(acc[2 * np], fl, bh[0], bh[1]);
                    mma_bf16(acc[2 * np + 1], fh, bh[2], bh[3]);
                    mma_bf16(acc[2 * np + 1], fh, bl[2], bl[3]);
                    mma_bf16(acc[2 * np + 1], fl, bh[2], bh[3]);
                }
            }
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int row = m0 + gq + 8 * hh;
                if (row >= n) continue;
                const float w = p.scale * s.rq[row] * exp2f(s.gl2[row]);
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    const __nv_bfloat162 o2 = __floats2bfloat162_rn(acc[nt][2 * hh] + w * acc_o[nt][2 * hh],
                                                                    acc[nt][2 * hh + 1] + w * acc_o[nt][2 * hh + 1]);
                    *reinterpret_cast<__nv_bfloat162 *>(og + ((size_t)(t0 + row) * p.Hv + h) * V + v0 + 8 * nt +
                                                        2 * cq) = o2;
                }
            }
        }

        // ---- S = gamma_L S0 + K^T U'  (rows 32w..32w+31 of the state slice)
        {
            const float gl = exp2f(s.gl2[n - 1]);
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) st[mt][nt][e] *= gl;
#pragma unroll
            for (int ss = 0; ss < kL / 16; ++ss) {
                uint32_t bh[2][4], bl[2][4];
#pragma unroll
                for (int np = 0; np < 2; ++np) {
                    const int off = (16 * np + (lane & 7) + ((lane >> 4) << 3)) * kLdP + ss * 16 + ((lane >> 3) & 1) * 8;
                    ldsm_x4(bh[np], u2h + off);
                    ldsm_x4(bl[np], u2l + off);
                }
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    uint32_t fa[4];
                    const int mat = lane >> 3;
                    ldsm_x4_t(fa, s.k + (ss * 16 + (lane & 7) + ((mat >> 1) << 3)) * kLdK + 32 * warp + 16 * mt +
                                      ((mat & 1) << 3));
#pragma unroll
                    for (int np = 0; np < 2; ++np) {
                        mma_bf16(st[mt][2 * np], fa, bh[np][0], bh[np][1]);
                        mma_bf16(st[mt][2 * np], fa, bl[np][0], bl[np][1]);
                        mma_bf16(st[mt][2 * np + 1], fa, bh[np][2], bh[np][3]);
                        mma_bf16(st[mt][2 * np + 1], fa, bl[np][2], bl[np][3]);
                    }
                }
            }
        }

        // ---- state outputs at this chunk's end
        const int64_t abs_end = abs0 + n;
        if (io.chunk_states) write_state(io.chunk_states + ((size_t)(fc + j) * p.Hv + h) * state_elems);
        if (io.block_table && p.bs > 0 && abs_end % p.bs == 0) {
            const int64_t colb = abs_end / p.bs - 1;
            if (colb >= p.btw) {
                if (tid == 0) atomicOr(err, SSD_DEVERR_BLOCK_TABLE);
            } else {
                const int slot = io.block_table[(size_t)i * p.btw + colb];
                if (slot >= p.num_slots || !io.state_pool) {
                    if (tid == 0 && slot >= 0) atomicOr(err, SSD_DEVERR_BLOCK_SLOT);
                } else if (slot >= 0) {
                    write_state(io.state_pool + ((size_t)slot * p.Hv + h) * state_elems);
                }
            }
        }
        publish_state();
        pos += n;
        __syncthreads();
    }

    if (io.final_states) write_state(io.final_states + ((size_t)i * p.Hv + h) * state_elems);
    if (io.final_slots && io.state_pool) {
        const int fs = io.final_slots[i];
        if (fs >= p.num_slots) {
            if (tid == 0) atomicOr(err, SSD_DEVERR_FINAL_SLOT);
        } else if (fs >= 0) {
            write_state(io.state_pool + ((size_t)fs * p.Hv + h) * state_elems);
        }
    }
}

bool aligned_to(const void *ptr, uintptr_t al) { return ((uintptr_t)ptr & (al - 1)) == 0; }

}  // namespace
}  // namespace ssd

using namespace ssd;

extern "C" int ssd_varlen_gdn_forward(const ssd_gdn_dims *d, const int32_t *cu_seqlens, const ssd_gdn_io *io,
                                      cudaStream_t stream) {
    if (!d || !cu_seqlens || !io) return SSD_ERR_NULL;
    if (d->T < 0 || d->T > 0x7fffffffLL || d->R < 1 || d->Hk < 1 || d->Hv < 1 || d->num_slots < 0 ||
        d->block_table_width < 0)
        return SSD_ERR_DIMS;
    if (d->Hv % d->Hk != 0) return SSD_ERR_GROUPS;
    if (d->dtype != SSD_DTYPE_BF16 && d->dtype != SSD_DTYPE_F32) return SSD_ERR_DTYPE;
    if (d->dtype != SSD_DTYPE_BF16 || d->K != kK || d->V < kBV || d->V > 256 || d->V % kBV != 0)
        return SSD_ERR_UNSUPPORTED;
    if (d->chunk_size != kL) return SSD_ERR_UNSUPPORTED;
    if (io->block_table && (d->block_size <= 0 || d->block_size % kL != 0 || d->block_table_width < 1))
        return SSD_ERR_BLOCK_SIZE;
    if (!io->device_err) return SSD_ERR_NULL;
    if (d->T > 0 && (!io->q || !io->k || !io->v || !io->g || !io->beta || !io->o)) return SSD_ERR_NULL;
    if ((io->init_slots || io->final_slots || io->block_table) && (!io->state_pool || d->num_slots < 1))
        return SSD_ERR_NULL;
    const void *vec[] = {io->q, io->k, io->v, io->o, io->state_pool, io->final_states, io->chunk_states};
    for (const void *ptr : vec)
        if (ptr && !aligned_to(ptr, 16)) return SSD_ERR_ALIGN;
    const void *small[] = {cu_seqlens, io->g, io->beta, io->num_computed, io->init_slots, io->final_slots,
                           io->block_table, io->device_err};
    for (const void *ptr : small)
        if (ptr && !aligned_to(ptr, 4)) return SSD_ERR_ALIGN;
    if (gdn_tc_supported(d)) return launch_gdn_tc(d, cu_seqlens, io, stream);
    const int nvb = d->V / kBV;
    const int64_t ctas = (int64_t)d->R * d->Hv * nvb;
    if (ctas > 0x7fffffffLL) return SSD_ERR_DIMS;
    GdnParams p{};
    p.T = d->T;
    p.R = d->R;
    p.Hk = d->Hk;
    p.Hv = d->Hv;
    p.V = d->V;
    p.nvb = nvb;
    p.bs = io->block_table ? d->block_size : 0;
    p.btw = d->block_table_width;
    p.num_slots = d->num_slots;
    p.l2norm = d->l2norm ? 1 : 0;
    p.scale = d->scale != 0.f ? d->scale : 1.f / sqrtf((float)d->K);
    p.cu = cu_seqlens;
    p.io = *io;
    const int smem = (int)sizeof(GdnSmem);
    if (cudaFuncSetAttribute(gdn_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return SSD_ERR_CUDA;
    gdn_chunk_kernel<<<(unsigned)ctas, kThreads, smem, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}
