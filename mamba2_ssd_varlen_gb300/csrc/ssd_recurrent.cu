// ssd_recurrent.cu -- token-serial SSD scan on CUDA cores.
//
// The general path: any dtype (fp32 or bf16), any P, N up to 256.  It runs
// the recurrence of the SSD scan directly, one token after the other, with the
// (P x N) state of one (request, head) held in registers across a CTA:
//     h = exp(dt' A) h + dt' x (outer) B ;  y = (h C + D x) * silu(z)
// Each warp owns 2 rows p of the state and each lane N/32 columns n, so a
// token costs two fused multiply-adds per state element plus a warp-shuffle
// reduction per row.  fp32 throughout; no rounding of intermediate operands.
// Requests restart from their own initial state (pool slot or zeros), which
// decays from the request's first token (the initial-state decay fix of the
// "[Bugfix] Mamba2 SSD varlen bug fix initstates decay" page).  State outputs
// (chunk export, block checkpoints, finals) are written at the token where
// the absolute position crosses the boundary.
#include "ssd_internal.cuh"

namespace ssd {
namespace {

constexpr int kRecThreads = 256;
constexpr int kRowsPerWarp = 2;
constexpr int kRowsPerCta = kRowsPerWarp * (kRecThreads / 32);

template <int NPL>
__device__ __forceinline__ void store_state_rows(float *slot_base, const FwdParams &p, int h, int prow0,
                                                 const bool (&rowv)[kRowsPerWarp], int n0, bool nv,
                                                 const float (&st)[kRowsPerWarp][NPL]) {
    if (!nv) return;
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        if (!rowv[r]) continue;
        float *dst = slot_base + ((size_t)h * p.P + prow0 + r) * p.N + n0;
#pragma unroll
        for (int k = 0; k < NPL; ++k) dst[k] = st[r][k];
    }
}

template <typename Tin, int NPL>
__global__ void __launch_bounds__(kRecThreads) recurrent_kernel(const FwdParams p) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int PB = (p.P + kRowsPerCta - 1) / kRowsPerCta;
    int64_t bid = blockIdx.x;
    const int pb = (int)(bid % PB);
    bid /= PB;
    const int h = (int)(bid % p.H);
    const int i = (int)(bid / p.H);
    if (i >= p.R || p.hdr[kHdrSegs] == 0) return;  // plan rejected the batch

    const Tin *__restrict__ x = static_cast<const Tin *>(p.x);
    const Tin *__restrict__ dtv = static_cast<const Tin *>(p.dt);
    const Tin *__restrict__ Bv = static_cast<const Tin *>(p.B);
    const Tin *__restrict__ Cv = static_cast<const Tin *>(p.C);
    const Tin *__restrict__ zv = static_cast<const Tin *>(p.z);
    Tin *__restrict__ y = static_cast<Tin *>(p.y);

    const int g = h / (p.H / p.G);
    const int64_t a = p.cu_seqlens[i];
    const int64_t L = (int64_t)p.cu_seqlens[i + 1] - a;
    const int64_t s = p.num_computed ? (int64_t)p.num_computed[i] : 0;
    const int prow0 = pb * kRowsPerCta + warp * kRowsPerWarp;
    bool rowv[kRowsPerWarp];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) rowv[r] = prow0 + r < p.P;
    const int n0 = lane * NPL;
    const bool nv = n0 < p.N;
    const size_t slot_elems = (size_t)p.H * p.P * p.N;

    int slot = -1;
    if (p.init_slots) {
        slot = p.init_slots[i];
        if (slot >= p.num_slots) {
            if (pb == 0 && threadIdx.x == 0) set_err(p.hdr, SSD_DEVERR_INIT_SLOT);
            slot = -1;
        }
    }
    float st[kRowsPerWarp][NPL];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
        for (int k = 0; k < NPL; ++k)
            st[r][k] = (slot >= 0 && rowv[r] && nv)
                           ? p.pool[slot * slot_elems + ((size_t)h * p.P + prow0 + r) * p.N + n0 + k]
                           : 0.f;

    const float dtb = p.dt_bias[h], Ah = p.A[h], Dh = p.D ? p.D[h] : 0.f;
    const int64_t first_row = p.chunk_states ? (int64_t)p.req_first_chunk[i] - s / p.Q : 0;
    // Inputs of the next token are loaded one iteration ahead (the loop is
    // latency-bound: one dependent state update per token).
    float n_dt = 0.f, n_x[kRowsPerWarp], n_b[NPL], n_c[NPL];
    auto load_token = [&](int64_t t) {
        n_dt = to_f32(dtv[t * p.H + h]);
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r)
            n_x[r] = rowv[r] ? to_f32(x[((size_t)t * p.H + h) * p.P + prow0 + r]) : 0.f;
        const size_t bc = ((size_t)t * p.G + g) * p.N + n0;
#pragma unroll
        for (int q = 0; q < NPL; ++q) {
            n_b[q] = nv ? to_f32(Bv[bc + q]) : 0.f;
            n_c[q] = nv ? to_f32(Cv[bc + q]) : 0.f;
        }
    };
    if (L > 0) load_token(a);
    for (int64_t k = 0; k < L; ++k) {
        const int64_t t = a + k;
        const float dtp = softplus_f32(n_dt + dtb);
        const float dec = expf(dtp * Ah);
        float xv[kRowsPerWarp], bv[NPL], cv[NPL];
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) xv[r] = n_x[r];
#pragma unroll
        for (int q = 0; q < NPL; ++q) {
            bv[q] = n_b[q];
            cv[q] = n_c[q];
        }
        if (k + 1 < L) load_token(t + 1);
        float acc[kRowsPerWarp];
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
            const float u = dtp * xv[r];
            float sum = 0.f;
#pragma unroll
            for (int q = 0; q < NPL; ++q) {
                st[r][q] = fmaf(dec, st[r][q], u * bv[q]);
                sum = fmaf(st[r][q], cv[q], sum);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
            acc[r] = sum;
        }
        if (lane < kRowsPerWarp) {
            const int r = lane;
            const float xr = (r == 0) ? xv[0] : xv[kRowsPerWarp - 1];
            float v = ((r == 0) ? acc[0] : acc[kRowsPerWarp - 1]) + Dh * xr;
            if (prow0 + r < p.P) {
                const size_t yi = ((size_t)t * p.H + h) * p.P + prow0 + r;
                if (zv) v *= silu_f32(to_f32(zv[yi]));
                y[yi] = from_f32<Tin>(v);
            }
        }
        const int64_t pos = s + k + 1;  // absolute position just after this token
        if (p.chunk_states && (pos % p.Q == 0 || k + 1 == L)) {
            const int64_t row = first_row + (pos - 1) / p.Q;
            store_state_rows<NPL>(p.chunk_states + row * slot_elems, p, h, prow0, rowv, n0, nv, st);
        }
        if (p.block_table && p.block_size > 0 && pos % p.block_size == 0) {
            const int64_t col = pos / p.block_size - 1;
            if (col >= p.bt_width) {
                if (pb == 0 && threadIdx.x == 0) set_err(p.hdr, SSD_DEVERR_BLOCK_TABLE);
            } else {
                const int bslot = p.block_table[(size_t)i * p.bt_width + col];
                if (bslot >= p.num_slots) {
                    if (pb == 0 && threadIdx.x == 0) set_err(p.hdr, SSD_DEVERR_BLOCK_SLOT);
                } else if (bslot >= 0) {
                    store_state_rows<NPL>(p.pool + (size_t)bslot * slot_elems, p, h, prow0, rowv, n0, nv, st);
                }
            }
        }
    }
    if (p.final_states)
        store_state_rows<NPL>(p.final_states + (size_t)i * slot_elems, p, h, prow0, rowv, n0, nv, st);
    if (p.final_slots) {
        const int fslot = p.final_slots[i];
        if (fslot >= p.num_slots) {
            if (pb == 0 && threadIdx.x == 0) set_err(p.hdr, SSD_DEVERR_FINAL_SLOT);
        } else if (fslot >= 0) {
            store_state_rows<NPL>(p.pool + (size_t)fslot * slot_elems, p, h, prow0, rowv, n0, nv, st);
        }
    }
}

template <typename Tin>
cudaError_t launch_t(const FwdParams &p, cudaStream_t stream) {
    const int PB = (p.P + kRowsPerCta - 1) / kRowsPerCta;
    const int64_t blocks = (int64_t)p.R * p.H * PB;
    if (blocks == 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const int npl = p.N <= 32 ? 1 : p.N / 32;
    switch (npl) {
#define SSD_REC_CASE(K) \
    case K: recurrent_kernel<Tin, K><<<(unsigned)blocks, kRecThreads, 0, stream>>>(p); break;
        SSD_REC_CASE(1)
        SSD_REC_CASE(2)
        SSD_REC_CASE(3)
        SSD_REC_CASE(4)
        SSD_REC_CASE(5)
        SSD_REC_CASE(6)
        SSD_REC_CASE(7)
        SSD_REC_CASE(8)
#undef SSD_REC_CASE
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_recurrent(const FwdParams &p, int dtype, cudaStream_t stream) {
    return dtype == SSD_DTYPE_F32 ? launch_t<float>(p, stream) : launch_t<__nv_bfloat16>(p, stream);
}

}  // namespace ssd
