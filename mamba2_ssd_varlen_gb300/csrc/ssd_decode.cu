// ssd_decode.cu -- decode and speculative-decode step with dual read/write
// state anchors ("Automatic prefix caching for GDN hybrid models
// (mamba_cache_mode=all) with MTP speculative decoding", Purpose, the
// Kernels/layers bullet: the decode kernels read the previous step's running
// state from one slot while writing the current step's states to others).
//
// The same recurrence as the forward, for short per-request windows:
//   h   <- state_pool[read_slots[i]]  (zeros when the slot is < 0)
//   for each token t of request i:
//       dt' = softplus(dt[t,h] + dt_bias[h])
//       h   = exp(dt' A[h]) h + dt' x[t,h,:] (outer) B[t,g,:]
//       y[t,h,:] = (h C[t,g,:] + D[h] x[t,h,:]) * silu(z[t,h,:])
//       state_pool[write_slots[t]] <- h   when write_slots[t] >= 0
//
// One CTA of 256 threads per (request, head).  The (P, N) fp32 state lives in
// registers: thread k owns KV elements of one state row p (KV divides N, the
// N / KV threads of a row are adjacent lanes), in chunks of 4 columns
// interleaved with the row's other threads, so the state is read once and each
// write anchor is a run of 16-byte stores that fill whole sectors; the row's
// C.h dot product is a shuffle reduction over its lanes.  The window's B and C
// rows, the head's x row, dt', the decay and the write slot of up to
// kStageTok tokens are staged in shared memory by the whole CTA, so the P
// state rows that read the same values do so from shared memory and the
// global load path carries each value once.  The step is bound by the state
// traffic (4 P N bytes read, 4 P N per written anchor).
#include "pdl.cuh"
#include "ssd_internal.cuh"

namespace ssd {
namespace {

constexpr int kDecThreads = 256;
constexpr int kStageTok = 8;  // window tokens staged in shared memory at a time

// Shared-memory layout of one stage (bytes): B rows, C rows, x rows of the head,
// then dt', the decay and the write slot of each token.
struct DecStage {
    int off_c, off_x, off_f, bytes;
    __host__ __device__ DecStage(int N, int P, int esize) {
        const int nb = N * esize;  // a multiple of 32 (N a power of two >= 16)
        off_c = kStageTok * nb;
        off_x = 2 * kStageTok * nb;
        off_f = off_x + (kStageTok * P * esize + 15) / 16 * 16;
        bytes = off_f + 3 * kStageTok * 4;
    }
};

struct DecParams {
    int64_t T;
    int32_t R, H, P, N, G, num_slots;
    const int32_t *cu;
    ssd_decode_io io;
};

template <typename T>
__device__ __forceinline__ float ld_val(const void *base, size_t i) {
    return to_f32(static_cast<const T *>(base)[i]);
}

// A thread's KV state elements of row p are KV / CW chunks of CW = min(KV, 4)
// consecutive columns, chunk m at column CW (l + lanes m) for the thread's index l
// among the row's `lanes` threads: one 16-byte store instruction of a warp then
// writes lanes x 16 consecutive bytes of each row (whole 32-byte sectors)
// instead of 16 bytes every 4 KV.
template <int KV>
struct Chunks {
    static constexpr int CW = KV < 4 ? KV : 4;
    static constexpr int NC = KV / CW;
};

template <int KV>
__device__ __forceinline__ void load_row_chunks(const float *row, int col0, int stride, float (&h)[KV]) {
    constexpr int CW = Chunks<KV>::CW;
#pragma unroll
    for (int m = 0; m < Chunks<KV>::NC; ++m) {
        const float *src = row + col0 + m * stride;
        if constexpr (CW == 4) {
            const float4 q = *reinterpret_cast<const float4 *>(src);
            h[4 * m] = q.x;
            h[4 * m + 1] = q.y;
            h[4 * m + 2] = q.z;
            h[4 * m + 3] = q.w;
        } else {
#pragma unroll
            for (int c = 0; c < CW; ++c) h[CW * m + c] = src[c];
        }
    }
}

template <int KV>
__device__ __forceinline__ void store_row_chunks(float *row, int col0, int stride, const float (&h)[KV]) {
    constexpr int CW = Chunks<KV>::CW;
#pragma unroll
    for (int m = 0; m < Chunks<KV>::NC; ++m) {
        float *dst = row + col0 + m * stride;
        if constexpr (CW == 4) {
            *reinterpret_cast<float4 *>(dst) = make_float4(h[4 * m], h[4 * m + 1], h[4 * m + 2], h[4 * m + 3]);
        } else {
#pragma unroll
            for (int c = 0; c < CW; ++c) dst[c] = h[CW * m + c];
        }
    }
}

// The same chunks of a staged bf16 or fp32 B or C row, into fp32.
template <typename T, int KV>
__device__ __forceinline__ void load_vec_chunks(const T *row, int col0, int stride, float (&dst)[KV]) {
    constexpr int CW = Chunks<KV>::CW;
#pragma unroll
    for (int m = 0; m < Chunks<KV>::NC; ++m) {
        const T *src = row + col0 + m * stride;
        if constexpr (CW == 4 && sizeof(T) == 2) {
            const uint2 q = *reinterpret_cast<const uint2 *>(src);
            dst[4 * m] = __uint_as_float(q.x << 16);
            dst[4 * m + 1] = __uint_as_float(q.x & 0xFFFF0000u);
            dst[4 * m + 2] = __uint_as_float(q.y << 16);
            dst[4 * m + 3] = __uint_as_float(q.y & 0xFFFF0000u);
        } else if constexpr (CW == 4) {
            const float4 q = *reinterpret_cast<const float4 *>(src);
            dst[4 * m] = q.x;
            dst[4 * m + 1] = q.y;
            dst[4 * m + 2] = q.z;
            dst[4 * m + 3] = q.w;
        } else {
#pragma unroll
            for (int c = 0; c < CW; ++c) dst[CW * m + c] = to_f32(src[c]);
        }
    }
}

template <typename T, int KV>
// Four CTAs per SM up to KV = 32 (64 registers a thread: the bf16 instance fits,
// the fp32 one spills 12 bytes); KV = 64 keeps all the registers it needs.
__global__ void __launch_bounds__(kDecThreads, KV <= 32 ? 4 : 1) decode_kernel(const __grid_constant__ DecParams p) {
    pdl_wait();  // a dependent launch: the stream's previous kernel has finished
    const int i = blockIdx.x / p.H, hh = blockIdx.x % p.H;
    const int g = hh / (p.H / p.G);
    const int rowlanes = p.N / KV;                   // threads per state row (power of 2, <= 32)
    const int tl = threadIdx.x % rowlanes;           // this thread's index among them
    const bool active = (int)threadIdx.x < p.P * rowlanes;
    const int pr = active ? (int)threadIdx.x / rowlanes : 0;  // state row p
    constexpr int CW = Chunks<KV>::CW;
    const int col0 = CW * tl, cstride = CW * rowlanes;  // chunk m at column col0 + m cstride
    const size_t pn = (size_t)p.P * p.N, slot_elems = (size_t)p.H * pn;
    const size_t row_off = (size_t)hh * pn + (size_t)pr * p.N;
    const ssd_decode_io &io = p.io;

    const int64_t a = p.cu[i], b = p.cu[i + 1];
    if (b < a || a < 0 || b > p.T || (i == 0 && a != 0) || (i == p.R - 1 && b != p.T)) {
        if (threadIdx.x == 0 && hh == 0) atomicOr(io.device_err, SSD_DEVERR_CU_SEQLENS);
        return;
    }
    if (b == a) return;  // an empty window reads and writes nothing

    float h[KV];
    const int rs = io.read_slots[i];
    if (rs >= p.num_slots) {
        if (threadIdx.x == 0 && hh == 0) atomicOr(io.device_err, SSD_DEVERR_INIT_SLOT);
    }
    if (active && rs >= 0 && rs < p.num_slots) {
        load_row_chunks<KV>(io.state_pool + (size_t)rs * slot_elems + row_off, col0, cstride, h);
    } else {
#pragma unroll
        for (int j = 0; j < KV; ++j) h[j] = 0.f;
    }
    const float dtb = io.dt_bias[hh], Ah = io.A[hh];
    const float Dh = io.D ? io.D[hh] : 0.f;
    const T *Bv = static_cast<const T *>(io.B);
    const T *Cv = static_cast<const T *>(io.C);
    const T *Xv = static_cast<const T *>(io.x);
    extern __shared__ __align__(16) uint8_t dec_smem[];
    const DecStage L(p.N, p.P, (int)sizeof(T));
    const T *sB = reinterpret_cast<const T *>(dec_smem);
    const T *sC = reinterpret_cast<const T *>(dec_smem + L.off_c);
    T *sX = reinterpret_cast<T *>(dec_smem + L.off_x);
    float *sDtp = reinterpret_cast<float *>(dec_smem + L.off_f);
    float *sDec = sDtp + kStageTok;
    int *sWs = reinterpret_cast<int *>(sDec + kStageTok);
    const int vrow = p.N * (int)sizeof(T) / 16;  // 16-byte vectors per B or C row
    for (int64_t tc = a; tc < b; tc += kStageTok) {
        const int nt = (int)min((int64_t)kStageTok, b - tc);
        // ---- stage tokens tc .. tc+nt-1 (every thread, active or not)
        for (int v = threadIdx.x; v < 2 * nt * vrow; v += kDecThreads) {
            const int cmat = v / (nt * vrow), rem = v % (nt * vrow);
            const int tt = rem / vrow, c = rem % vrow;
            const T *src = (cmat ? Cv : Bv) + ((size_t)(tc + tt) * p.G + g) * p.N;
            reinterpret_cast<uint4 *>(dec_smem + (cmat ? L.off_c : 0) + (size_t)tt * p.N * sizeof(T))[c] =
                reinterpret_cast<const uint4 *>(src)[c];
        }
        for (int v = threadIdx.x; v < nt * p.P; v += kDecThreads) {
            const int tt = v / p.P, c = v % p.P;
            sX[v] = Xv[((size_t)(tc + tt) * p.H + hh) * p.P + c];
        }
        if (threadIdx.x < nt) {
            const int64_t t = tc + threadIdx.x;
            const float dtp = softplus_f32(ld_val<T>(io.dt, (size_t)t * p.H + hh) + dtb);
            sDtp[threadIdx.x] = dtp;
            sDec[threadIdx.x] = expf(dtp * Ah);
            sWs[threadIdx.x] = io.write_slots ? io.write_slots[t] : -1;
        }
        __syncthreads();
        for (int tt = 0; tt < nt; ++tt) {
            const int64_t t = tc + tt;
            const float dtp = sDtp[tt], decay = sDec[tt];
            const size_t xi = ((size_t)t * p.H + hh) * p.P + pr;
            const float xv = active ? to_f32(sX[tt * p.P + pr]) : 0.f;
            const float coef = dtp * xv;
            float acc = 0.f;
            if (active) {
                float bv[KV], cv[KV];
                load_vec_chunks<T, KV>(sB + (size_t)tt * p.N, col0, cstride, bv);
                load_vec_chunks<T, KV>(sC + (size_t)tt * p.N, col0, cstride, cv);
#pragma unroll
                for (int j = 0; j < KV; ++j) {
                    h[j] = fmaf(decay, h[j], coef * bv[j]);
                    acc = fmaf(cv[j], h[j], acc);
                }
            }
            // the row's C.h over its rowlanes adjacent lanes
            for (int o = rowlanes >> 1; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (active && tl == 0) {
                float yv = fmaf(Dh, xv, acc);
                if (io.z) yv *= silu_f32(ld_val<T>(io.z, xi));
                static_cast<T *>(io.y)[xi] = from_f32<T>(yv);
            }
            const int ws = sWs[tt];
            if (ws >= p.num_slots) {
                if (threadIdx.x == 0 && hh == 0) atomicOr(io.device_err, SSD_DEVERR_FINAL_SLOT);
            } else if (ws >= 0 && active) {
                store_row_chunks<KV>(io.state_pool + (size_t)ws * slot_elems + row_off, col0, cstride, h);
            }
        }
        __syncthreads();  // the stage is rewritten by the next tokens
    }
}

template <typename T>
cudaError_t launch_decode_t(const DecParams &p, int kv, cudaStream_t stream) {
    const dim3 grid((unsigned)((int64_t)p.R * p.H)), block(kDecThreads);
    const size_t smem = (size_t)DecStage(p.N, p.P, (int)sizeof(T)).bytes;
    switch (kv) {
        case 1: return launch_after_prev(decode_kernel<T, 1>, grid, block, smem, stream, p);
        case 2: return launch_after_prev(decode_kernel<T, 2>, grid, block, smem, stream, p);
        case 4: return launch_after_prev(decode_kernel<T, 4>, grid, block, smem, stream, p);
        case 8: return launch_after_prev(decode_kernel<T, 8>, grid, block, smem, stream, p);
        case 16: return launch_after_prev(decode_kernel<T, 16>, grid, block, smem, stream, p);
        case 32: return launch_after_prev(decode_kernel<T, 32>, grid, block, smem, stream, p);
        case 64: return launch_after_prev(decode_kernel<T, 64>, grid, block, smem, stream, p);
        default: return cudaErrorInvalidValue;
    }
}

// State elements per thread: the smallest power of two that spreads the (P, N)
// state over the CTA with a row split over at most 32 adjacent lanes.
int pick_kv(int P, int N) {
    const int64_t elems = (int64_t)P * N;
    for (int kv = 1; kv <= 64; kv <<= 1) {
        if (N % kv != 0 || N / kv > 32) continue;
        if (elems <= (int64_t)kDecThreads * kv) return kv;
    }
    return 0;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }
bool aligned4(const void *p) { return ((uintptr_t)p & 3u) == 0; }

}  // namespace
}  // namespace ssd

using namespace ssd;

extern "C" int ssd_varlen_decode(const ssd_dims *d, const int32_t *cu_seqlens, const ssd_decode_io *io,
                                 cudaStream_t stream) {
    if (!d || !cu_seqlens || !io) return SSD_ERR_NULL;
    if (d->reserved != 0) return SSD_ERR_DIMS;
    if (d->T < 0 || d->T > 0x7fffffffLL || d->R < 1 || d->H < 1 || d->P < 1 || d->N < 1 || d->G < 1 ||
        d->num_slots < 1 || d->H > 65535 || (int64_t)d->R * d->H > 0x7fffffffLL)
        return SSD_ERR_DIMS;
    if (d->H % d->G != 0) return SSD_ERR_GROUPS;
    if (d->dtype != SSD_DTYPE_BF16 && d->dtype != SSD_DTYPE_F32) return SSD_ERR_DTYPE;
    if ((d->N & (d->N - 1)) != 0 || d->N < 16 || d->N > 256) return SSD_ERR_UNSUPPORTED;
    const int kv = pick_kv(d->P, d->N);
    if (kv == 0) return SSD_ERR_UNSUPPORTED;
    if (!io->dt_bias || !io->A || !io->state_pool || !io->read_slots || !io->device_err) return SSD_ERR_NULL;
    // with no tokens (every window empty) the token buffers may be NULL
    if (d->T > 0 && (!io->x || !io->dt || !io->B || !io->C || !io->y)) return SSD_ERR_NULL;
    const void *big[] = {io->x, io->dt, io->B, io->C, io->z, io->y, io->state_pool};
    for (const void *ptr : big)
        if (ptr && !aligned16(ptr)) return SSD_ERR_ALIGN;
    const void *small[] = {cu_seqlens, io->dt_bias, io->A, io->D, io->read_slots, io->write_slots, io->device_err};
    for (const void *ptr : small)
        if (ptr && !aligned4(ptr)) return SSD_ERR_ALIGN;
    DecParams p{};
    p.T = d->T;
    p.R = d->R;
    p.H = d->H;
    p.P = d->P;
    p.N = d->N;
    p.G = d->G;
    p.num_slots = d->num_slots;
    p.cu = cu_seqlens;
    p.io = *io;
    const cudaError_t e = d->dtype == SSD_DTYPE_BF16 ? launch_decode_t<__nv_bfloat16>(p, kv, stream)
                                                     : launch_decode_t<float>(p, kv, stream);
    return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}
