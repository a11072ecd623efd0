// ssd_conv1d.cu -- varlen causal depthwise conv1d with conv-state anchors, the
// step before the SSD in a Mamba2 layer ("[Model] Mamba2 varlen and metadata
// refactor", Purpose items 1-2: packed varlen inputs; the causal_conv1d decode
// kernel with dual read/write state anchors of "Automatic prefix caching for
// GDN hybrid models (mamba_cache_mode=all) with MTP speculative decoding",
// Purpose, Kernels/layers).
//
//   xin      = [conv state (W-1 inputs, oldest first), the request's inputs]
//   y[t, c]  = act(bias[c] + sum_k weight[c, k] xin[t - (W-1) + k, c])
//   new conv state = the last W-1 values of xin
//
// Streaming and HBM-bound: a warp takes a strip of consecutive tokens over 32 x kN
// channels; each thread owns one 16-byte vector of kN channels and slides a
// W-deep register window down the strip, so every input and output row is one
// coalesced vector access and every input is read once (plus a W-1 halo per
// strip).  Request boundaries inside a strip restart the window from the next
// request's conv state.
#include "pdl.cuh"
#include "ssd_internal.cuh"

namespace ssd {
namespace {

constexpr int kConvThreads = 128;
constexpr int kMinStrip = 64;  // tokens per warp at least, when the grid need not fill the GPU
constexpr int kMaxDevices = 64;

struct ConvParams {
    int64_t T;
    int32_t R, D, W, num_slots, silu;
    const int32_t *cu;
    ssd_conv_io io;
};

template <typename T>
struct Vec {  // one 16-byte vector of channels
    static constexpr int kN = 16 / sizeof(T);
    float v[kN];
    __device__ __forceinline__ void load(const T *p) { set(*reinterpret_cast<const uint4 *>(p)); }
    __device__ __forceinline__ void set(const uint4 q) {
        if constexpr (sizeof(T) == 2) {
            const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                v[2 * e] = __uint_as_float(w[e] << 16);
                v[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
            }
        } else {
            v[0] = __uint_as_float(q.x);
            v[1] = __uint_as_float(q.y);
            v[2] = __uint_as_float(q.z);
            v[3] = __uint_as_float(q.w);
        }
    }
    __device__ __forceinline__ void store(T *p) const {
        uint4 q;
        if constexpr (sizeof(T) == 2) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const __nv_bfloat162 b2 = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
                w[e] = *reinterpret_cast<const uint32_t *>(&b2);
            }
            q = make_uint4(w[0], w[1], w[2], w[3]);
        } else {
            q = make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]), __float_as_uint(v[3]));
        }
        *reinterpret_cast<uint4 *>(p) = q;
    }
    __device__ __forceinline__ void zero() {
#pragma unroll
        for (int e = 0; e < kN; ++e) v[e] = 0.f;
    }
};

// Conv state of kN channels c0.. of one slot: (W-1) values per channel, channel
// major (kN * (W-1) consecutive elements); win[k+1] holds the k-th oldest input.
template <typename T, int W>
__device__ __forceinline__ void store_conv_state(T *slot, int c0, const Vec<T> (&win)[W]) {
    constexpr int kN = Vec<T>::kN;
    T *dst = slot + (size_t)c0 * (W - 1);
#pragma unroll
    for (int e = 0; e < kN; ++e)
#pragma unroll
        for (int k = 0; k < W - 1; ++k) dst[e * (W - 1) + k] = from_f32<T>(win[k + 1].v[e]);
}

// The request holding token t: the last i with cu[i] <= t < cu[i+1].
__device__ __forceinline__ int request_of(const int32_t *cu, int R, int64_t t) {
    int lo = 0, hi = R;  // invariant: cu[lo] <= t, answer in [lo, hi)
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if ((int64_t)cu[mid] <= t) lo = mid;
        else hi = mid;
    }
    return lo;
}

// Packed fp32 pairs (one 64-bit register pair) for the f32x2 instructions: two
// channels per fused multiply-add.
__device__ __forceinline__ uint64_t pair(float a, float b) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(a), "f"(b));
    return d;
}
__device__ __forceinline__ void unpair(uint64_t d, float &a, float &b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(d));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
// SiLU of a pair from half its argument, h = v / 2: v * sigmoid(v) = h (1 + tanh h),
// one tanh per value on the special-function unit and one packed multiply-add.
// The caller feeds h by convolving with halved taps and bias (a power-of-two
// scaling, exact).  tanh.approx.f32 is good to about 2^-11, so the result is off
// by at most about |h| 2^-11: h is first raised to -8 at least, which keeps that
// below 3.9e-3 (inside the 5e-3 absolute tolerance) where SiLU is near zero --
// below v = -16 SiLU is smaller than 2e-6 -- and for large positive h it is a
// relative 2^-12.
__device__ __forceinline__ uint64_t silu_of_half_pair(uint64_t h) {
    float a, b;
    unpair(h, a, b);
    a = fmaxf(a, -8.f);
    b = fmaxf(b, -8.f);
    float ta, tb;
    asm("tanh.approx.f32 %0, %1;" : "=f"(ta) : "f"(a));
    asm("tanh.approx.f32 %0, %1;" : "=f"(tb) : "f"(b));
    const uint64_t hc = pair(a, b);
    return fma2(hc, pair(ta, tb), hc);
}

// 16-byte asynchronous global -> shared copy that bypasses L1 (the input is
// streamed once), with commit / wait on the issuing thread's copy groups.
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(smem)), "l"(gmem)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int kPending>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(kPending) : "memory"); }

constexpr int kStages = 16;  // input rows in flight per thread
constexpr int kUnroll = 6;   // a multiple of W-1 for every W, so the window shifts by renaming

// Work units are (channel group g, token t), g major; channel group g is the 32
// consecutive 16-byte channel vectors g*32 .. g*32+31 (lane l the vector g*32+l).
// The grid is what stays resident on the GPU at once, and its warps split the
// units evenly in order: every warp streams one strip (two where its strip
// crosses into the next channel group), so there is no tail wave and each warp
// fills its input ring once per strip.  Each thread streams its inputs through a
// private kStages-deep ring in shared memory filled by asynchronous copies, so
// the loads in flight cost no registers; only the W-1 previous inputs stay in
// registers.
template <typename T, int W, bool kSilu>
__global__ void __launch_bounds__(kConvThreads) conv1d_kernel(const __grid_constant__ ConvParams p) {
    pdl_wait();  // a dependent launch: the stream's previous kernel has finished
    constexpr int kN = Vec<T>::kN;
    __shared__ __align__(16) uint4 ring[kStages][kConvThreads];
    const ssd_conv_io &io = p.io;
    const int nvec = p.D / kN;
    const int groups = (nvec + 31) / 32;
    const int64_t t_units = p.T > 0 ? p.T : 1;  // one unit per group when T = 0 (empty requests)
    const int64_t units = (int64_t)groups * t_units;
    const int64_t nwarps = (int64_t)gridDim.x * (kConvThreads / 32);
    const int64_t wid = (int64_t)blockIdx.x * (kConvThreads / 32) + (threadIdx.x >> 5);
    const T *__restrict__ xv = static_cast<const T *>(io.x);
    T *__restrict__ yv = static_cast<T *>(io.y);
    T *pool = static_cast<T *>(io.conv_pool);
    const size_t slot_elems = (size_t)p.D * (W - 1);
    const size_t row = (size_t)p.D;
    uint4 *mine = &ring[0][threadIdx.x];  // stage s at mine[s * kConvThreads]

    // cu_seqlens must start at 0, not decrease and end at T (checked once).
    if (blockIdx.x == 0) {
        for (int i = threadIdx.x; i < p.R; i += kConvThreads)
            if (p.cu[i + 1] < p.cu[i] || (i == 0 && p.cu[0] != 0) || (i == p.R - 1 && p.cu[p.R] != p.T))
                atomicOr(io.device_err, SSD_DEVERR_CU_SEQLENS);
    }

    int64_t u = wid * units / nwarps;
    const int64_t u_end = (wid + 1) * units / nwarps;
    while (u < u_end) {
        const int g = (int)(u / t_units);
        const int64_t t0 = u % t_units;
        const int n_units = (int)min(u_end - u, t_units - t0);
        u += n_units;
        const int c0 = (g * 32 + (threadIdx.x & 31)) * kN;  // first channel of this thread
        if (c0 >= p.D) continue;

        auto state_slot = [&](const int32_t *slots, int i, int bit) -> T * {
            if (!slots || !pool) return nullptr;
            const int s = slots[i];
            if (s >= p.num_slots) {
                if (c0 == 0) atomicOr(io.device_err, bit);
                return nullptr;
            }
            return s >= 0 ? pool + (size_t)s * slot_elems : nullptr;
        };

        // An empty request's conv state passes through (the strip holding token 0 does it).
        if (t0 == 0) {
            for (int i = 0; i < p.R; ++i) {
                if (p.cu[i + 1] != p.cu[i]) continue;
                T *dst = state_slot(io.write_slots, i, SSD_DEVERR_FINAL_SLOT);
                if (!dst) continue;
                const T *src = state_slot(io.read_slots, i, SSD_DEVERR_INIT_SLOT);
                for (int e = 0; e < kN * (W - 1); ++e)
                    dst[(size_t)c0 * (W - 1) + e] = src ? src[(size_t)c0 * (W - 1) + e] : from_f32<T>(0.f);
            }
        }
        if (t0 >= p.T) continue;
        const int n = n_units;  // tokens of this strip
        const T *xt = xv + (size_t)t0 * row + c0;  // this thread's vector of token t0
        T *yt = yv + (size_t)t0 * row + c0;

#pragma unroll
        for (int s = 0; s < kStages; ++s) {  // one copy group per stage, empty past the strip
            if (s < n) cp_async16(mine + s * kConvThreads, xt + (size_t)s * row);
            cp_async_commit();
        }

        float wt[W][kN], bs[kN];
#pragma unroll
        for (int e = 0; e < kN; ++e) {
            // with SiLU the sum is formed at half scale (silu_of_half_pair)
            constexpr float kScale = kSilu ? 0.5f : 1.f;
            bs[e] = io.bias ? kScale * io.bias[c0 + e] : 0.f;
#pragma unroll
            for (int k = 0; k < W; ++k) wt[k][e] = kScale * io.weight[(size_t)(c0 + e) * W + k];
        }

        // window: win[0..W-2] the W-1 inputs before token t, win[W-1] token t
        Vec<T> win[W];
        int i = request_of(p.cu, p.R, t0);
        int64_t rs = p.cu[i];
        int rel_end = (int)min((int64_t)p.cu[i + 1] - t0, (int64_t)n + 1);  // request end, strip-relative
        auto enter = [&](int64_t t) {  // fill win[0..W-2] with the inputs before t in its request
            const T *src = nullptr;
            if (t - rs < W - 1) src = state_slot(io.read_slots, i, SSD_DEVERR_INIT_SLOT);
#pragma unroll
            for (int k = 0; k < W - 1; ++k) {
                const int64_t v = t - (W - 1) + k;
                if (v >= rs && v >= 0) {
                    win[k].load(xv + (size_t)v * row + c0);
                } else if (src) {
                    const int j = (int)(W - 1 - (rs - v));  // index in the conv state, oldest first
#pragma unroll
                    for (int e = 0; e < kN; ++e) win[k].v[e] = to_f32(src[(size_t)(c0 + e) * (W - 1) + j]);
                } else {
                    win[k].zero();
                }
            }
        };
        enter(t0);
        for (int jb = 0; jb < n; jb += kUnroll) {
            const int sb = jb % kStages;
#pragma unroll
            for (int q = 0; q < kUnroll; ++q) {
                const int j = jb + q;
                if (j >= n) break;
                if (j == rel_end) {  // the next non-empty request starts here
                    const int64_t t = t0 + j;
                    while (i + 1 < p.R && p.cu[i + 1] <= t) ++i;
                    rs = p.cu[i];
                    rel_end = (int)min((int64_t)p.cu[i + 1] - t0, (int64_t)n + 1);
                    enter(t);
                }
                const int st = sb + q < kStages ? sb + q : sb + q - kStages;
                cp_async_wait<kStages - 1>();  // token j's copy group has landed
                win[W - 1].set(mine[st * kConvThreads]);
                Vec<T> out;
#pragma unroll
                for (int e = 0; e < kN; e += 2) {  // two channels per packed instruction
                    uint64_t acc = pair(bs[e], bs[e + 1]);
#pragma unroll
                    for (int k = 0; k < W; ++k)
                        acc = fma2(pair(wt[k][e], wt[k][e + 1]), pair(win[k].v[e], win[k].v[e + 1]), acc);
                    if (kSilu) acc = silu_of_half_pair(acc);
                    unpair(acc, out.v[e], out.v[e + 1]);
                }
                out.store(yt + (size_t)j * row);
                if (j + 1 == rel_end) {  // the request's last token: its conv state goes out
                    T *dst = state_slot(io.write_slots, i, SSD_DEVERR_FINAL_SLOT);
                    if (dst) store_conv_state<T, W>(dst, c0, win);
                }
                // refill the stage just read (its value is consumed above)
                if (j + kStages < n) cp_async16(mine + st * kConvThreads, xt + (size_t)(j + kStages) * row);
                cp_async_commit();
#pragma unroll
                for (int k = 0; k < W - 1; ++k) win[k] = win[k + 1];
            }
        }
        cp_async_wait<0>();  // the ring is free for the next strip
    }
}

// CTAs of one conv kernel that fit on the current device at once (queried once
// per device).
template <typename T, int W, bool kSilu>
cudaError_t conv_resident_ctas(int64_t &out) {
    static int64_t cached[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const bool cacheable = dev >= 0 && dev < kMaxDevices;
    if (cacheable && cached[dev] > 0) {
        out = cached[dev];
        return cudaSuccess;
    }
    int per_sm = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, conv1d_kernel<T, W, kSilu>, kConvThreads, 0);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (per_sm < 1 || sms < 1) return cudaErrorInvalidConfiguration;
    out = (int64_t)per_sm * sms;
    if (cacheable) cached[dev] = out;
    return cudaSuccess;
}

// The grid: every resident CTA, or fewer when the strips would fall below
// kMinStrip units a warp.
template <typename T, int W, bool kSilu>
cudaError_t launch_conv_k(const ConvParams &p, int64_t units, cudaStream_t stream) {
    int64_t resident = 0;
    const cudaError_t e = conv_resident_ctas<T, W, kSilu>(resident);
    if (e != cudaSuccess) return e;
    const int64_t warps = (units + kMinStrip - 1) / kMinStrip;
    const int64_t ctas = std::max<int64_t>(1, std::min(resident, (warps + kConvThreads / 32 - 1) / (kConvThreads / 32)));
    return launch_after_prev(conv1d_kernel<T, W, kSilu>, dim3((unsigned)ctas), dim3(kConvThreads), 0, stream, p);
}

template <typename T, int W>
cudaError_t launch_conv_w(const ConvParams &p, int64_t units, cudaStream_t stream) {
    return p.silu ? launch_conv_k<T, W, true>(p, units, stream) : launch_conv_k<T, W, false>(p, units, stream);
}

template <typename T>
cudaError_t launch_conv_t(const ConvParams &p, cudaStream_t stream) {
    constexpr int kN = 16 / sizeof(T);
    const int64_t groups = (p.D / kN + 31) / 32;
    const int64_t units = groups * (p.T > 0 ? p.T : 1);  // as the kernel counts them
    switch (p.W) {
        case 2: return launch_conv_w<T, 2>(p, units, stream);
        case 3: return launch_conv_w<T, 3>(p, units, stream);
        case 4: return launch_conv_w<T, 4>(p, units, stream);
        default: return cudaErrorInvalidValue;
    }
}

bool aligned_to(const void *p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

}  // namespace
}  // namespace ssd

using namespace ssd;

extern "C" int ssd_varlen_conv1d(const ssd_conv_dims *d, const int32_t *cu_seqlens, const ssd_conv_io *io,
                                 cudaStream_t stream) {
    if (!d || !cu_seqlens || !io) return SSD_ERR_NULL;
    if (d->T < 0 || d->T > 0x7fffffffLL || d->R < 1 || d->D < 1 || d->num_slots < 0) return SSD_ERR_DIMS;
    if (d->dtype != SSD_DTYPE_BF16 && d->dtype != SSD_DTYPE_F32) return SSD_ERR_DTYPE;
    if (d->W < 2 || d->W > 4 || d->D % 8 != 0) return SSD_ERR_UNSUPPORTED;
    if (!io->weight || !io->device_err) return SSD_ERR_NULL;
    if (d->T > 0 && (!io->x || !io->y)) return SSD_ERR_NULL;  // optional with no tokens
    const bool uses_pool = io->read_slots || io->write_slots;
    if (uses_pool && (!io->conv_pool || d->num_slots < 1)) return SSD_ERR_NULL;
    const void *vec[] = {io->x, io->y, io->conv_pool};
    for (const void *ptr : vec)
        if (ptr && !aligned_to(ptr, 16)) return SSD_ERR_ALIGN;
    const void *small[] = {cu_seqlens, io->weight, io->bias, io->read_slots, io->write_slots, io->device_err};
    for (const void *ptr : small)
        if (ptr && !aligned_to(ptr, 4)) return SSD_ERR_ALIGN;
    ConvParams p{};
    p.T = d->T;
    p.R = d->R;
    p.D = d->D;
    p.W = d->W;
    p.num_slots = d->num_slots;
    p.silu = d->silu ? 1 : 0;
    p.cu = cu_seqlens;
    p.io = *io;
    const cudaError_t e = d->dtype == SSD_DTYPE_BF16 ? launch_conv_t<__nv_bfloat16>(p, stream)
                                                     : launch_conv_t<float>(p, stream);
    return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}
