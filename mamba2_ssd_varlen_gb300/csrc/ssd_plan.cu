// ssd_plan.cu -- device-side varlen metadata builder, run once per batch.
//
// "[Model] Mamba2 varlen and metadata refactor", Purpose item 2: the varlen
// metadata is computed once while the batch is prepared, not inside the first
// layer's forward.  Here that metadata is, from cu_seqlens (and the optional
// num_computed_tokens of each request):
//   * req_first_chunk[i]: the request's first row in the chunk-state export
//     (exclusive prefix sum of chunk counts; chunks cut at absolute multiples
//     of chunk_size, so a resumed request's first chunk may be partial);
//   * req_first_seg[i] and the segment list: runs of at most seg_len tokens
//     (2048, or 8192 on the one-head path) that the forward kernels walk, cut at
//     absolute multiples of seg_len or, for batches of mid-length requests,
//     tail-shortened (SegCuts below);
//   * how the state is carried from one segment of a request to the next, and
//     the order in which the forward kernels take the segments (seg_order):
//       chained: the kernel that finishes a segment publishes its end state,
//       and the next segment of the request, ordered at least one round of
//       first segments later (the k-th segments of all requests are taken
//       after every (k-1)-th one), picks it up -- one pass over the data;
//       pre-pass: every segment's state from zero and its total decay are
//       computed first (ssd_segstate.cu for headdim 64, the state-only mode of
//       ssd_chunk_tc.cu otherwise) and chained (seg_pass_kernel), for batches
//       whose longest request would otherwise be a serial chain longer than
//       the work of a CTA (a few long requests);
//   * validation bits for the device error word.
// One CTA of up to 1024 threads (one per request, at least 64); no host
// synchronisation.
#include <algorithm>

#include "pdl.cuh"
#include "ssd_internal.cuh"

namespace ssd {
namespace {

constexpr int kPlanThreads = 1024;  // at most; the launch sizes the block to the batch

// Block-wide exclusive scan of two counters; returns the block totals.  Any block
// of whole warps (at most 32).
__device__ void block_scan2(int a, int b, int &ea, int &eb, int &ta, int &tb) {
    __shared__ int wa[32], wb[32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (int)(blockDim.x >> 5);
    int ia = a, ib = b;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int va = __shfl_up_sync(0xffffffffu, ia, o), vb = __shfl_up_sync(0xffffffffu, ib, o);
        if (lane >= o) { ia += va; ib += vb; }
    }
    if (lane == 31) { wa[warp] = ia; wb[warp] = ib; }
    __syncthreads();
    if (warp == 0) {
        int sa = lane < nw ? wa[lane] : 0, sb = lane < nw ? wb[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int va = __shfl_up_sync(0xffffffffu, sa, o), vb = __shfl_up_sync(0xffffffffu, sb, o);
            if (lane >= o) { sa += va; sb += vb; }
        }
        wa[lane] = sa;
        wb[lane] = sb;
    }
    __syncthreads();
    const int pa = warp ? wa[warp - 1] : 0, pb = warp ? wb[warp - 1] : 0;
    ea = pa + ia - a;
    eb = pb + ib - b;
    ta = wa[nw - 1];
    tb = wb[nw - 1];
    __syncthreads();
}

// Segments per request at most for the chained mode (one ordering pass each).
constexpr int kMaxChainSegs = 16;
// Batches of at most this many requests rank them by segment count and length
// (each thread counts over all of them); larger ones by segment count only.
constexpr int kRankByLength = 256;

// How a request at absolute positions [s, s + L), L >= 1, is cut into work
// segments: segment k spans [lo(k), lo(k + 1)), lo(0) = s, lo(count()) = s + L.
//   Multiples (tail false): cuts at the multiples of len strictly inside.
//   Tail-shortened (tail true): the last segment starts at t1, the last multiple
//   of 256 at least 129 tokens before the end (so it holds 129-384 tokens),
//   provided t1 - s >= 256; the one before it at t2 = t1 - 512, provided
//   t2 - s >= 512; the part before the first of these cuts, the head, is cut
//   from its end backwards into n = ceil(length / 2048) segments of one stride,
//   the smallest multiple of 256 not below length / n (the first segment takes
//   the rest).  Every cut is a multiple of 256; every segment holds 1 to len
//   tokens (len = 2048 for the tail-shortened rule).
struct SegCuts {
    int64_t s, e, head_end, stride, t1;
    int32_t len;
    int n_head, n_tail;
    bool tail;
    __device__ SegCuts(int64_t s_, int64_t L, int32_t len_, bool tail_)
        : s(s_), e(s_ + L), head_end(s_ + L), stride(0), t1(0), len(len_), n_head(1), n_tail(0), tail(tail_) {
        if (!tail) return;
        if (L >= 385) {
            t1 = (e - 129) / 256 * 256;
            if (t1 - s >= 256) {
                n_tail = t1 - 512 - s >= 512 ? 2 : 1;
                head_end = n_tail == 2 ? t1 - 512 : t1;
            }
        }
        const int64_t hlen = head_end - s;
        n_head = (int)((hlen + 2047) / 2048);
        stride = n_head > 1 ? ((hlen + n_head - 1) / n_head + 255) / 256 * 256 : hlen;
    }
    __device__ int count() const {
        if (!tail) return (int)((e - 1) / len - s / len + 1);
        return n_head + n_tail;
    }
    __device__ int64_t lo(int k) const {
        if (k <= 0) return s;
        if (k >= count()) return e;
        if (!tail) return (s / len + k) * (int64_t)len;
        if (k < n_head) return head_end - stride * (n_head - k);
        return k == n_head ? head_end : t1;  // the tail cuts: head_end (t2 or t1), then t1
    }
};

__device__ __forceinline__ int segs_of(const int32_t *cu, const int32_t *ncomp, int i, int32_t seg_len, bool tail) {
    const int64_t L = (int64_t)cu[i + 1] - cu[i];
    const int64_t s = ncomp ? (int64_t)ncomp[i] : 0;
    if (L <= 0) return 1;
    return SegCuts(s, L, seg_len, tail).count();
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const PlanArgs a) {
    const int32_t *__restrict__ cu = a.cu;
    const int32_t *__restrict__ ncomp = a.ncomp;
    const int32_t R = a.R, Q = a.Q, seg_len = a.seg_len;
    const bool tail = a.seg_tail != 0;
    const int64_t T = a.T;
    int32_t *hdr = a.hdr;
    int32_t *__restrict__ req_first_chunk = a.req_first_chunk;
    int32_t *__restrict__ req_first_seg = a.req_first_seg;
    Seg *__restrict__ segs = a.segs;
    // the forward's first kernel may be scheduled now; it waits for this one.
    // This kernel is itself a dependent launch: it waits for the stream's previous
    // kernel (which may have written cu_seqlens) before reading anything.
    pdl_launch_dependents();
    pdl_wait();
    __shared__ int s_err, s_empty, s_max_segs;
    __shared__ long long s_max_len;
    if (threadIdx.x == 0) {
        s_err = s_empty = s_max_segs = 0;
        s_max_len = 0;
    }
    __syncthreads();
    int err = 0, n_empty = 0, my_max_segs = 0;
    long long my_max_len = 0;
    int carry_c = 0, carry_s = 0;
    const int nt = (int)blockDim.x;
    for (int base = 0; base < R; base += nt) {
        const int i = base + threadIdx.x;
        int nc = 0, ns = 0;
        if (i < R) {
            const int64_t a = cu[i], b = cu[i + 1];
            int64_t L = b - a;
            int64_t s = ncomp ? (int64_t)ncomp[i] : 0;
            if (L < 0 || (i == 0 && a != 0)) { err |= SSD_DEVERR_CU_SEQLENS; L = 0; }
            if (s < 0 || s + L > 0x7fffffffLL) { err |= SSD_DEVERR_NUM_COMPUTED; s = 0; }
            if (L > 0) {
                nc = (int)((s + L - 1) / Q - s / Q + 1);
                ns = SegCuts(s, L, seg_len, tail).count();
            } else {
                ns = 1;  // an empty request still gets one (empty) segment: final = initial
                ++n_empty;
            }
            my_max_segs = max(my_max_segs, ns);
            my_max_len = max(my_max_len, (long long)L);
        }
        int ec, es, tc, ts;
        block_scan2(nc, ns, ec, es, tc, ts);
        if (i < R) {
            req_first_chunk[i] = carry_c + ec;
            req_first_seg[i] = carry_s + es;
        }
        carry_c += tc;
        carry_s += ts;
    }
    if (threadIdx.x == 0) {
        if ((int64_t)cu[R] != T) err |= SSD_DEVERR_CU_SEQLENS;
        req_first_chunk[R] = carry_c;
        req_first_seg[R] = carry_s;
    }
    if (err) atomicOr(&s_err, err);
    if (n_empty) atomicAdd(&s_empty, n_empty);
    if (my_max_segs) atomicMax(&s_max_segs, my_max_segs);
    if (my_max_len) atomicMax(&s_max_len, my_max_len);
    __syncthreads();
    const int all_err = s_err;
    const bool bad = (all_err & (SSD_DEVERR_CU_SEQLENS | SSD_DEVERR_NUM_COMPUTED)) != 0 ||
                     (int64_t)carry_s > a.max_segs;
    // Chained when some request has more than one segment, none has more than
    // kMaxChainSegs, and the longest request is no longer than chain_max_len
    // tokens (its serial chain then fits the work one CTA does anyway).
    const int maxk = s_max_segs;
    const bool chained = !bad && maxk > 1 && maxk <= kMaxChainSegs && (int64_t)s_max_len <= a.chain_max_len;
    if (threadIdx.x == 0) {
        hdr[kHdrErr] = all_err;
        hdr[kHdrChunks] = bad ? 0 : carry_c;
        hdr[kHdrSegs] = bad ? 0 : carry_s;
        hdr[kHdrTicket] = 0;
        hdr[kHdrTimeoutAt] = hdr[kHdrTimeoutAt + 1] = hdr[kHdrTimeoutAt + 2] = 0;
        // every request has exactly one final segment
        hdr[kHdrNonFinal] = bad ? 0 : carry_s - R;
        hdr[kHdrEmpty] = bad ? 0 : s_empty;
        hdr[kHdrMode] = chained ? kModeChained : kModePrepass;
        hdr[kHdrEpoch] = 0;
        hdr[kHdrTestHook] = 0;
    }
    if (bad) return;  // forward kernels see zero segments and write nothing
    __syncthreads();
    // The order the forward kernels take the segments in: chained, the k-th
    // segments of all requests (k = 0, 1, ...), round by round; otherwise the
    // segment list itself.  Within a round the requests with the most segments
    // go first (their chains are the longest, and start first) and, among
    // those, the longest (the longest items first: the last ones to finish are
    // short), ties in request order -- by segment count alone past
    // kRankByLength requests; batches past one pass of the block keep request
    // order.  Chained, the per-(segment, head) publication counters start from
    // zero.
    if (chained && R <= nt) {
        __shared__ int cnt_w[kPlanThreads / 32][kMaxChainSegs + 1];
        __shared__ int bin_base[kMaxChainSegs + 1];
        __shared__ int perm[kPlanThreads], segc[kPlanThreads], lens[kPlanThreads];
        const int t = threadIdx.x, lane = t & 31, w = t >> 5, nw = nt >> 5;
        const int c = t < R ? segs_of(cu, ncomp, t, seg_len, tail) : 0;  // 1 .. maxk; 0: no request
        const int len_t = t < R ? cu[t + 1] - cu[t] : 0;
        segc[t] = c;
        lens[t] = len_t;
        if (R <= kRankByLength) {
            __syncthreads();
            if (t < R) {  // place = the requests ahead of this one
                int place = 0;
                for (int j = 0; j < R; ++j) {
                    const int cj = segc[j], lj = lens[j];
                    place += (cj > c || (cj == c && (lj > len_t || (lj == len_t && j < t)))) ? 1 : 0;
                }
                perm[place] = t;
            }
        } else {
            // stable counting sort by segment count: the warp's requests with the
            // same count and how many of them come before this one, then per count
            // an exclusive prefix over the warps, then the counts from the largest down
            for (int j = t; j < nw * (kMaxChainSegs + 1); j += nt) cnt_w[j / (kMaxChainSegs + 1)][j % (kMaxChainSegs + 1)] = 0;
            __syncthreads();
            const unsigned same = __match_any_sync(0xffffffffu, c);
            const int before = __popc(same & ((1u << lane) - 1u));
            if (c > 0 && before == 0) cnt_w[w][c] = __popc(same);
            __syncthreads();
            if (t >= 1 && t <= kMaxChainSegs) {
                int run = 0;
                for (int ww = 0; ww < nw; ++ww) {
                    const int x = cnt_w[ww][t];
                    cnt_w[ww][t] = run;
                    run += x;
                }
                bin_base[t] = run;
            }
            __syncthreads();
            if (t == 0) {
                int run = 0;
                for (int v = kMaxChainSegs; v >= 1; --v) {
                    const int x = bin_base[v];
                    bin_base[v] = run;
                    run += x;
                }
            }
            __syncthreads();
            if (c > 0) perm[bin_base[c] + cnt_w[w][c] + before] = t;
        }
        __syncthreads();
        const int ic = t < R ? perm[t] : 0;  // the request at place t of a round
        const int cc = t < R ? segc[ic] : 0;
        int base = 0;
        for (int k = 0; k < maxk; ++k) {
            const int has = cc > k ? 1 : 0;
            int e1, e2, t1, t2;
            block_scan2(has, 0, e1, e2, t1, t2);
            if (has) a.seg_order[base + e1] = req_first_seg[ic] + k;
            base += t1;
        }
    } else if (chained) {
        int base = 0;
        for (int k = 0; k < maxk; ++k) {
            for (int b0 = 0; b0 < R; b0 += nt) {
                const int i = b0 + threadIdx.x;
                const int has = (i < R && segs_of(cu, ncomp, i, seg_len, tail) > k) ? 1 : 0;
                int e1, e2, t1, t2;
                block_scan2(has, 0, e1, e2, t1, t2);
                if (has) a.seg_order[base + e1] = req_first_seg[i] + k;
                base += t1;
            }
        }
    }
    if (chained) {
        const int64_t nflags = (int64_t)(carry_s - R) * a.H;
        for (int64_t j = threadIdx.x; j < nflags; j += nt) a.seg_flags[j] = 0;
    } else {
        for (int j = threadIdx.x; j < carry_s; j += nt) a.seg_order[j] = j;
    }
    // Fill the segment list (one thread per request; long requests loop).
    for (int i = threadIdx.x; i < R; i += nt) {
        const int64_t a = cu[i], L = (int64_t)cu[i + 1] - a;
        const int64_t s = ncomp ? (int64_t)ncomp[i] : 0;
        const int first = req_first_seg[i], cnt = req_first_seg[i + 1] - first;
        if (L == 0) {
            segs[first] = Seg{i, (int32_t)a, 0, (int32_t)s};
            continue;
        }
        const SegCuts c(s, L, seg_len, tail);
        for (int k = 0; k < cnt; ++k) {
            const int64_t lo = c.lo(k), hi = c.lo(k + 1);
            segs[first + k] = Seg{i, (int32_t)(a + (lo - s)), (int32_t)(hi - lo), (int32_t)lo};
        }
    }
}

}  // namespace

cudaError_t launch_plan(const PlanArgs &a, cudaStream_t stream) {
    // one warp per 32 requests, at least two (the flag zeroing), at most 32
    const int threads = (int)std::min<int64_t>(kPlanThreads, std::max<int64_t>(64, ((int64_t)a.R + 31) / 32 * 32));
    return launch_after_prev(plan_kernel, dim3(1), dim3(threads), 0, stream, a);
}

}  // namespace ssd
