// ssd_api.cu -- the C ABI: argument validation, workspace layout, dispatch.
//
// Checks every host-visible precondition before launching anything (the
// chunk_size power-of-two rule of the "[Bugfix] Mamba2 SSD varlen bug fix
// initstates decay" page, documentation note; the block-size-is-a-multiple-
// of-the-kernel-chunk rule of the "Automatic prefix caching for GDN hybrid
// models" page, platform-level block-size validation), then launches the
// metadata builder (plan) or the forward kernels on the caller's stream.
#include <string.h>

#include <algorithm>

#include "ssd_internal.cuh"

namespace ssd {

static bool is_pow2(int v) { return v > 0 && (v & (v - 1)) == 0; }

static int check_dims(const ssd_dims *d) {
    if (!d) return SSD_ERR_NULL;
    if (d->reserved != 0) return SSD_ERR_DIMS;
    if (d->T < 0 || d->T > 0x7fffffffLL || d->R < 1 || d->H < 1 || d->P < 1 || d->N < 1 || d->G < 1)
        return SSD_ERR_DIMS;
    if (d->P > 256 || d->N > 256 || d->H > 65535) return SSD_ERR_DIMS;
    if (d->N > 32 && d->N % 32 != 0) return SSD_ERR_UNSUPPORTED;
    if (d->H % d->G != 0) return SSD_ERR_GROUPS;
    if (!is_pow2(d->chunk_size) || d->chunk_size < 16 || d->chunk_size > 256) return SSD_ERR_CHUNK_SIZE;
    if (d->dtype != SSD_DTYPE_BF16 && d->dtype != SSD_DTYPE_F32) return SSD_ERR_DTYPE;
    if (d->num_slots < 0 || d->block_table_width < 0) return SSD_ERR_DIMS;
    if (d->block_size < 0) return SSD_ERR_BLOCK_SIZE;
    if (d->block_size > 0 && d->block_size % d->chunk_size != 0) return SSD_ERR_BLOCK_SIZE;
    return SSD_OK;
}

// How requests are cut into work segments, which CTAs walk in parallel (the
// state chain between the segments of a request is resolved by the forward
// path).  Every cut is at an absolute position that is a multiple of 256 (the
// largest chunk size), every segment holds at most 2048 tokens.
//   * Batches of requests averaging 1024-2048 tokens: tail-shortened segments
//     (the plan's rule): a request ends with a short segment (129-384 tokens)
//     and a 512-token one before it, the rest in segments of up to 2048, so that
//     the last rounds of the schedule hold short items and the SMs finish
//     together (a 2048-token request: 1280 + 512 + 256).
//   * Others: cuts at the multiples of 2048 where the segment-state pre-pass is
//     the two-head contraction (P = 64, N = 128, an even number of heads per
//     group: its token weights hold 2048 tokens), 8192 otherwise -- few items,
//     little start-up; the chained rounds take the longest chains first.
constexpr int32_t kPlanTailSegs = 1;  // ssd_plan.flags bit: tail-shortened segments

struct SegRule {
    int32_t len;  // longest segment
    bool tail;    // tail-shortened segments
};

static SegRule pick_seg_rule(const ssd_dims *d) {
    if (d->T > 1024LL * d->R && d->T <= 2048LL * d->R) return {2048, true};
    const bool two_head_prepass = d->P == 64 && d->N == 128 && d->G > 0 && (d->H / d->G) % 2 == 0;
    return {two_head_prepass ? 2048 : 8192, false};
}

static SegRule rule_of(const ssd_plan *plan) { return {plan->seg_len, (plan->flags & kPlanTailSegs) != 0}; }

// The longest request the chained mode takes: its segments form one serial
// chain per head, which must not outlast the work a CTA does anyway
// (T H / (2 SMs) tokens of one head's worth).
static int64_t chain_max_len_of(const ssd_dims *d) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                   cudaSuccess || sms < 1)
        sms = 1;
    return d->T * (int64_t)d->H / (2LL * sms);
}

// Work segments of a batch that are not the last of their request, at most.
// Every request has exactly one final segment (an empty request one empty
// segment).  Cut at the multiples of len, its other segments end on such a
// multiple strictly inside its positions (s, s + L - 1]: at most
// ceil((L - 1) / len) per request, so over the batch at most
// floor((T + R (len - 2)) / len).  Tail-shortened, a request of L tokens has at
// most ceil(L / 2048) head segments and two tail segments, so at most
// (L + 4095) / 2048 that are not its last: over the batch at most
// floor((T + 4095 R) / 2048).  As every segment holds a token, at most T - 1.
static int64_t nonfinal_segs_of(const ssd_dims *d, SegRule rule) {
    const int64_t by_len = rule.tail ? (d->T + 4095LL * d->R) / 2048
                                     : (d->T + (int64_t)d->R * (rule.len - 2)) / rule.len;
    const int64_t by_tokens = d->T - 1;
    return std::max<int64_t>(0, std::min(by_len, by_tokens));
}

static int64_t max_segs_of(const ssd_dims *d, SegRule rule) { return nonfinal_segs_of(d, rule) + d->R; }

static WsLayout layout_of(const ssd_dims *d, SegRule rule) {
    WsLayout w{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off = align_up(off + bytes, 256);
        return o;
    };
    const int64_t ms = max_segs_of(d, rule);
    w.hdr = take(sizeof(int32_t) * kHdrInts);
    w.req_first_chunk = take(sizeof(int32_t) * ((size_t)d->R + 1));
    w.req_first_seg = take(sizeof(int32_t) * ((size_t)d->R + 1));
    w.segs = take(sizeof(Seg) * (size_t)ms);
    w.seg_order = take(sizeof(int32_t) * (size_t)ms);
    // one state (and one decay per head) for each segment that is not the last of
    // its request, indexed compactly: segment k of request i uses entry k - i
    const int64_t nf = nonfinal_segs_of(d, rule);
    w.seg_state = take(sizeof(float) * (size_t)nf * d->H * d->P * d->N);
    w.seg_decay = take(sizeof(float) * (size_t)nf * d->H);
    w.seg_flags = take(sizeof(int32_t) * (size_t)nf * d->H);
    w.total = off;
    return w;
}

static bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }
static bool aligned4(const void *p) { return ((uintptr_t)p & 3u) == 0; }

// Checks every host-visible precondition of a forward and fills the kernel
// parameters.  Launches nothing.
static int forward_params(const ssd_plan *plan, const ssd_inputs *in, const ssd_outputs *out, FwdParams *p) {
    if (!plan || !in || !out) return SSD_ERR_NULL;
    if (plan->magic != kPlanMagic) return SSD_ERR_PLAN;
    const ssd_dims *d = &plan->dims;
    int rc = check_dims(d);
    if (rc != SSD_OK) return rc;
    if (!in->dt_bias || !in->A) return SSD_ERR_NULL;
    // with no tokens (every request empty) the token buffers may be NULL
    if (d->T > 0 && (!in->x || !in->dt || !in->B || !in->C || !out->y)) return SSD_ERR_NULL;
    const void *big[] = {in->x, in->dt, in->B, in->C, in->z, out->y, in->state_pool,
                         out->final_states, out->chunk_states};
    for (const void *ptr : big)
        if (ptr && !aligned16(ptr)) return SSD_ERR_ALIGN;
    const void *small[] = {in->dt_bias, in->A, in->D, in->init_slots, out->final_slots, out->block_table};
    for (const void *ptr : small)
        if (ptr && !aligned4(ptr)) return SSD_ERR_ALIGN;
    const bool uses_pool = in->init_slots || out->final_slots || out->block_table;
    if (uses_pool && (!in->state_pool || d->num_slots < 1)) return SSD_ERR_NULL;
    if (out->block_table && (d->block_size <= 0 || d->block_table_width < 1)) return SSD_ERR_BLOCK_SIZE;

    const WsLayout w = layout_of(d, rule_of(plan));
    if (plan->workspace_bytes < w.total) return SSD_ERR_WORKSPACE;
    char *ws = static_cast<char *>(plan->workspace);
    p->T = d->T;
    p->R = d->R;
    p->H = d->H;
    p->P = d->P;
    p->N = d->N;
    p->G = d->G;
    p->Q = d->chunk_size;
    p->num_slots = d->num_slots;
    p->block_size = d->block_size;
    p->bt_width = d->block_table_width;
    p->seg_len = plan->seg_len;
    p->cu_seqlens = plan->cu_seqlens;
    p->num_computed = plan->num_computed;
    p->hdr = (int32_t *)(ws + w.hdr);
    p->req_first_chunk = (const int32_t *)(ws + w.req_first_chunk);
    p->req_first_seg = (const int32_t *)(ws + w.req_first_seg);
    p->segs = (const Seg *)(ws + w.segs);
    p->seg_state = (float *)(ws + w.seg_state);
    p->seg_decay = (float *)(ws + w.seg_decay);
    p->seg_order = (const int32_t *)(ws + w.seg_order);
    p->seg_flags = (int32_t *)(ws + w.seg_flags);
    p->x = in->x;
    p->dt = in->dt;
    p->B = in->B;
    p->C = in->C;
    p->z = in->z;
    p->dt_bias = in->dt_bias;
    p->A = in->A;
    p->D = in->D;
    p->init_slots = in->init_slots;
    p->pool = in->state_pool;
    p->y = out->y;
    p->final_states = out->final_states;
    p->final_slots = out->final_slots;
    p->chunk_states = out->chunk_states;
    p->block_table = out->block_table;
    return SSD_OK;
}

// The kernel path a forward takes.  An empty batch (final = initial state for
// every request) takes the general path, which needs no tensor maps over the
// absent token buffers.
static int path_of(const FwdParams &p, const ssd_dims *d) {
    if (d->T > 0 && chunk_tc_supported(p, d->dtype))
        return pair_supported(p) ? SSD_PATH_TENSOR_CORE_PAIRED : SSD_PATH_TENSOR_CORE;
    return SSD_PATH_GENERAL;
}

}  // namespace ssd

using namespace ssd;

extern "C" {

size_t ssd_varlen_workspace_size(const ssd_dims *dims) {
    if (check_dims(dims) != SSD_OK) return 0;
    return layout_of(dims, pick_seg_rule(dims)).total;
}

int64_t ssd_varlen_count_chunks(const int32_t *cu, const int32_t *ncomp, int32_t R, int32_t Q) {
    if (!cu || R < 1 || !is_pow2(Q)) return SSD_ERR_DIMS;
    if (cu[0] != 0) return SSD_ERR_DIMS;
    int64_t n = 0;
    for (int32_t i = 0; i < R; ++i) {
        const int64_t L = (int64_t)cu[i + 1] - cu[i];
        const int64_t s = ncomp ? ncomp[i] : 0;
        if (L < 0 || s < 0) return SSD_ERR_DIMS;
        if (L > 0) n += (s + L - 1) / Q - s / Q + 1;
    }
    return n;
}

int ssd_varlen_plan(const ssd_dims *dims, const int32_t *cu_seqlens, const int32_t *num_computed,
                    void *workspace, size_t workspace_bytes, cudaStream_t stream, ssd_plan *out) {
    int rc = check_dims(dims);
    if (rc != SSD_OK) return rc;
    if (!cu_seqlens || !workspace || !out) return SSD_ERR_NULL;
    if (!aligned4(cu_seqlens) || (num_computed && !aligned4(num_computed))) return SSD_ERR_ALIGN;
    const SegRule rule = pick_seg_rule(dims);
    const WsLayout w = layout_of(dims, rule);
    if (!aligned16(workspace)) return SSD_ERR_WORKSPACE;
    if (workspace_bytes < w.total) return SSD_ERR_WORKSPACE;
    char *ws = static_cast<char *>(workspace);
    PlanArgs a{};
    a.cu = cu_seqlens;
    a.ncomp = num_computed;
    a.R = dims->R;
    a.H = dims->H;
    a.Q = dims->chunk_size;
    a.seg_len = rule.len;
    a.seg_tail = rule.tail ? 1 : 0;
    a.T = dims->T;
    a.max_segs = max_segs_of(dims, rule);
    a.chain_max_len = chain_max_len_of(dims);
    a.hdr = (int32_t *)(ws + w.hdr);
    a.req_first_chunk = (int32_t *)(ws + w.req_first_chunk);
    a.req_first_seg = (int32_t *)(ws + w.req_first_seg);
    a.segs = (Seg *)(ws + w.segs);
    a.seg_order = (int32_t *)(ws + w.seg_order);
    a.seg_flags = (int32_t *)(ws + w.seg_flags);
    cudaError_t e = launch_plan(a, stream);
    if (e != cudaSuccess) return SSD_ERR_CUDA;
    memset(out, 0, sizeof(*out));
    out->dims = *dims;
    out->workspace = workspace;
    out->workspace_bytes = workspace_bytes;
    out->cu_seqlens = cu_seqlens;
    out->num_computed = num_computed;
    out->max_chunks = (dims->T + dims->chunk_size - 1) / dims->chunk_size + dims->R;
    out->max_segs = max_segs_of(dims, rule);
    out->seg_len = rule.len;
    out->flags = rule.tail ? kPlanTailSegs : 0;
    out->magic = kPlanMagic;
    out->stream = stream;
    return SSD_OK;
}

int ssd_varlen_forward(const ssd_plan *plan, const ssd_inputs *in, const ssd_outputs *out,
                       cudaStream_t stream) {
    FwdParams p{};
    const int rc = forward_params(plan, in, out, &p);
    if (rc != SSD_OK) return rc;
    const ssd_dims *d = &plan->dims;
    if (d->T == 0 && !out->final_states && !out->final_slots) return SSD_OK;
    cudaError_t e = path_of(p, d) == SSD_PATH_GENERAL ? launch_recurrent(p, d->dtype, stream)
                                                       : launch_chunk_tc(p, plan->max_segs, stream);
    return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

int ssd_varlen_forward_path(const ssd_plan *plan, const ssd_inputs *in, const ssd_outputs *out, int *path,
                            int *tile) {
    if (!path) return SSD_ERR_NULL;
    FwdParams p{};
    const int rc = forward_params(plan, in, out, &p);
    if (rc != SSD_OK) return rc;
    *path = path_of(p, &plan->dims);
    if (tile) *tile = *path == SSD_PATH_GENERAL ? 1 : chunk_tc_tile(p);
    return SSD_OK;
}

int ssd_varlen_status(const ssd_plan *plan, int *device_err) {
    if (!plan || !device_err) return SSD_ERR_NULL;
    if (plan->magic != kPlanMagic) return SSD_ERR_PLAN;
    const WsLayout w = layout_of(&plan->dims, rule_of(plan));
    int32_t *hdr = (int32_t *)((char *)plan->workspace + w.hdr);
    // Only the plan's stream is synchronised (its work, then the read and the
    // clear, in stream order); other streams of the device keep running.
    int v = 0;
    if (cudaMemcpyAsync(&v, hdr + kHdrErr, sizeof(int), cudaMemcpyDeviceToHost, plan->stream) != cudaSuccess)
        return SSD_ERR_CUDA;
    if (cudaMemsetAsync(hdr + kHdrErr, 0, sizeof(int), plan->stream) != cudaSuccess) return SSD_ERR_CUDA;
    if (cudaStreamSynchronize(plan->stream) != cudaSuccess) return SSD_ERR_CUDA;
    *device_err = v;
    return SSD_OK;
}

const char *ssd_varlen_strerror(int code) {
    switch (code) {
        case SSD_OK: return "ok";
        case SSD_ERR_NULL: return "a required pointer is NULL";
        case SSD_ERR_DIMS: return "a size is out of range";
        case SSD_ERR_CHUNK_SIZE: return "chunk_size must be integer power of 2 in [16, 256]";
        case SSD_ERR_GROUPS: return "H must be a multiple of G";
        case SSD_ERR_BLOCK_SIZE: return "block_size must be a positive multiple of chunk_size";
        case SSD_ERR_DTYPE: return "unknown dtype";
        case SSD_ERR_ALIGN: return "a device pointer is not aligned (16 bytes for tensors)";
        case SSD_ERR_WORKSPACE: return "workspace too small or not 16-byte aligned";
        case SSD_ERR_PLAN: return "plan not built for this call";
        case SSD_ERR_CUDA: return "a CUDA runtime call failed";
        case SSD_ERR_UNSUPPORTED: return "unsupported size combination";
        default: break;
    }
    if (code > 0) return "device error bits set (see SSD_DEVERR_*)";
    return "unknown status";
}

}  // extern "C"
