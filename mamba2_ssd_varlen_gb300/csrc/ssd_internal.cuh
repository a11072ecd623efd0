// ssd_internal.cuh -- shared declarations of the SSD varlen library (device + host).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ssd_varlen.h"

namespace ssd {

constexpr uint64_t kPlanMagic = 0x5353445641524C31ull;  // "SSDVARL1"
constexpr int kHdrInts = 64;                             // header words at the workspace start
// Header word indices.
constexpr int kHdrErr = 0;       // device error bits (SSD_DEVERR_*)
constexpr int kHdrChunks = 1;    // export rows of the batch
constexpr int kHdrSegs = 2;      // work segments of the batch
constexpr int kHdrTicket = 3;    // next work item of the scan kernel (a ticket counter)
constexpr int kHdrTimeoutAt = 4; // words 4-6: where the first timed-out wait of a launch was
constexpr int kHdrNonFinal = 7;  // segments that are not the last of their request (chained states)
constexpr int kHdrEmpty = 8;     // empty requests (final state = initial state)
constexpr int kHdrMode = 9;      // how segment states are carried (kMode*)
constexpr int kHdrEpoch = 10;    // forwards run on this plan (bumped by each forward's first kernel)
constexpr int kHdrTestHook = 11; // zero; read only by the timeout-test build of the scan
// kHdrMode values: chained (a segment's end state is published for the next
// segment of its request) or pre-pass (all segment states computed first).
constexpr int kModePrepass = 0;
constexpr int kModeChained = 1;
// Timeout site recorded for a wait on a previous segment's published state
// (the other sites are barrier offsets in shared memory, all below it).
constexpr int kSiteSegState = 0x40000;

// Byte offsets of the workspace regions (each 256-byte aligned).
struct WsLayout {
    size_t hdr, req_first_chunk, req_first_seg, segs, seg_order, seg_state, seg_decay, seg_flags, total;
};

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// One work segment: a run of consecutive tokens of one request that a CTA walks.
// Segments split requests at absolute multiples of seg_len.
struct Seg {
    int32_t req;        // request index
    int32_t tok;        // first packed token index
    int32_t len;        // tokens (0 only for an empty request)
    int32_t abs_start;  // absolute position of the first token (num_computed + offset)
};

// Everything a forward kernel needs, by value.
struct FwdParams {
    // sizes
    int64_t T;
    int32_t R, H, P, N, G, Q;
    int32_t num_slots, block_size, bt_width;
    int32_t seg_len;
    // plan metadata (device)
    const int32_t *cu_seqlens;
    const int32_t *num_computed;
    int32_t *hdr;
    const int32_t *req_first_chunk;
    const int32_t *req_first_seg;
    const Seg *segs;
    // Chained states of the segments that are not the last of their request,
    // indexed compactly: segment k of request i (k not its last) is entry k - i.
    float *seg_state;   // (non-final segments, H, P, N) workspace (see kernels)
    float *seg_decay;   // (non-final segments, H) workspace
    const int32_t *seg_order;  // segments in the order the kernels take them
    int32_t *seg_flags;        // (non-final segments, H): publication counters (chained mode)
    // inputs
    const void *x, *dt, *B, *C, *z;
    const float *dt_bias, *A, *D;
    const int32_t *init_slots;
    float *pool;
    // outputs
    void *y;
    float *final_states;
    const int32_t *final_slots;
    float *chunk_states;
    const int32_t *block_table;
};

// ---- device helpers -------------------------------------------------------
__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

// softplus(v) = log(1 + e^v); the identity above 20 (where the two agree to fp32).
__device__ __forceinline__ float softplus_f32(float v) { return v > 20.f ? v : log1pf(expf(v)); }
__device__ __forceinline__ float silu_f32(float v) { return v / (1.f + expf(-v)); }

__device__ __forceinline__ void set_err(int32_t *hdr, int bits) { atomicOr(hdr + kHdrErr, bits); }

// ---- launchers (defined in the .cu files) ---------------------------------
struct PlanArgs {
    const int32_t *cu, *ncomp;
    int32_t R, H, Q, seg_len;
    int32_t seg_tail;  // nonzero: tail-shortened segments (ssd_plan.cu), else cuts at multiples of seg_len
    int64_t T, max_segs;
    int64_t chain_max_len;  // longest request (tokens) the chained mode takes
    int32_t *hdr, *req_first_chunk, *req_first_seg;
    Seg *segs;
    int32_t *seg_order, *seg_flags;
};
cudaError_t launch_plan(const PlanArgs &a, cudaStream_t stream);

cudaError_t launch_recurrent(const FwdParams &p, int dtype, cudaStream_t stream);

// Tensor-core chunked path (bf16, P in {64, 128}, N = 128).
bool chunk_tc_supported(const FwdParams &p, int dtype);
int chunk_tc_tile(const FwdParams &p);
cudaError_t launch_chunk_tc(const FwdParams &p, int64_t max_segs, cudaStream_t stream);
// The scan with two heads of a group per CTA (P = 64, N = 128, an even number of
// heads per group); launched by launch_chunk_tc after the segment-state passes.
bool pair_supported(const FwdParams &p);
cudaError_t launch_pair_scan(const FwdParams &p, int Qi, int64_t max_items, cudaStream_t stream);
// The segment-state pre-pass as one contraction per segment (P = 64, N = 128);
// launched by launch_chunk_tc first (it also rewinds the ticket and counts the forward).
bool seg_state_supported(const FwdParams &p);
cudaError_t launch_seg_state(const FwdParams &p, int64_t max_items, cudaStream_t stream);
// The gated delta rule prefill on the tcgen05 tensor cores (bf16, K = V = 128,
// 64-token chunks); ssd_varlen_gdn_forward validates the call, then launches it.
bool gdn_tc_supported(const ssd_gdn_dims *d);
int launch_gdn_tc(const ssd_gdn_dims *d, const int32_t *cu_seqlens, const ssd_gdn_io *io, cudaStream_t stream);

}  // namespace ssd
