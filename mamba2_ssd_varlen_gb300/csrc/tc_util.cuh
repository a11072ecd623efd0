// tc_util.cuh -- small device helpers shared by the tensor-core SSD kernels:
// hardware transcendentals, packed fp32-pair arithmetic (the f32x2
// instructions), the bf16 hi/lo operand split and barrier phase parity.
#pragma once

#include <stdint.h>

#include "sm100.cuh"

namespace ssd {
namespace tc {
using namespace sm100;

constexpr float kLog2e = 1.4426950408889634f;

// Phase parity of a barrier's use-th completion.
__device__ __forceinline__ uint32_t par(uint32_t use) { return use & 1u; }

__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 2^x on the special-function unit (flushes denormal results to zero).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float fast_rcp(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float fast_lg2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// softplus(v) = ln 2 * log2(1 + 2^(v log2 e)); the identity above 20
__device__ __forceinline__ float softplus_fast(float v) {
    return v > 20.f ? v : 0.69314718055994531f * fast_lg2(1.f + fast_exp2(v * kLog2e));
}

// ---- packed fp32 pairs (one 64-bit register pair) for the f32x2 instructions
__device__ __forceinline__ uint64_t f2(float a, float b) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(a), "f"(b));
    return d;
}
__device__ __forceinline__ void f2_get(uint64_t d, float &a, float &b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(d));
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
// bf16x2 word (low half first) -> the two values as an exact fp32 pair
__device__ __forceinline__ uint64_t f2_bf16x2(uint32_t w) {
    return f2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// silu of a pair, v / (1 + e^-v), on the special-function unit (exp2 and an
// approximate reciprocal, both to ~2^-22 relative).
__device__ __forceinline__ uint64_t silu2(uint64_t z) {
    float a, b;
    f2_get(f2_mul(z, f2(-kLog2e, -kLog2e)), a, b);
    const uint64_t den = f2_add(f2(fast_exp2(a), fast_exp2(b)), f2(1.f, 1.f));
    float da, db;
    f2_get(den, da, db);
    return f2_mul(z, f2(fast_rcp(da), fast_rcp(db)));
}

// Pair (a, b) ~= hi + lo in bf16x2: hi is each value truncated to bf16 (its
// upper 16 bits, exact), lo = bf16(v - hi) rounded; 16 significant bits kept.
__device__ __forceinline__ void split_pair(uint64_t ab, uint32_t &hi, uint32_t &lo) {
    uint32_t ua, ub;
    asm("mov.b64 {%0, %1}, %2;" : "=r"(ua), "=r"(ub) : "l"(ab));
    hi = __byte_perm(ua, ub, 0x7632);
    const uint64_t rest = f2_sub(ab, f2(__uint_as_float(ua & 0xFFFF0000u), __uint_as_float(ub & 0xFFFF0000u)));
    float ra, rb;
    f2_get(rest, ra, rb);
    lo = pack_bf16x2(ra, rb);
}

// ---- segment-state hand-off between CTAs (chained mode) ---------------------
// The CTA that finishes a segment writes its end state with plain stores, then
// every writing warp publishes: each lane fences its stores, then lane 0 adds
// one to the segment's counter.  A reader polls the counter with acquire loads
// until it reaches count x epoch (counters grow by `count` per forward) or the
// time limit passes.
__device__ __forceinline__ int ld_acquire(const int32_t *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void publish_warp(int32_t *counter, int lane) {
    __threadfence();
    __syncwarp();
    if (lane == 0) atomicAdd(counter, 1);
}
__device__ __forceinline__ bool poll_counter(const int32_t *counter, int target, uint64_t limit_ns) {
    if (ld_acquire(counter) >= target) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        __nanosleep(64);
        if (ld_acquire(counter) >= target) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

}  // namespace tc
}  // namespace ssd
