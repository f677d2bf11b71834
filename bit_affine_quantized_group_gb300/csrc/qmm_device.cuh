// Device primitives for the qmm kernels (sm_103a): inline PTX for mbarriers,
// bulk (TMA) and cp.async copies, programmatic dependent launch, the warp-level
// bf16 / f16 tensor-core MMA, and the in-register code unpackers.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "qmm_layout.h"

namespace qmmk {

// Error bits written to the plan's device error word.
constexpr uint32_t kErrFullWait = 1u;     // consumer gave up waiting for a stage
constexpr uint32_t kErrEmptyWait = 2u;    // producer gave up waiting for a free slot
constexpr uint32_t kErrDrainWait = 4u;    // producer gave up draining its copies
constexpr uint32_t kErrBadCopy = 8u;      // a copy failed its bounds/alignment check and was skipped

// Record a rejected copy: error bit plus (first) offending address and size in
// err[2..5]; the copy itself is skipped.
__device__ __forceinline__ void record_bad_copy(uint32_t* err, const void* a, uint64_t b, uint32_t what) {
    if (atomicOr(err, kErrBadCopy) & kErrBadCopy) return;
    const uint64_t av = reinterpret_cast<uint64_t>(a);
    err[2] = static_cast<uint32_t>(av);
    err[3] = static_cast<uint32_t>(av >> 32);
    err[4] = static_cast<uint32_t>(b);
    err[5] = what;
}

// A pipeline wait that has not finished after this long is treated as a hang:
// the kernel records it and returns instead of spinning forever.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;   // 2 s

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---- programmatic dependent launch ----------------------------------------
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- mbarrier ---------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
// Make barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
                 ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait on a phase parity; on timeout sets `code` in *err and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t* err, uint32_t code) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 0 && global_timer_ns() - t0 > kWaitLimitNs) {
            atomicOr(err, code);
            return false;
        }
    }
}

// ---- copies -----------------------------------------------------------------
// 1-D bulk copy global -> shared, completion counted in bytes on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
// Same with an L2 evict-first hint (for data read exactly once).
__device__ __forceinline__ void bulk_g2s_stream(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                                uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
        ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}
// 2-D TMA tile load: the box at element coordinates (x, y) of `map` into shared
// memory at dst (aligned to the map's swizzle atom), completion counted in bytes
// on `bar`. x times the element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
// Per-thread asynchronous copies (LDGSTS).
// 16 bytes, L2-only, with an L2 eviction-priority policy (for streamed data).
__device__ __forceinline__ void cp_async_16_hint(void* dst, const void* src, uint64_t policy) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;"
                 ::"r"(smem_u32(dst)), "l"(src), "l"(policy) : "memory");
}
__device__ __forceinline__ void cp_async_16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_4(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
// Wait until all of this thread's cp.async copies have landed.
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// Arrive on `bar` once this thread's earlier cp.async copies have landed
// (the arrival is pre-counted in the barrier's initial count).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// ---- tensor-core MMA (warp level) -------------------------------------------
// D = A*B + C, m16n8k16, A/B bf16, C/D fp32.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// D = A*B (zero accumulator), m16n8k16, A/B bf16.
__device__ __forceinline__ void mma_bf16_zc(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                            uint32_t b0, uint32_t b1) {
    const float z = 0.0f;
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(z));
}
// D = A*B (zero accumulator), m16n8k16, A/B binary16.
__device__ __forceinline__ void mma_f16_zc(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                           uint32_t b0, uint32_t b1) {
    const float z = 0.0f;
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(z));
}
// Same with binary16 operands.
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---- code unpacking ----------------------------------------------------------
// Every unpacker produces four bf16x2 registers r[i] = (128 + c_i, 128 + c_{i+4})
// for the 8 codes c_0..c_7 a lane owns in one virtual k32 block. A code q < 128
// written into the low mantissa bits of the bf16 pattern 0x4300 (= 128.0) is
// the exact value 128 + q; the 128 offset is removed later through the bias
// term (sum x*(128+q) = P + 128*XS).
constexpr uint32_t kBf16x2_128 = 0x43004300u;

// `magic` is kBf16x2_128, passed in as a run-time value by the hot loop: a
// three-input logic op takes a single immediate, so with both the mask and the
// pattern as literals every (w & mask) | pattern would compile to two ops.

// 4-bit (and each word of an 8-bit row read as 8 nibbles): one word holds the
// lane's 8 codes, nibble i = code i.
__device__ __forceinline__ void unpack_nibbles(uint32_t w, uint32_t (&r)[4], uint32_t magic = kBf16x2_128) {
    constexpr uint32_t m = 0x000F000Fu;
    r[0] = (w & m) | magic;
    r[1] = ((w >> 4) & m) | magic;
    r[2] = ((w >> 8) & m) | magic;
    r[3] = ((w >> 12) & m) | magic;
}

// 5- or 6-bit: the lane's 8 codes are 5 or 6 bytes starting at byte BITS*t of
// the block; `lo`, `hi` are the two words covering them and `sh` (0, 8, 16,
// 24) the bit offset of the first code inside `lo`.
template <int BITS>
__device__ __forceinline__ void unpack_odd(uint32_t lo, uint32_t hi, uint32_t sh, uint32_t (&r)[4],
                                           uint32_t magic = kBf16x2_128) {
    const uint64_t v = ((static_cast<uint64_t>(hi) << 32) | lo) >> sh;
    constexpr uint32_t mk = (1u << BITS) - 1u;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t a = static_cast<uint32_t>(v >> (BITS * i)) & mk;
        const uint32_t b = static_cast<uint32_t>(v >> (BITS * (i + 4))) & mk;
        r[i] = a | (b << 16) | magic;
    }
}

// Word index (within a virtual block) and bit shift of lane t's codes for odd widths.
template <int BITS>
__device__ __forceinline__ int odd_word(int t) { return (BITS * t) >> 2; }
template <int BITS>
__device__ __forceinline__ uint32_t odd_shift(int t) { return static_cast<uint32_t>(((BITS * t) & 3) * 8); }

// Unpack lane t's 8 codes of the virtual block starting at `blk` (4-byte aligned).
template <int BITS>
__device__ __forceinline__ void unpack_block(const uint32_t* blk, int t, uint32_t (&r)[4]) {
    if constexpr (BITS == 4 || BITS == 8) {
        unpack_nibbles(blk[t], r);
    } else {
        const int w = odd_word<BITS>(t);
        unpack_odd<BITS>(blk[w], blk[w + 1], odd_shift<BITS>(t), r);
    }
}

}  // namespace qmmk
