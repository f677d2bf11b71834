// Device primitives for the qmm kernels (sm_103a): inline PTX for mbarriers,
// bulk (TMA) and cp.async copies, programmatic dependent launch, the warp-level
// binary16 tensor-core MMA, and the in-register code unpackers.
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
static __device__ __noinline__ void record_bad_copy(uint32_t* err, const void* a, uint64_t b, uint32_t what) {
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
// As mbar_try_wait, but the thread may stay suspended (without issuing) for up
// to `hint_ns` nanoseconds while the phase is incomplete.
__device__ __forceinline__ bool mbar_try_wait_suspend(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Bounded wait on a phase parity; on timeout sets `code` in *err and returns
// false. The first test is inline; the retry loop is out of line (it runs only
// when the phase has not completed yet).
static __device__ __noinline__ bool mbar_wait_slow(uint64_t* bar, uint32_t parity, uint32_t* err, uint32_t code) {
    // each try sleeps until the phase completes or 20 us pass, so a waiting warp
    // leaves the issue slots to the others
    const unsigned long long t0 = global_timer_ns();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait_suspend(bar, parity, 20000u)) return true;
        // after any recorded failure the kernel stops waiting (its output is then
        // incomplete; the host sees the error word) so that no warp spends the
        // limit again; the word is read only every 64 tries, off the path of a
        // wait that ends soon
        if ((n & 63u) == 0 &&
            (*reinterpret_cast<volatile uint32_t*>(err) & (kErrFullWait | kErrEmptyWait | kErrDrainWait)))
            return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            atomicOr(err, code);
            return false;
        }
    }
}
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t* err, uint32_t code) {
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_slow(bar, parity, err, code);
}
// As mbar_wait, for a warp that runs ahead of the one it waits for (a
// producer refilling a slot, a stager waiting for a slot to empty): between
// tries it sleeps about `ns` nanoseconds, leaving the issue slots to the warps
// on the critical path.
static __device__ __noinline__ bool mbar_wait_sleep_slow(uint64_t* bar, uint32_t parity, uint32_t* err, uint32_t code,
                                                         uint32_t ns) {
    const unsigned long long t0 = global_timer_ns();
    for (uint32_t n = 1;; ++n) {
        __nanosleep(ns);
        if (mbar_try_wait(bar, parity)) return true;
        if ((n & 63u) == 0 &&
            (*reinterpret_cast<volatile uint32_t*>(err) & (kErrFullWait | kErrEmptyWait | kErrDrainWait)))
            return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            atomicOr(err, code);
            return false;
        }
    }
}
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t* err, uint32_t code,
                                                uint32_t ns) {
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_sleep_slow(bar, parity, err, code, ns);
}
// Bounded wait for this warp's own copies still in flight after a failure
// (before the CTA exits): unlike mbar_wait it waits even when an error is
// already recorded; on timeout it sets kErrDrainWait and returns false.
static __device__ __noinline__ bool mbar_drain(uint64_t* bar, uint32_t parity, uint32_t* err) {
    const unsigned long long t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait_suspend(bar, parity, 20000u)) return true;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            atomicOr(err, kErrDrainWait);
            return false;
        }
    }
}

// ---- paired fp32 arithmetic ---------------------------------------------------
// One instruction for two lanes of fp32 work; each half is rounded exactly as
// the scalar operation (fmaf, +, *) would round it.
__device__ __forceinline__ void fma_x2(float& d0, float& d1, float a0, float a1, float b0, float b1, float c0,
                                       float c1) {
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
__device__ __forceinline__ void add_x2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ void mul_x2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
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
// 3-D TMA tile load, as tma_load_2d with coordinates (x, y, z).
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
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
// Per-thread asynchronous 4-byte copy (for scale and bias rows that are not
// 16-byte multiples).
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

// Order this thread's earlier generic-proxy shared-memory accesses before its
// later async-proxy (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Named barrier over `count` threads (a multiple of 32).
__device__ __forceinline__ void named_barrier(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ---- shared-memory loads ---------------------------------------------------
// Four 8x8 b16 matrices; lane l gives the row address of row (l & 7) of
// matrix (l >> 3) (16-byte aligned), and receives in register i the 32-bit
// word (l & 3) of row (l >> 2) of matrix i.
__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& d0, uint32_t& d1, uint32_t& d2, uint32_t& d3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(d0), "=r"(d1), "=r"(d2), "=r"(d3)
                 : "r"(addr));
}
// Shared loads at base + a compile-time byte offset ([reg + imm] addressing).
template <int OFF>
__device__ __forceinline__ uint4 lds128_at(uint32_t base) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4 + %5];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(base), "n"(OFF));
    return v;
}
template <int OFF>
__device__ __forceinline__ uint2 lds64_at(uint32_t base) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2 + %3];" : "=r"(v.x), "=r"(v.y) : "r"(base), "n"(OFF));
    return v;
}
template <int OFF>
__device__ __forceinline__ uint32_t lds32_at(uint32_t base) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1 + %2];" : "=r"(v) : "r"(base), "n"(OFF));
    return v;
}
template <int OFF>
__device__ __forceinline__ void ldmatrix_x4_at(uint32_t base, uint32_t& d0, uint32_t& d1, uint32_t& d2, uint32_t& d3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4 + %5];"
                 : "=r"(d0), "=r"(d1), "=r"(d2), "=r"(d3)
                 : "r"(base), "n"(OFF));
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// Per-half max of |a|, |b| of two bfloat16 pairs (the sign bits of the result
// are the xor of the operands' and are masked by the caller).
__device__ __forceinline__ uint32_t bf16x2_absmax(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// ---- tensor-core MMA (warp level) -------------------------------------------
// D = A*B (zero accumulator), m16n8k16, A/B binary16.
__device__ __forceinline__ void mma_f16_zc(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                           uint32_t b0, uint32_t b1) {
    const float z = 0.0f;
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(z));
}
// D = A*B + C, m16n8k16, A/B binary16, C/D fp32.
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---- code unpacking ----------------------------------------------------------
// Every unpacker turns the 8 codes c_0..c_7 a lane owns in one k32 block into
// four binary16x2 registers. A code q placed at bits j..j+bits-1 of the
// mantissa of the binary16 pattern 0x6400 (= 1024.0) is the exact value
// 1024 + q * 2^j (the mantissa has 10 bits). Register r, half h holds code
// slot_code(r, h) with shift slot_shift(r, h); the staged activation in the
// same slot is multiplied by 2^-j, so each product is x * q plus an offset
// x * 1024 * 2^-j that the bias term removes exactly.
constexpr uint32_t kF16x2_1024 = 0x64006400u;

// `magic` is kF16x2_1024, passed in as a run-time value by the hot loop: a
// three-input logic op takes a single immediate, so with both the mask and the
// pattern as literals every (w & mask) | pattern would compile to two ops.

// Slot tables: which code of the k32 block lane t holds in register r, half
// h, and its mantissa shift j. Lane t holds codes 8t .. 8t + 7 of the block,
// except with 8-bit codes, where it holds codes 4t .. 4t + 3 and
// 16 + 4t .. 16 + 4t + 3 (word t of each 16-byte half of the block's row, as
// ldmatrix delivers them).
QMM_HD constexpr int slot_code(int bits, int r, int h) {
    return bits == 2 ? r + 4 * h
         : bits == 3 ? (r < 3 ? (h == 0 ? r : r + 5) : 3 + h)
         : bits == 4 ? (h == 0 ? r : r + 4)
         : bits == 8 ? ((r >> 1) * 4 + (r & 1) + 2 * h)
         : bits == 5 ? (h == 0 ? r : r + 4)
         : /* 6 */     (r < 3 ? (h == 0 ? r : r + 3) : 6 + h);
}
QMM_HD constexpr int block_code(int bits, int t, int r, int h) {
    return bits == 8 ? 4 * t + 16 * (r >> 1) + (r & 1) + 2 * h : 8 * t + slot_code(bits, r, h);
}
QMM_HD constexpr int slot_shift(int bits, int r, int h) {
    return bits == 2 ? 2 * r
         : bits == 3 ? ((r < 3 && h == 0) ? 1 : 0)
         : bits == 4 ? ((r & 1) ? 4 : 0)
         : bits == 8 ? 0
         : bits == 5 ? (h == 0 ? 0 : 4)
         : /* 6 */     ((r < 3 && h == 1) ? 2 : 0);
}

// 4-bit: one word holds the lane's 8 codes, nibble i = code i.
__device__ __forceinline__ void unpack4(uint32_t w, uint32_t (&r)[4], uint32_t magic = kF16x2_1024) {
    r[0] = (w & 0x000F000Fu) | magic;          // c0, c4          (shift 0)
    r[1] = (w & 0x00F000F0u) | magic;          // c1, c5          (shift 4)
    const uint32_t w8 = w >> 8;
    r[2] = (w8 & 0x000F000Fu) | magic;         // c2, c6
    r[3] = (w8 & 0x00F000F0u) | magic;         // c3, c7
}

// 8-bit: two words hold the lane's 8 codes, byte i of w0 = code 4t + i and
// byte i of w1 = code 16 + 4t + i.
__device__ __forceinline__ void unpack8(uint32_t w0, uint32_t w1, uint32_t (&r)[4],
                                        uint32_t magic = kF16x2_1024) {
    r[0] = (w0 & 0x00FF00FFu) | magic;         // bytes 0, 2 of w0
    r[1] = ((w0 >> 8) & 0x00FF00FFu) | magic;  // bytes 1, 3 of w0
    r[2] = (w1 & 0x00FF00FFu) | magic;         // bytes 0, 2 of w1
    r[3] = ((w1 >> 8) & 0x00FF00FFu) | magic;  // bytes 1, 3 of w1
}

// 2-bit: the lane's 8 codes are the 16 bits at bit 16 * (t & 1) of word w.
// `sel` is the byte-permute selector that moves those two bytes to bytes 0
// and 2 (0x4140 for t even, 0x4342 for t odd; selector 4 picks a zero byte),
// after which code q sits at bit 2q of the low half and code q + 4 at bit 2q
// of the high half.
__device__ __forceinline__ void unpack2(uint32_t w, uint32_t sel, uint32_t (&r)[4], uint32_t magic = kF16x2_1024) {
    const uint32_t y = __byte_perm(w, 0u, sel);
    r[0] = (y & 0x00030003u) | magic;          // c0, c4   (shift 0)
    r[1] = (y & 0x000C000Cu) | magic;          // c1, c5   (shift 2)
    r[2] = (y & 0x00300030u) | magic;          // c2, c6   (shift 4)
    r[3] = (y & 0x00C000C0u) | magic;          // c3, c7   (shift 6)
}
QMM_HD constexpr uint32_t unpack2_selector(int t) { return (t & 1) ? 0x4342u : 0x4140u; }

// 3-, 5- or 6-bit: the lane's 8 codes are 3, 5 or 6 bytes starting at byte
// BITS*t of the block; `lo`, `hi` are the two words covering them and `sh`
// (0, 8, 16, 24) the bit offset of the first code inside `lo`.
template <int BITS>
__device__ __forceinline__ void unpack_odd(uint32_t lo, uint32_t hi, uint32_t sh, uint32_t (&r)[4],
                                           uint32_t magic = kF16x2_1024) {
    const uint64_t v = ((static_cast<uint64_t>(hi) << 32) | lo) >> sh;
    if constexpr (BITS == 3) {
        // the 24 code bits sit in the low word: c_i at bit 3i. (c_i, c_{i+5}) are
        // 15 bits apart, so one left shift by 1 puts c_i at bit 1 and c_{i+5} at
        // bit 16 (shifts 1 and 0); c3 and c4 take a shift each.
        const uint32_t u = static_cast<uint32_t>(v);
        r[0] = ((u << 1) & 0x0007000Eu) | magic;               // c0 (shift 1), c5
        r[1] = ((u >> 2) & 0x0007000Eu) | magic;               // c1 (shift 1), c6
        r[2] = ((u >> 5) & 0x0007000Eu) | magic;               // c2 (shift 1), c7
        r[3] = ((u >> 9) & 0x7u) | ((u << 4) & 0x00070000u) | magic;   // c3, c4
    } else if constexpr (BITS == 5) {
        // c_i at bit 0 and c_{i+4} at bit 20 (= 16 + 4) of the same window
#pragma unroll
        for (int i = 0; i < 4; ++i) r[i] = (static_cast<uint32_t>(v >> (5 * i)) & 0x01F0001Fu) | magic;
    } else {
        // c_i at bit 0 and c_{i+3} at bit 18 (= 16 + 2); c6 and c7 from two windows
#pragma unroll
        for (int i = 0; i < 3; ++i) r[i] = (static_cast<uint32_t>(v >> (6 * i)) & 0x00FC003Fu) | magic;
        r[3] = (static_cast<uint32_t>(v >> 36) & 0x3Fu) | (static_cast<uint32_t>(v >> 26) & 0x003F0000u) | magic;
    }
}

// Word index (within a k32 block) and bit shift of lane t's codes for odd widths.
template <int BITS>
__device__ __forceinline__ int odd_word(int t) { return (BITS * t) >> 2; }
template <int BITS>
__device__ __forceinline__ uint32_t odd_shift(int t) { return static_cast<uint32_t>(((BITS * t) & 3) * 8); }

// Unpack lane t's 8 codes of the k32 block starting at `blk` (4-byte aligned).
// Used by the unpack diagnostic.
template <int BITS>
__device__ __forceinline__ void unpack_block(const uint32_t* blk, int t, uint32_t (&r)[4]) {
    if constexpr (BITS == 2) {
        unpack2(blk[t >> 1], unpack2_selector(t), r);
    } else if constexpr (BITS == 4) {
        unpack4(blk[t], r);
    } else if constexpr (BITS == 8) {
        unpack8(blk[t], blk[4 + t], r);
    } else {
        // a block holds BITS words; the next word is read only when it is still
        // inside the block (3-bit lane 3 fits in its first word)
        const int w = odd_word<BITS>(t);
        unpack_odd<BITS>(blk[w], w + 1 < BITS ? blk[w + 1] : 0u, odd_shift<BITS>(t), r);
    }
}

}  // namespace qmmk
