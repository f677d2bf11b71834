// qmm kernels for sm_103a.
//
// Per forward call, in stream order:
//   1. qmm_xprep_kernel   -- stages x once per call: MMA B fragments in the
//                            permuted k order the unpackers produce, the per-group
//                            activation sums XS (the "b*XS" term of the
//                            dequant-after-dot form, vmlx-swift PR #565, LaneQMM
//                            commit) as split binary16 fragments, and one
//                            power-of-two range factor per (row, chunk).
//   2. qmm_main_kernel    -- one CTA per SM; a producer warp streams packed code
//                            rows (TMA 2-D tensor boxes), scales and biases (TMA
//                            boxes, or 4-byte cp.async pieces when a row of them
//                            is not 16-byte aligned) and the staged activations
//                            (one bulk copy per chunk) into a ring of shared-
//                            memory stages; eight consumer warps unpack the
//                            codes in registers and contract them on tensor cores,
//                            reading each code byte once for all M rows (same
//                            page, qwen_qmv_rows_full commit: weights read once per
//                            k-block for all rows). Launched as a programmatic
//                            dependent of (1): code loads start before (1) ends.
//   3. qmm_splitk_reduce_kernel (splits > 1 only) -- sums the fp32 slice
//                            partials in slice order (same page, "JANGH split-K
//                            verify tile" commit: FP32 partials, then a sum).
//
// Per scale group g the main kernel forms, with the unpacked binary16 weights
// A[n,k] = 1024 + q[n,k] * 2^j(k) and the staged activations
// x'[m,k] = f[m,c] * x[m,k] * 2^-j(k) (f a power-of-two range factor per
// activation row and 8-group chunk c, j(k) the code's mantissa shift),
//   P'[m,n,g] = sum_{k in g} x'[m,k] * A[n,k] = f * (P + XSc),
//   XSc[m,g]  = sum_{k in g} x[m,k] * 1024 * 2^-j(k),
// and then
//   y += (1/f) * sum_g s*P'  +  sum_g (b*XS - s*XSc),
// which is  sum_g s*P + b*XS.  The s*P' part is one FMA per accumulator per
// group (plus one per chunk for 1/f); the (b, s) x (XS, -XSc) part is a small
// binary16 MMA per chunk, with XS and XSc split into high and low binary16
// halves so each keeps ~22 bits.
#pragma once

#include <cuda_runtime.h>

#include <type_traits>

#include "qmm_device.cuh"

namespace qmmk {

constexpr int kMaxBanks = 64;

struct BankPtrs {
    const uint32_t* w;
    const uint16_t* s;
    const uint16_t* b;
    void* out;
};

enum OutMode : int { kOutF32 = 0, kOutBF16 = 1, kOutPartial = 2 };

// Kernel parameters. CAP = number of bank slots carried (1 for a single
// projection, kMaxBanks for banked calls), so single calls pass a small block.
struct MainHeader {
    const uint8_t* xprep;   // per chunk: xprep_chunk_bytes(bits, group, MB)
    float* partial;         // [banks][splits][M][N] when out_mode == kOutPartial
    uint32_t* err;          // device error word
    int64_t N;
    int64_t K;
    int64_t row_bytes;      // K*bits/8
    int64_t rows_total;     // banks * splits * N
    int64_t xprep_bytes;    // extent of the staged-activation region (for copy checks)
    int G;                  // K / group
    int C;                  // chunks = ceil(G / 8)
    int splits;
    int M;
    int stages;
    int out_mode;
    int sb_tma;             // scales/biases by TMA boxes (G % 8 == 0), else cp.async
    int sb_vec16;           // scale/bias rows 16-byte aligned (G % 8 == 0)
    int banks;
    int swiglu;             // fused gate/up (the two-bank kernel): out = silu(gate) * up
    float* gate;            // [M][N] fp32 gate results of the current call (swiglu, unsliced)
    uint32_t unpack_magic;  // kF16x2_1024, given at run time so it stays in a register
};

template <int CAP>
struct MainParams {
    MainHeader h;
    BankPtrs bank[CAP];
    CUtensorMap tmw[CAP];   // packed codes: uint8 [N][row_bytes], box kTN x W, swizzled
    CUtensorMap tms[CAP];   // scales: uint16 [N][G], box kTN x 8 (when sb_tma)
    CUtensorMap tmb[CAP];   // biases: same
};

struct ReduceParams {
    const float* partial;
    int64_t N;
    int M;
    int splits;
    int banks;
    int out_bf16;
    int swiglu;             // out[0] = silu(sum of bank 0) * (sum of bank 1)
    void* out[kMaxBanks];
};

// ---------------------------------------------------------------------------
// Work enumeration shared by the producer and the consumers: the flattened
// (bank, split, row) space is cut evenly over the CTAs; a CTA's range is cut at
// (bank, split) boundaries and then into balanced row blocks of <= kTN rows.
// ---------------------------------------------------------------------------
template <bool SWIGLU, typename F>
__device__ __forceinline__ void for_each_row_block(const MainHeader& p, F&& f) {
    const int64_t r_begin = p.rows_total * blockIdx.x / gridDim.x;
    const int64_t r_end = p.rows_total * (blockIdx.x + 1) / gridDim.x;
    int64_t r = r_begin;
    while (r < r_end) {
        const int64_t seg = r / p.N;                                  // bank * splits + split
        const int64_t seg_end = min(r_end, (seg + 1) * p.N);
        const int64_t len = seg_end - r;
        const int nb = static_cast<int>((len + kTN - 1) / kTN);
        // fused gate/up: the flattened space is (split, row) and every row block
        // is run for bank 0 (gate) and then bank 1 (up) by the same CTA
        const int bank = SWIGLU ? 0 : static_cast<int>(seg / p.splits);
        const int split = static_cast<int>(seg % p.splits);
        const int c0 = static_cast<int>(static_cast<int64_t>(split) * p.C / p.splits);
        const int c1 = static_cast<int>(static_cast<int64_t>(split + 1) * p.C / p.splits);
        for (int ib = 0; ib < nb; ++ib) {
            const int64_t a = r + len * ib / nb;
            const int64_t e = r + len * (ib + 1) / nb;
            if constexpr (SWIGLU) {
                if (!f(0, split, a - seg * p.N, static_cast<int>(e - a), c0, c1)) return;
                if (!f(1, split, a - seg * p.N, static_cast<int>(e - a), c0, c1)) return;
            } else {
                if (!f(bank, split, a - seg * p.N, static_cast<int>(e - a), c0, c1)) return;
            }
        }
        r = seg_end;
    }
}

// ---------------------------------------------------------------------------
// 1. Activation staging.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t pack_half2(__half lo, __half hi) {
    return static_cast<uint32_t>(__half_as_ushort(lo)) | (static_cast<uint32_t>(__half_as_ushort(hi)) << 16);
}
__device__ __forceinline__ float bf16_bits_to_float(uint32_t v) { return __uint_as_float(v << 16); }

// 16 bytes of x through L2 (x may have been written on other SMs just before).
__device__ __forceinline__ uint4 ld_cg_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// One CTA per chunk, one warp per scale group of the chunk. For 8-row tile j,
// lane (g, t) of warp gg holds activation row m = 8j + g and, of each k32 block
// vb of the group, the 8-code piece 4vb + t (codes 32vb + 8t .. 32vb + 8t + 7),
// so the four lanes of a quad hold the group's codes of one row:
//   XS[m,g]  = sum_{k in g} x[m,k],   XSc[m,g] = sum_{k in g} x[m,k] * 1024 * 2^-j(k),
// summed over each piece in code order, then over the lane's pieces and the
// quad in a fixed tree order. f = 2^(14 - e) from the binary exponent e of the
// chunk's largest |x| (clamped so f and 1/f stay normal), sigma = 2^(e' - 13)
// from the largest |XS|, |XSc| of the chunk (exponent e'), both over the eight
// groups through shared memory. Rows m >= M and codes past the end of K stage
// as zeros (f = sigma = 1).
template <int BITS, int GROUP, int MB>
__global__ void __launch_bounds__(kXprepThreads)
qmm_xprep_kernel(const uint16_t* __restrict__ x, int M, int64_t K, int G, uint8_t* __restrict__ xprep) {
    static_assert(kXprepThreads == 32 * kGPC, "one warp per scale group");
    constexpr int CK = kGPC * GROUP;                 // codes per chunk
    constexpr int VPG = GROUP / 32;                  // k32 blocks per group
    constexpr int NT = n8_tiles(MB);
    constexpr int XFB = xprep_frag_bytes(BITS, GROUP, MB);
    constexpr int XPB = xprep_chunk_bytes(BITS, GROUP, MB);

    // The main kernel may start loading weights while this runs. This kernel may
    // itself be launched as a programmatic dependent of whatever ran before it on
    // the stream, so it waits for that work (which may produce x, or still read
    // the staging buffer) before touching x or the buffer.
    griddep_launch_dependents();
    griddep_wait();

    __shared__ float s_xs[MB][kGPC];      // XS
    __shared__ float s_xsc[MB][kGPC];     // XSc
    __shared__ uint32_t s_mag[MB][kGPC];  // largest |x| bit pattern of the group

    const int c = blockIdx.x;
    const int gg = threadIdx.x >> 5;                 // this warp's group
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2;
    const int t = lane & 3;
    const int64_t k0 = static_cast<int64_t>(c) * CK;
    const int kc = min(kGPC, G - c * kGPC) * GROUP;  // codes of this chunk inside K
    const bool x16 = (reinterpret_cast<uintptr_t>(x) & 15) == 0;

    // every load first
    uint4 v[NT][VPG];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        const int m = 8 * j + g;
        const uint16_t* row = x + static_cast<int64_t>(m) * K + k0;
#pragma unroll
        for (int u = 0; u < VPG; ++u) {
            const int k = 32 * (gg * VPG + u) + 8 * t;
            v[j][u] = make_uint4(0, 0, 0, 0);
            if (m < M && k < kc) {
                if (x16) {
                    v[j][u] = ld_cg_v4(row + k);
                } else {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        w[e] = static_cast<uint32_t>(__ldcg(row + k + 2 * e)) |
                               (static_cast<uint32_t>(__ldcg(row + k + 2 * e + 1)) << 16);
                    v[j][u] = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
        }
    }
    // group sums and magnitude of each row
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        float s = 0.0f, sc = 0.0f;
        uint32_t mag = 0;
#pragma unroll
        for (int u = 0; u < VPG; ++u) {
            const uint32_t wv[4] = {v[j][u].x, v[j][u].y, v[j][u].z, v[j][u].w};
            float ps = 0.0f, psc = 0.0f;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const uint32_t hbits = (wv[e >> 1] >> (16 * (e & 1))) & 0xFFFFu;
                const float xv = bf16_bits_to_float(hbits);
                ps += xv;
                psc = fmaf(xv, 1024.0f / static_cast<float>(1 << code_shift(BITS, e)), psc);
                mag = max(mag, hbits & 0x7FFFu);
            }
            s = u == 0 ? ps : s + ps;
            sc = u == 0 ? psc : sc + psc;
        }
        s += __shfl_xor_sync(0xFFFFFFFFu, s, 1);
        sc += __shfl_xor_sync(0xFFFFFFFFu, sc, 1);
        s += __shfl_xor_sync(0xFFFFFFFFu, s, 2);
        sc += __shfl_xor_sync(0xFFFFFFFFu, sc, 2);
        mag = max(mag, __shfl_xor_sync(0xFFFFFFFFu, mag, 1));
        mag = max(mag, __shfl_xor_sync(0xFFFFFFFFu, mag, 2));
        if (t == 0) {
            s_xs[8 * j + g][gg] = s;
            s_xsc[8 * j + g][gg] = sc;
            s_mag[8 * j + g][gg] = mag;
        }
    }
    __syncthreads();

    uint8_t* out = xprep + static_cast<size_t>(c) * XPB;
    uint4* frag = reinterpret_cast<uint4*>(out);
    uint4* bias = reinterpret_cast<uint4*>(out + XFB);
    float* tail = reinterpret_cast<float*>(out + XFB + xprep_bias_bytes(MB));
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        const int m = 8 * j + g;
        float amax = 0.0f;
        uint32_t mag = 0;
#pragma unroll
        for (int q = 0; q < kGPC; ++q) {
            amax = fmaxf(amax, fmaxf(fabsf(s_xs[m][q]), fabsf(s_xsc[m][q])));
            mag = max(mag, s_mag[m][q]);
        }
        // sigma puts the largest |XS/sigma|, |XSc/sigma| in [2^13, 2^14): inside the
        // binary16 range with room to spare
        float sg = 1.0f;
        if (amax > 0.0f && amax <= 3.0e38f) sg = ldexpf(1.0f, ilogbf(amax) - 13);
        const float rsig = 1.0f / sg;    // exact: power of two
        // every f*x*2^-j is below 2^15, and any x within 2^27 of the largest is
        // exact in binary16
        int ex = 0;
        if (mag != 0) ex = min(127, max(-100, static_cast<int>(mag >> 7) - 127));
        const float f = (mag != 0) ? ldexpf(1.0f, 14 - ex) : 1.0f;
        if (gg == 0 && t == 0) {
            tail[m] = sg;
            tail[MB + m] = 1.0f / f;   // exact: power of two
        }
        // MMA B fragments of this group's k32 blocks, in the unpackers' slot order
#pragma unroll
        for (int u = 0; u < VPG; ++u) {
            const int vb = gg * VPG + u;
            const uint32_t wv[4] = {v[j][u].x, v[j][u].y, v[j][u].z, v[j][u].w};
            uint32_t r[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int c0 = slot_code(BITS, q, 0), c1 = slot_code(BITS, q, 1);
                const float lo = bf16_bits_to_float((wv[c0 >> 1] >> (16 * (c0 & 1))) & 0xFFFFu) * f *
                                 (1.0f / static_cast<float>(1 << slot_shift(BITS, q, 0)));
                const float hi = bf16_bits_to_float((wv[c1 >> 1] >> (16 * (c1 & 1))) & 0xFFFFu) * f *
                                 (1.0f / static_cast<float>(1 << slot_shift(BITS, q, 1)));
                r[q] = pack_half2(__float2half_rn(lo), __float2half_rn(hi));
            }
            frag[(vb * NT + j) * 32 + lane] = make_uint4(r[0], r[1], r[2], r[3]);
        }
        // bias-term fragments of tile j (warp j): groups 2t and 2t + 1 of row m,
        // XS and -XSc over sigma, each as a high and a low binary16 half
        if (gg == j) {
            const float v0 = s_xs[m][2 * t] * rsig;
            const float v1 = s_xs[m][2 * t + 1] * rsig;
            const float w0 = -s_xsc[m][2 * t] * rsig;
            const float w1 = -s_xsc[m][2 * t + 1] * rsig;
            const __half v0h = __float2half_rn(v0), v1h = __float2half_rn(v1);
            const __half w0h = __float2half_rn(w0), w1h = __float2half_rn(w1);
            const __half v0l = __float2half_rn(v0 - __half2float(v0h)), v1l = __float2half_rn(v1 - __half2float(v1h));
            const __half w0l = __float2half_rn(w0 - __half2float(w0h)), w1l = __float2half_rn(w1 - __half2float(w1h));
            bias[j * 32 + lane] =
                make_uint4(pack_half2(v0h, v1h), pack_half2(w0h, w1h), pack_half2(v0l, v1l), pack_half2(w0l, w1l));
        }
    }
}

// ---------------------------------------------------------------------------
// 2. Main kernel.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void consumer_barrier() {
    asm volatile("bar.sync 1, %0;" ::"n"(kNCW * 32) : "memory");
}

// Byte offset, inside a stage, of byte b of weight-tile row r (TMA box layout
// with the W-byte swizzle: 16-byte chunk bits 4.. of the in-box address are
// XORed with its bits 7..).
template <int BITS, int GROUP>
__device__ __forceinline__ int wtile_off(int r, int b) {
    constexpr int W = wbox_width(BITS, GROUP);
    constexpr int LW = log2i(W);
    constexpr int MASK = W / 16 - 1;
    const int lin = r * W + (b & (W - 1));
    return ((b >> LW) << (LW + 7)) + (lin ^ (((lin >> 7) & MASK) << 4));
}

template <int BITS, int GROUP, int MB, int CAP>
__global__ void __launch_bounds__(kThreads, 1) qmm_main_kernel(const __grid_constant__ MainParams<CAP> P) {
    constexpr int VB = vblocks_per_group(BITS, GROUP);
    constexpr int NT = n8_tiles(MB);
    constexpr int BB = vblock_bytes(BITS);
    constexpr int RB = chunk_row_bytes(BITS, GROUP);
    constexpr int W = wbox_width(BITS, GROUP);
    constexpr int NBOX = wbox_count(BITS, GROUP);
    constexpr int SW = stage_weight_bytes(BITS, GROUP);
    constexpr int SSB = stage_sb_bytes();
    constexpr int XFB = xprep_frag_bytes(BITS, GROUP, MB);
    constexpr int XPB = xprep_chunk_bytes(BITS, GROUP, MB);
    constexpr int SB = stage_bytes(BITS, GROUP, MB);
    constexpr int NV = kGroupsPerWarp * VB;        // k32 blocks per consumer warp per stage
    const MainHeader& p = P.h;
    // the two-bank parameter block is the fused gate/up projection's
    constexpr bool SWIGLU = CAP == 2;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte aligned ring base, derived by pointer arithmetic on the shared
    // array so every access below stays a shared-memory access
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int S = p.stages;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * SB);
    uint64_t* empty = full + S;
    float* scratch = reinterpret_cast<float*>(smem + S * SB + S * 16);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1 + 32);      // producer lane 0 (expect_tx) + 32 cp.async arrivals
            mbar_init(&empty[i], kNCW);
        }
        fence_barrier_init();
    }
    __syncthreads();
    griddep_launch_dependents();

    if (warp == kNCW) {
        // ------------------------------ producer ------------------------------
        // Lane 0 issues the TMA boxes of a stage (packed codes, scales, biases)
        // and the bulk copy of its staged activations. Scales and biases whose
        // rows are not 16-byte multiples go through per-lane cp.async instead.
        const uint64_t pol = policy_evict_first();
        if (lane == 0)
            for (int i = 0; i < p.banks && i < CAP; ++i) {
                prefetch_tensormap(&P.tmw[i]);
                if (p.sb_tma) {
                    prefetch_tensormap(&P.tms[i]);
                    prefetch_tensormap(&P.tmb[i]);
                }
            }
        const uint32_t tx_stage =
            static_cast<uint32_t>(NBOX * kTN * W + (p.sb_tma ? 2 * SSB : 0) + XPB);
        uint32_t it = 0;
        int pslot = 0;            // it % S, kept incrementally (S is a run-time value)
        uint32_t pround = 0;      // it / S
        bool waited = false;
        bool ok = true;
        int npend = 0;
        int pend_slot[kMaxStages];
        int pend_chunk[kMaxStages];
        auto issue_xprep = [&](int slot, int c) {
            uint8_t* d = smem + slot * SB + SW + 2 * SSB;
            const int64_t off = static_cast<int64_t>(c) * XPB;
            if (slot < 0 || slot >= S || c < 0 || off + XPB > p.xprep_bytes ||
                ((reinterpret_cast<uintptr_t>(p.xprep + off) | smem_u32(d)) & 15)) {
                record_bad_copy(p.err, p.xprep + off, static_cast<uint64_t>(slot) << 32 | static_cast<uint32_t>(c), 3u);
                return;
            }
            bulk_g2s(d, p.xprep + off, XPB, &full[slot]);
        };
        auto flush_pending = [&]() {
            griddep_wait();   // the staged activations of this call are ready
            waited = true;
            if (lane == 0)
                for (int i = 0; i < npend; ++i) issue_xprep(pend_slot[i], pend_chunk[i]);
            npend = 0;
        };
        for_each_row_block<SWIGLU>(p, [&](int bank, int split, int64_t n0, int rows, int c0, int c1) -> bool {
            (void)split;
            const BankPtrs bp = P.bank[bank];
            // the cp.async path for scales/biases checks its buffers once per row block
            const bool sb_ok = p.sb_tma ||
                (n0 >= 0 && rows >= 1 && rows <= kTN && n0 + rows <= p.N && c0 >= 0 && c1 <= p.C &&
                 ((reinterpret_cast<uintptr_t>(bp.s) | reinterpret_cast<uintptr_t>(bp.b)) & 3) == 0);
            if (!sb_ok && lane == 0) record_bad_copy(p.err, bp.s, static_cast<uint64_t>(rows), 4u);
            for (int c = c0; c < c1; ++c) {
                const int slot = pslot;
                // After a timed-out wait the error is recorded and no further waits are
                // made; the loop still runs to the end so that every warp finishes.
                // (The slot's previous use was in round pround - 1: parity pround ^ 1.)
                if (it >= static_cast<uint32_t>(S) && ok &&
                    !mbar_wait(&empty[slot], (pround ^ 1u) & 1u, p.err, kErrEmptyWait))
                    ok = false;
                uint8_t* st = smem + slot * SB;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&full[slot], tx_stage);
                    const int y = static_cast<int>(n0);
#pragma unroll
                    for (int bi = 0; bi < NBOX; ++bi)
                        tma_load_2d(st + bi * (kTN * W), &P.tmw[bank], c * RB + bi * W, y, &full[slot], pol);
                    if (p.sb_tma) {
                        tma_load_2d(st + SW, &P.tms[bank], c * kGPC, y, &full[slot], pol);
                        tma_load_2d(st + SW + SSB, &P.tmb[bank], c * kGPC, y, &full[slot], pol);
                    }
                }
                __syncwarp();
                if (!p.sb_tma && sb_ok) {
                    const int ng = min(kGPC, p.G - c * kGPC);
                    const int nq = ng >> 1;   // 4-byte pieces per row
                    uint8_t* sdst = st + SW;
                    uint8_t* bdst = sdst + SSB;
                    const uint16_t* ssrc = bp.s + n0 * p.G + c * kGPC;
                    const uint16_t* bsrc = bp.b + n0 * p.G + c * kGPC;
                    for (int i = lane; i < rows * nq; i += 32) {
                        const int r = i / nq, q = i - (i / nq) * nq;
                        cp_async_4(sdst + r * 16 + 4 * q, ssrc + static_cast<int64_t>(r) * p.G + 2 * q);
                        cp_async_4(bdst + r * 16 + 4 * q, bsrc + static_cast<int64_t>(r) * p.G + 2 * q);
                    }
                }
                cp_async_arrive_noinc(&full[slot]);
                if (waited) {
                    if (lane == 0) issue_xprep(slot, c);
                } else {
                    pend_slot[npend] = slot;
                    pend_chunk[npend] = c;
                    if (++npend == S) flush_pending();
                }
                ++it;
                if (++pslot == S) {
                    pslot = 0;
                    ++pround;
                }
            }
            return true;
        });
        if (!waited) flush_pending();
        // This warp's own cp.async copies must land before it exits.
        cp_async_wait_all();
        if (!ok) {
            // Give the copies already issued a bounded chance to land before exiting.
            const uint32_t first = it > static_cast<uint32_t>(S) ? it - S : 0u;
            for (uint32_t i = first; i < it; ++i)
                if (!mbar_wait(&full[i % S], (i / S) & 1u, p.err, kErrDrainWait)) break;
        }
        return;
    }

    // -------------------------------- consumers --------------------------------
    const uint32_t magic = p.unpack_magic;
    const int g = lane >> 2;
    const int t = lane & 3;
    const uint32_t sel2 = unpack2_selector(t);   // 2-bit codes only
    const int sp = warp % kSlabPairs;        // slabs sp and sp + 4
    const int kh = warp / kSlabPairs;        // chunk groups 4*kh .. 4*kh + 3
    const int gbase = kh * kGroupsPerWarp;
    const int vbw = gbase * VB;              // first k32 block of this warp in a chunk
    // Offsets of this lane's codes in each of the warp's k32 blocks, for a tile
    // row r with r % 8 == 0 (add r * W): box base + swizzled 16-byte chunk +
    // byte. 4-bit: one word (block = one 16-byte chunk); 8-bit: two words
    // (block = two chunks). Both use 128-byte boxes.
    int cx[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int vb = vbw + i;
        if constexpr (BITS == 4)
            cx[i] = ((vb >> 3) << 14) + ((((vb & 7) ^ g) << 4) | (4 * t));
        else if constexpr (BITS == 8)
            cx[i] = ((vb >> 2) << 14) + (((((2 * vb + (t >> 1)) & 7) ^ g) << 4) | (8 * (t & 1)));
        else
            cx[i] = 0;
    }
    int cslot = 0;            // stage index % S, kept incrementally
    uint32_t cphase = 0;      // (stage index / S) & 1
    bool ok = true;
    for_each_row_block<SWIGLU>(p, [&](int bank, int split, int64_t n0, int rows, int c0, int c1) -> bool {
        const int nsl = (rows + kSlab - 1) / kSlab;
        bool act[kSPW];
        int row0[kSPW];
#pragma unroll
        for (int sw = 0; sw < kSPW; ++sw) {
            const int slab = sp + sw * kSlabPairs;
            act[sw] = slab < nsl;
            row0[sw] = slab * kSlab + g;
        }
        float acc[kSPW][NT][4];
#pragma unroll
        for (int sw = 0; sw < kSPW; ++sw)
#pragma unroll
            for (int j = 0; j < NT; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[sw][j][e] = 0.0f;

        for (int c = c0; c < c1; ++c) {
            const int slot = cslot;
            // a timed-out wait is recorded; the warp then stops waiting but keeps the
            // same control flow, so the consumer barriers below are always reached
            if (ok && !mbar_wait(&full[slot], cphase, p.err, kErrFullWait)) ok = false;
            const int ng = min(kGPC, p.G - c * kGPC);
            const uint8_t* st = smem + slot * SB;
            const uint8_t* wst = st;
            const uint16_t* sst = reinterpret_cast<const uint16_t*>(st + SW);
            const uint16_t* bst = reinterpret_cast<const uint16_t*>(st + SW + SSB);
            const uint4* xfr = reinterpret_cast<const uint4*>(st + SW + 2 * SSB);
            const uint4* xbias = reinterpret_cast<const uint4*>(st + SW + 2 * SSB + XFB);
            const float* xsig = reinterpret_cast<const float*>(st + SW + 2 * SSB + XFB + xprep_bias_bytes(MB));
            const float* xrf = xsig + MB;            // 1/f per activation row

            // this warp's 4 scales for each of its slab rows (binary16 pairs)
            uint2 sv0[kSPW], sv1[kSPW];
#pragma unroll
            for (int sw = 0; sw < kSPW; ++sw) {
                sv0[sw] = *reinterpret_cast<const uint2*>(sst + row0[sw] * 8 + gbase);
                sv1[sw] = *reinterpret_cast<const uint2*>(sst + (row0[sw] + 8) * 8 + gbase);
            }

            // The group loop, instantiated twice: without any guard for the common
            // case (full chunk, both slabs live) so loads of later groups can be
            // scheduled under the tensor-core work of earlier ones, and guarded for
            // partial chunks and partial row blocks.
            // Per-chunk sums sum_g s*P' (still scaled by f), folded into acc with 1/f.
            float accc[kSPW][NT][4];
            auto groups = [&](auto full_tag) {
                constexpr bool FULL = decltype(full_tag)::value;
                if constexpr (!FULL) {
#pragma unroll
                    for (int sw = 0; sw < kSPW; ++sw)
#pragma unroll
                        for (int j = 0; j < NT; ++j)
#pragma unroll
                            for (int e = 0; e < 4; ++e) accc[sw][j][e] = 0.0f;
                }
#pragma unroll
                for (int gl = 0; gl < kGroupsPerWarp; ++gl) {
                    if (!FULL && gbase + gl >= ng) continue;
                    float P[kSPW][NT][4];
#pragma unroll
                    for (int v = 0; v < VB; ++v) {
                        const int vi = gl * VB + v;          // block index within the warp
                        const int vb = vbw + vi;             // block index within the chunk
                        uint4 bf[NT];
#pragma unroll
                        for (int j = 0; j < NT; ++j) bf[j] = xfr[(vb * NT + j) * 32 + lane];
#pragma unroll
                        for (int sw = 0; sw < kSPW; ++sw) {
                            if (!FULL && !act[sw]) continue;
                            uint32_t ra[4], rb[4];
                            if constexpr (BITS == 4) {
                                const uint8_t* a0 = wst + (row0[sw] - g) * W + cx[vi];
                                unpack4(*reinterpret_cast<const uint32_t*>(a0 + g * W), ra, magic);
                                unpack4(*reinterpret_cast<const uint32_t*>(a0 + (g + 8) * W), rb, magic);
                            } else if constexpr (BITS == 8) {
                                const uint8_t* a0 = wst + (row0[sw] - g) * W + cx[vi];
                                const uint2 u0 = *reinterpret_cast<const uint2*>(a0 + g * W);
                                const uint2 u1 = *reinterpret_cast<const uint2*>(a0 + (g + 8) * W);
                                unpack8(u0.x, u0.y, ra, magic);
                                unpack8(u1.x, u1.y, rb, magic);
                            } else if constexpr (BITS == 2) {
                                // lane t's 8 codes are half of word t / 2 of the block
                                const int b0 = vb * BB + 4 * odd_word<BITS>(t);
                                const uint32_t w0 = *reinterpret_cast<const uint32_t*>(wst + wtile_off<BITS, GROUP>(row0[sw], b0));
                                const uint32_t w1 = *reinterpret_cast<const uint32_t*>(wst + wtile_off<BITS, GROUP>(row0[sw] + 8, b0));
                                unpack2(w0, sel2, ra, magic);
                                unpack2(w1, sel2, rb, magic);
                            } else {
                                const int b0 = vb * BB + 4 * odd_word<BITS>(t);
                                const int r0 = row0[sw], r1 = row0[sw] + 8;
                                const uint32_t lo0 = *reinterpret_cast<const uint32_t*>(wst + wtile_off<BITS, GROUP>(r0, b0));
                                const uint32_t hi0 = *reinterpret_cast<const uint32_t*>(wst + wtile_off<BITS, GROUP>(r0, b0 + 4));
                                const uint32_t lo1 = *reinterpret_cast<const uint32_t*>(wst + wtile_off<BITS, GROUP>(r1, b0));
                                const uint32_t hi1 = *reinterpret_cast<const uint32_t*>(wst + wtile_off<BITS, GROUP>(r1, b0 + 4));
                                unpack_odd<BITS>(lo0, hi0, odd_shift<BITS>(t), ra, magic);
                                unpack_odd<BITS>(lo1, hi1, odd_shift<BITS>(t), rb, magic);
                            }
#pragma unroll
                            for (int j = 0; j < NT; ++j) {
                                if (v == 0)
                                    mma_f16_zc(P[sw][j], ra[0], rb[0], ra[1], rb[1], bf[j].x, bf[j].y);
                                else
                                    mma_f16(P[sw][j], ra[0], rb[0], ra[1], rb[1], bf[j].x, bf[j].y);
                                mma_f16(P[sw][j], ra[2], rb[2], ra[3], rb[3], bf[j].z, bf[j].w);
                            }
                        }
                    }
#pragma unroll
                    for (int sw = 0; sw < kSPW; ++sw) {
                        if (!FULL && !act[sw]) continue;
                        const uint32_t w0 = (gl < 2) ? sv0[sw].x : sv0[sw].y;
                        const uint32_t w1 = (gl < 2) ? sv1[sw].x : sv1[sw].y;
                        const float s0 = __half2float(__ushort_as_half(static_cast<uint16_t>(w0 >> (16 * (gl & 1)))));
                        const float s1 = __half2float(__ushort_as_half(static_cast<uint16_t>(w1 >> (16 * (gl & 1)))));
#pragma unroll
                        for (int j = 0; j < NT; ++j) {
                            if (FULL && gl == 0) {
                                accc[sw][j][0] = s0 * P[sw][j][0];
                                accc[sw][j][1] = s0 * P[sw][j][1];
                                accc[sw][j][2] = s1 * P[sw][j][2];
                                accc[sw][j][3] = s1 * P[sw][j][3];
                            } else {
                                accc[sw][j][0] = fmaf(s0, P[sw][j][0], accc[sw][j][0]);
                                accc[sw][j][1] = fmaf(s0, P[sw][j][1], accc[sw][j][1]);
                                accc[sw][j][2] = fmaf(s1, P[sw][j][2], accc[sw][j][2]);
                                accc[sw][j][3] = fmaf(s1, P[sw][j][3], accc[sw][j][3]);
                            }
                        }
                    }
                }
            };
            if (ng == kGPC && act[0] && act[1])
                groups(std::true_type{});
            else
                groups(std::false_type{});
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                const float2 rf = *reinterpret_cast<const float2*>(xrf + 8 * j + 2 * t);
#pragma unroll
                for (int sw = 0; sw < kSPW; ++sw) {
                    if (!act[sw]) continue;
                    acc[sw][j][0] = fmaf(rf.x, accc[sw][j][0], acc[sw][j][0]);
                    acc[sw][j][1] = fmaf(rf.y, accc[sw][j][1], acc[sw][j][1]);
                    acc[sw][j][2] = fmaf(rf.x, accc[sw][j][2], acc[sw][j][2]);
                    acc[sw][j][3] = fmaf(rf.y, accc[sw][j][3], acc[sw][j][3]);
                }
            }

            // bias and offset terms of the chunk, (b | s) x (XS | -XSc) / sigma:
            // K half kh takes slab kh of its pair
#pragma unroll
            for (int sw = 0; sw < kSPW; ++sw) {
                if (sw != kh || !act[sw]) continue;
                uint32_t a0 = *reinterpret_cast<const uint32_t*>(bst + row0[sw] * 8 + 2 * t);
                uint32_t a1 = *reinterpret_cast<const uint32_t*>(bst + (row0[sw] + 8) * 8 + 2 * t);
                uint32_t a2 = *reinterpret_cast<const uint32_t*>(sst + row0[sw] * 8 + 2 * t);
                uint32_t a3 = *reinterpret_cast<const uint32_t*>(sst + (row0[sw] + 8) * 8 + 2 * t);
                if (ng < kGPC) {
                    // groups past the end of K: stale shared memory, zero it
                    const uint32_t keep = (2 * t + 1 < ng) ? 0xFFFFFFFFu : (2 * t < ng ? 0x0000FFFFu : 0u);
                    a0 &= keep;
                    a1 &= keep;
                    a2 &= keep;
                    a3 &= keep;
                }
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    const uint4 bb = xbias[j * 32 + lane];
                    float D[4];
                    mma_f16_zc(D, a0, a1, a2, a3, bb.x, bb.y);
                    mma_f16(D, a0, a1, a2, a3, bb.z, bb.w);
                    const float2 sg = *reinterpret_cast<const float2*>(xsig + 8 * j + 2 * t);
                    acc[sw][j][0] = fmaf(sg.x, D[0], acc[sw][j][0]);
                    acc[sw][j][1] = fmaf(sg.y, D[1], acc[sw][j][1]);
                    acc[sw][j][2] = fmaf(sg.x, D[2], acc[sw][j][2]);
                    acc[sw][j][3] = fmaf(sg.y, D[3], acc[sw][j][3]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
            if (++cslot == S) {
                cslot = 0;
                cphase ^= 1u;
            }
        }

        // combine the two K halves in a fixed order: (first half) + (second half)
        float* sc = scratch + ((sp * kSPW) * NT * 4) * 32;
        if (kh == 1) {
#pragma unroll
            for (int sw = 0; sw < kSPW; ++sw)
#pragma unroll
                for (int j = 0; j < NT; ++j)
#pragma unroll
                    for (int e = 0; e < 4; ++e) sc[((sw * NT + j) * 4 + e) * 32 + lane] = acc[sw][j][e];
        }
        consumer_barrier();
        if (kh == 0) {
            const BankPtrs bp = P.bank[bank];
#pragma unroll
            for (int sw = 0; sw < kSPW; ++sw) {
                if (!act[sw]) continue;
#pragma unroll
                for (int j = 0; j < NT; ++j) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int nl = row0[sw] + 8 * h;
                        if (nl >= rows) continue;
                        const int64_t n = n0 + nl;
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int m = 8 * j + 2 * t + e;
                            if (m >= p.M) continue;
                            float v = acc[sw][j][2 * h + e] + sc[((sw * NT + j) * 4 + 2 * h + e) * 32 + lane];
                            if (p.out_mode == kOutPartial) {
                                p.partial[((static_cast<int64_t>(bank) * p.splits + split) * p.M + m) * p.N + n] = v;
                                continue;
                            }
                            if constexpr (SWIGLU) {
                                // gate pass: keep the fp32 gate; up pass: the same thread
                                // wrote this (m, n) gate in the gate pass of this row block
                                if (bank == 0) {
                                    p.gate[m * p.N + n] = v;
                                    continue;
                                }
                                const float gv = p.gate[m * p.N + n];
                                v = gv / (1.0f + expf(-gv)) * v;
                            }
                            if (p.out_mode == kOutF32) {
                                static_cast<float*>(bp.out)[m * p.N + n] = v;
                            } else {
                                static_cast<__nv_bfloat16*>(bp.out)[m * p.N + n] = __float2bfloat16_rn(v);
                            }
                        }
                    }
                }
            }
        }
        consumer_barrier();   // the scratch is free again
        return true;
    });
    (void)ok;
}

// ---------------------------------------------------------------------------
// 3. Split-K reduce: out = sum_{s=0..S-1} partial[s] in slice order.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kReduceThreads) qmm_splitk_reduce_kernel(const __grid_constant__ ReduceParams p);

// ---------------------------------------------------------------------------
// Diagnostic unpack: one thread per (row, k32 block, lane position t). Runs the
// main kernel's unpacker and reads each code back out of its binary16 value
// 1024 + q * 2^j (0xFF where the pattern is not of that form).
// ---------------------------------------------------------------------------
template <int BITS>
__global__ void __launch_bounds__(256) qmm_unpack_kernel(const uint32_t* __restrict__ w, int64_t K, int64_t N,
                                                         uint8_t* __restrict__ codes) {
    constexpr int BB = vblock_bytes(BITS);
    const int64_t vbk = K / 32;                                  // k32 blocks per row
    const int64_t total = N * vbk * 4;
    const int64_t row_bytes = K * BITS / 8;
    for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int t = static_cast<int>(idx & 3);
        const int64_t rest = idx >> 2;
        const int64_t vb = rest % vbk;
        const int64_t n = rest / vbk;
        const uint32_t* blk = reinterpret_cast<const uint32_t*>(reinterpret_cast<const uint8_t*>(w) + n * row_bytes + vb * BB);
        uint32_t r[4];
        unpack_block<BITS>(blk, t, r);
        uint8_t* out = codes + n * K + vb * 32 + 8 * t;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t v = (r[q] >> (16 * h)) & 0xFFFFu;
                const int j = slot_shift(BITS, q, h);
                const uint32_t mant = v & 0x3FFu;
                const bool okv = (v & 0xFC00u) == 0x6400u && (mant & ((1u << j) - 1u)) == 0 && (mant >> j) < (1u << BITS);
                out[slot_code(BITS, q, h)] = okv ? static_cast<uint8_t>(mant >> j) : static_cast<uint8_t>(0xFF);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Host-side launch helpers (defined per code width in qmm_inst_b*.cu).
// ---------------------------------------------------------------------------
struct LaunchCfg {
    const uint16_t* x;
    int M;
    int mb;            // 8 or 16
    int ctas;
    int smem;
    cudaStream_t stream;
};

template <int BITS>
cudaError_t configure_kernels(int group, int mb, int smem_bytes);

// Weight-box width for a format (host side, for encoding tensor maps).
inline int weight_box_width(int bits, int group) { return wbox_width(bits, group); }
template <int BITS>
cudaError_t launch_forward(int group, const LaunchCfg& L, const MainParams<1>* single, const MainParams<kMaxBanks>* banked,
                           const MainParams<2>* fused);
template <int BITS>
cudaError_t launch_unpack(const uint32_t* w, int64_t K, int64_t N, uint8_t* codes, cudaStream_t stream);

cudaError_t launch_reduce(const ReduceParams& rp, int64_t elems, cudaStream_t stream);

}  // namespace qmmk
