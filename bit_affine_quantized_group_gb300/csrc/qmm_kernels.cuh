// qmm kernels for sm_103a.
//
// Per forward call, in stream order:
//   1. qmm_main_kernel    -- one CTA per SM, launched as a programmatic
//                            dependent of the preceding work on the stream.
//                            A producer warp streams packed code rows (TMA 2-D
//                            tensor boxes), scales and biases (TMA boxes, or
//                            4-byte cp.async pieces when a row of them is not
//                            16-byte aligned) into a ring of shared-memory
//                            weight stages from the moment the CTA starts.
//                            Once the preceding work has finished, staging
//                            warps load each chunk's raw activation rows (one
//                            3-D TMA box per 8-row tile) into a separate ring
//                            of activation slots and turn them into the
//                            chunk's tensor-core fragments, the per-group
//                            activation sums XS (the "b*XS" term of the
//                            dequant-after-dot form, vmlx-swift PR #565,
//                            LaneQMM commit) and the range factors. Eight
//                            consumer warps unpack the codes in registers and
//                            contract them on tensor cores, reading each code
//                            byte once for all M rows (same page,
//                            qwen_qmv_rows_full commit: weights read once per
//                            k-block for all rows).
//   2. qmm_splitk_reduce_kernel (splits > 1 only) -- sums the fp32 slice
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
// halves so each keeps ~22 bits. The staging warps obtain f*XS and f*XSc/1024
// from the staged fragments themselves with a tensor-core MMA against a
// constant selector (column 2q sums group q with weights 2^j, column 2q + 1
// with weights 1).
#pragma once

#include <cuda_runtime.h>

#include <type_traits>

#include "qmm_device.cuh"

namespace qmmk {

// f(integral_constant<int, I>) for I = B .. E - 1, so that I is a compile-time
// constant inside f (shared-memory offsets become load immediates).
template <int B, int E, typename F>
__device__ __forceinline__ void static_for(F&& f) {
    if constexpr (B < E) {
        f(std::integral_constant<int, B>{});
        static_for<B + 1, E>(f);
    }
}

constexpr int kMaxBanks = 64;
constexpr int kMaxSplits = 16;

struct BankPtrs {
    const uint32_t* w;
    const uint16_t* s;
    const uint16_t* b;
    void* out;
};

enum OutMode : int { kOutF32 = 0, kOutBF16 = 1, kOutPartial = 2 };

// Kernel parameters. CAP = number of bank slots carried (1 for a single
// projection, kMaxBanks for banked calls, 2 for the fused gate/up projection),
// so single calls pass a small block.
struct MainHeader {
    const uint16_t* x;      // activations [M][K] bfloat16, 16-byte aligned
    float* partial;         // [banks][splits][M][N] when out_mode == kOutPartial
    uint32_t* err;          // device error word
    int64_t N;
    int64_t K;
    int64_t rows_total;     // banks * splits * N (1 * splits * N for the fused projection)
    int G;                  // K / group
    int C;                  // chunks = ceil(G / 8)
    int splits;
    int cb[kMaxSplits + 1];   // first chunk of K slice s (s = 0..splits): s * C / splits
    int M;
    int out_mode;
    int sb_tma;             // scales/biases by TMA boxes (G % 8 == 0), else cp.async
    int banks;
    float* gate;            // [M][N] fp32 gate results of the current call (fused gate/up, unsliced)
    uint32_t unpack_magic;  // kF16x2_1024, given at run time so it stays in a register
};

template <int CAP>
struct MainParams {
    MainHeader h;
    BankPtrs bank[CAP];
    CUtensorMap tmw[CAP];   // packed codes: uint8 [N][row_bytes], box (block rows) x W, swizzled
    CUtensorMap tms[CAP];   // scales: uint16 [N][G], box (block rows) x 8 (when sb_tma)
    CUtensorMap tmb[CAP];   // biases: same
    CUtensorMap tmx;        // activations: bf16 [M][K/64][64] (x rows in 64-code blocks), box 64 x CK/64 x 8
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
// Work enumeration shared by every warp role. The flattened (bank, split, row)
// space is cut evenly, in whole 16-row slabs, over the CTAs; a CTA's range is
// cut at (bank, split) boundaries (segments) and then into row blocks of TN
// rows (the last one shorter); every row block walks the chunks of its K
// slice. One item = one chunk of one row block (for the fused gate/up
// projection, each row block is walked for bank 0 (gate) and then for bank 1
// (up)).
// ---------------------------------------------------------------------------

// One CTA's share of the flattened rows: whole 16-row slabs (the last one of
// the range possibly ragged), so the consumers compute few empty slab rows.
// Computed once per CTA; the iterators of every warp role start from it and
// then only step, with no division.
struct CtaRange {
    int64_t r, r_end;       // flattened rows [r, r_end)
    int seg;                // segment of row r: bank * splits + split
    int split, bank;        // seg % splits, seg / splits
};
__device__ __forceinline__ CtaRange cta_range(const MainHeader& p) {
    const int64_t slabs = (p.rows_total + kSlab - 1) / kSlab;
    CtaRange cr;
    cr.r = min(p.rows_total, kSlab * (slabs * blockIdx.x / gridDim.x));
    cr.r_end = min(p.rows_total, kSlab * (slabs * (blockIdx.x + 1) / gridDim.x));
    cr.seg = static_cast<int>(cr.r / p.N);
    cr.split = cr.seg % p.splits;
    cr.bank = cr.seg / p.splits;
    return cr;
}

template <bool SWIGLU, int TN>
struct WorkIter {
    int64_t r, r_end;       // flattened rows of this CTA still to start, end
    int64_t seg_end;
    int64_t a0, len;        // first flattened row and length of the segment part
    int seg;                // bank * splits + split of the current segment
    int sbank;              // its bank
    int nb, ib;             // row blocks of the part, current one
    int pass;               // fused gate/up: 0 = gate, 1 = up
    int bank, split, rows, c0, c1, c;
    int64_t n0;             // first weight row of the current row block
    bool valid;

    __device__ __forceinline__ void init(const MainHeader& p, const CtaRange& cr) {
        r = cr.r;
        r_end = cr.r_end;
        seg = cr.seg;
        split = cr.split;
        sbank = cr.bank;
        start_segment(p);
    }
    __device__ __forceinline__ void start_segment(const MainHeader& p) {
        valid = r < r_end;
        if (!valid) return;
        seg_end = min(r_end, static_cast<int64_t>(seg + 1) * p.N);
        a0 = r;
        len = seg_end - r;
        nb = static_cast<int>((len + TN - 1) / TN);
        ib = 0;
        pass = 0;
        c0 = p.cb[split];
        c1 = p.cb[split + 1];
        start_block(p);
    }
    __device__ __forceinline__ void start_block(const MainHeader& p) {
        const int64_t a = a0 + static_cast<int64_t>(TN) * ib;
        const int64_t e = min(a0 + len, a + TN);
        n0 = a - static_cast<int64_t>(seg) * p.N;
        rows = static_cast<int>(e - a);
        bank = SWIGLU ? pass : sbank;
        c = c0;
    }
    // k steps of next(): one add while they stay in the current row block (and pass)
    __device__ __forceinline__ void advance(const MainHeader& p, int k) {
        if (c + k < c1) {
            c += k;
            return;
        }
#pragma unroll 1
        for (int i = 0; i < k; ++i) next(p);
    }
    __device__ __forceinline__ bool block_start() const { return c == c0; }
    __device__ __forceinline__ bool block_end() const { return c == c1 - 1; }
    __device__ __forceinline__ void next(const MainHeader& p) {
        if (++c < c1) return;
        if (SWIGLU && pass == 0) {
            pass = 1;
            bank = 1;
            c = c0;
            return;
        }
        pass = 0;
        if (++ib < nb) {
            start_block(p);
            return;
        }
        // the next segment starts where this one ended (seg_end = (seg + 1) * N
        // unless the CTA's range ends first)
        r = seg_end;
        ++seg;
        if (++split == p.splits) {
            split = 0;
            ++sbank;
        }
        start_segment(p);
    }
};

// ---------------------------------------------------------------------------
// Small helpers.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t pack_half2(__half lo, __half hi) {
    return static_cast<uint32_t>(__half_as_ushort(lo)) | (static_cast<uint32_t>(__half_as_ushort(hi)) << 16);
}
__device__ __forceinline__ uint32_t f2_to_h2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}
// float from a power-of-two exponent (e in the normal range)
__device__ __forceinline__ float pow2f(int e) { return __uint_as_float(static_cast<uint32_t>(e + 127) << 23); }
// bfloat16 half h of a packed pair, as float
__device__ __forceinline__ float bf16_half(uint32_t w, int h) {
    return __uint_as_float(h ? (w & 0xFFFF0000u) : (w << 16));
}
constexpr uint32_t kF16One = 0x3C00u;
QMM_HD constexpr uint32_t f16_pow2_bits(int e) { return static_cast<uint32_t>(e + 15) << 10; }   // 2^e, -14 <= e <= 15

// Byte offset, inside a stage's weight tile, of byte b of tile row r (TMA box
// layout with the W-byte swizzle: bits 4.. of the in-box address are XORed
// with its bits 7..).
template <int BITS, int GROUP, int TN>
__device__ __forceinline__ int wtile_off(int r, int b) {
    constexpr int W = wbox_width(BITS, GROUP);
    constexpr int LW = log2i(W);
    constexpr int MASK = W / 16 - 1;
    const int lin = r * W + (b & (W - 1));
    return (b >> LW) * (W * TN) + (lin ^ (((lin >> 7) & MASK) << 4));   // box b / W holds TN rows
}

// ---------------------------------------------------------------------------
// The main kernel.
// ---------------------------------------------------------------------------
template <int BITS, int GROUP, int MB, int CAP, int LAY>
__global__ void __launch_bounds__(main_threads(MB, GROUP, LAY), 1) qmm_main_kernel(const __grid_constant__ MainParams<CAP> P) {
    constexpr int NT = n8_tiles(MB);
    constexpr int NSW = staging_warps(MB, GROUP, LAY);
    static_assert(MB == 8 || LAY != kWide, "the wide consumer layout is for the 8-row kernel");
    constexpr int NCW = consumer_warps();
    constexpr int CPAR = consumer_parities(LAY);
    constexpr int TN = consumer_rows(LAY);       // rows of a row block and of a weight stage
    constexpr int WPPC = NCW / CPAR;             // consumer warps of one parity
    constexpr int VB = vblocks_per_group(GROUP);
    constexpr int VPC = vblocks_per_chunk(GROUP);
    constexpr int CK = chunk_codes(GROUP);
    constexpr int BB = vblock_bytes(BITS);
    constexpr int RB = chunk_row_bytes(BITS, GROUP);
    constexpr int W = wbox_width(BITS, GROUP);
    constexpr int NBOX = wbox_count(BITS, GROUP);
    constexpr int SWB = stage_weight_bytes(BITS, GROUP, LAY);
    constexpr int SSB = stage_sb_bytes(LAY);
    constexpr int WSB = wstage_bytes(BITS, GROUP, LAY);          // weight stage
    constexpr int ASB = aslot_bytes(GROUP, MB);             // activation slot
    constexpr int XRB = xraw_bytes(GROUP, MB);
    constexpr int NBX = CK / 64;                    // 64-code blocks per chunk
    // weight stage: codes [NBOX][TN][W] swizzled, then
    constexpr int OFF_S = SWB;                      // scales [TN][8] binary16
    constexpr int OFF_B = OFF_S + SSB;              // biases [TN][8] binary16
    // activation slot:
    constexpr int XRT = XRB / NT;                   // raw x of one 8-row tile
    constexpr int OFF_XR = 0;                       // raw x [NT][8][NBX][128 B], 128-byte swizzle
    constexpr int OFF_XF = XRB;                     // B fragments [VPC][NT][32] x 16 B
    constexpr int OFF_XB = OFF_XF + xfrag_bytes(GROUP, MB);   // bias fragments [NT][32] x 16 B
    constexpr int OFF_XT = OFF_XB + xbias_bytes(MB);          // sigma[MB], 1/f[MB]
    constexpr bool SWIGLU = CAP == 2;
    static_assert(W * NBOX == RB, "weight boxes");
    static_assert(XRT % 1024 == 0 && OFF_XT + 8 * MB <= ASB && OFF_B + SSB <= WSB, "stage layout");
    const MainHeader& p = P.h;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte aligned ring base, derived by pointer arithmetic on the shared
    // array so every access below stays a shared-memory access
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    constexpr int S = stage_count(BITS, GROUP, MB, LAY);     // weight stages
    constexpr int F = act_slots(BITS, GROUP, MB, LAY);       // activation slots
    static_assert(S >= 2 && F >= 2 && S % CPAR == 0 && F % CPAR == 0, "pipeline depth");
    uint8_t* aring = smem + S * WSB;                                        // activation slots
    uint64_t* wfull = reinterpret_cast<uint64_t*>(aring + F * ASB);        // weights, scales, biases landed
    uint64_t* wempty = wfull + S;                                          // weight stage consumed
    uint64_t* xfull = wempty + S;                                          // raw activations landed [F][NT]
    uint64_t* sfull = xfull + F * NT;                                      // fragments staged
    uint64_t* fempty = sfull + F;                                          // activation slot consumed
    float* combine = reinterpret_cast<float*>(fempty + F);                 // [kSlabs][NT][4][32]
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    CtaRange& s_range = *reinterpret_cast<CtaRange*>(reinterpret_cast<uint8_t*>(combine) + combine_bytes(MB, LAY));
    // first activation copies issued (the producer of the wide layout with a full
    // ring of small weight stages waits for them)
    constexpr bool XFIRST = LAY == kWide && S >= kMaxStages;
    uint64_t* const xissued =
        reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(combine) + combine_bytes(MB, LAY) + kRangeBytes);
    static_assert(sizeof(CtaRange) <= kRangeBytes && alignof(CtaRange) <= 8, "work range area");

    if (threadIdx.x == 0) {
        s_range = cta_range(p);
        for (int i = 0; i < S; ++i) {
            // producer lane 0 (expect_tx), plus 32 cp.async arrivals when the
            // scales and biases come by cp.async
            mbar_init(&wfull[i], p.sb_tma ? 1 : 1 + 32);
            mbar_init(&wempty[i], WPPC);          // one lane of each of the stage parity's consumer warps
        }
        for (int i = 0; i < F * NT; ++i)
            mbar_init(&xfull[i], 1);              // the owning staging warp's lane 0 (expect_tx), per tile
        for (int i = 0; i < F; ++i) {
            mbar_init(&sfull[i], NT);             // one lane of the owning staging warp of each tile
            mbar_init(&fempty[i], WPPC);          // one lane of each of the slot parity's consumer warps
        }
        // lane 0 of each staging warp that owns slots, once its first copies are issued
        if constexpr (XFIRST)
            mbar_init(xissued, (F <= staging_per_tile(MB, GROUP, LAY) ? F : staging_per_tile(MB, GROUP, LAY)) * NT);
        fence_barrier_init();
    }
    __syncthreads();
    // The next kernel on the stream may be scheduled now; its CTAs take the SMs
    // this grid's CTAs free and start streaming their own weights at once.
    griddep_launch_dependents();

    if (warp == NCW + NSW) {
        // ------------------------------ producer ------------------------------
        // Lane 0 issues the TMA boxes of a stage (packed codes, scales, biases).
        // Scales and biases whose rows are not 16-byte multiples go through
        // per-lane cp.async instead. The weights do not depend on the preceding
        // work on the stream, so this warp never waits for it.
        const uint64_t pol = policy_evict_first();
        if (lane == 0) {
            prefetch_tensormap(&P.tmx);
            for (int i = 0; i < p.banks && i < CAP; ++i) {
                prefetch_tensormap(&P.tmw[i]);
                if (p.sb_tma) {
                    prefetch_tensormap(&P.tms[i]);
                    prefetch_tensormap(&P.tmb[i]);
                }
            }
        }
        const uint32_t tx_stage = static_cast<uint32_t>(NBOX * TN * W + (p.sb_tma ? 2 * SSB : 0));
        WorkIter<SWIGLU, TN> wi;
        wi.init(p, s_range);
        uint32_t it = 0;
        int slot = 0;             // it % S, kept incrementally
        uint32_t round = 0;       // it / S
        bool ok = true;
        bool sb_ok = true;
        for (; wi.valid; wi.next(p)) {
            const BankPtrs bp = P.bank[wi.bank];
            if (wi.block_start()) {
                // the cp.async path for scales/biases checks its buffers once per row block
                sb_ok = p.sb_tma ||
                    (wi.n0 >= 0 && wi.rows >= 1 && wi.rows <= TN && wi.n0 + wi.rows <= p.N && wi.c0 >= 0 &&
                     wi.c1 <= p.C && ((reinterpret_cast<uintptr_t>(bp.s) | reinterpret_cast<uintptr_t>(bp.b)) & 3) == 0);
                if (!sb_ok && lane == 0) record_bad_copy(p.err, bp.s, static_cast<uint64_t>(wi.rows), 4u);
                // a row block longer than the layout covers would leave rows
                // unwritten (the row blocks are cut to TN rows, so this never fires)
                if (wi.rows > TN && lane == 0)
                    record_bad_copy(p.err, bp.w, static_cast<uint64_t>(wi.rows), 6u);
            }
            // After a timed-out wait the error is recorded and no further waits are
            // made; the loop still runs to the end so that every warp finishes.
            // In the wide layout with a full ring of small stages the producer,
            // after the first stages, waits until the staging warps have issued
            // their first activation copies (they do so once the preceding work
            // has finished): those copies then queue ahead of the rest of the
            // weight stream in the copy engine, and the first items are staged
            // sooner (1-2 % faster calls on 5120 x 17408; the other layouts and
            // rings of four large stages measured slower with the wait).
            if (XFIRST && it == static_cast<uint32_t>(kStagesBeforeX) && ok &&
                !mbar_wait(xissued, 0u, p.err, kErrEmptyWait))
                ok = false;
            // (The slot's previous use was in round `round - 1`: parity round ^ 1.)
            if (it >= static_cast<uint32_t>(S) && ok &&
                !mbar_wait_sleep(&wempty[slot], (round ^ 1u) & 1u, p.err, kErrEmptyWait, 128u))
                ok = false;
            uint8_t* st = smem + slot * WSB;
            if (lane == 0) {
                mbar_arrive_expect_tx(&wfull[slot], tx_stage);
                const int y = static_cast<int>(wi.n0);
#pragma unroll
                for (int bi = 0; bi < NBOX; ++bi)
                    tma_load_2d(st + bi * (TN * W), &P.tmw[wi.bank], wi.c * RB + bi * W, y, &wfull[slot], pol);
                if (p.sb_tma) {
                    tma_load_2d(st + OFF_S, &P.tms[wi.bank], wi.c * kGPC, y, &wfull[slot], pol);
                    tma_load_2d(st + OFF_B, &P.tmb[wi.bank], wi.c * kGPC, y, &wfull[slot], pol);
                }
            }
            __syncwarp();
            if (!p.sb_tma && sb_ok) {
                const int ng = min(kGPC, p.G - wi.c * kGPC);
                const int nq = ng >> 1;   // 4-byte pieces per row
                uint8_t* sdst = st + OFF_S;
                uint8_t* bdst = st + OFF_B;
                const uint16_t* ssrc = bp.s + wi.n0 * p.G + wi.c * kGPC;
                const uint16_t* bsrc = bp.b + wi.n0 * p.G + wi.c * kGPC;
                for (int i = lane; i < wi.rows * nq; i += 32) {
                    const int rr = i / nq, q = i - (i / nq) * nq;
                    cp_async_4(sdst + rr * 16 + 4 * q, ssrc + static_cast<int64_t>(rr) * p.G + 2 * q);
                    cp_async_4(bdst + rr * 16 + 4 * q, bsrc + static_cast<int64_t>(rr) * p.G + 2 * q);
                }
            }
            if (!p.sb_tma) cp_async_arrive_noinc(&wfull[slot]);
            ++it;
            if (++slot == S) {
                slot = 0;
                ++round;
            }
        }
        // This warp's own cp.async copies must land before it exits.
        cp_async_wait_all();
        if (!ok) {
            // Give the copies already issued a bounded chance to land before exiting.
            const uint32_t first = it > static_cast<uint32_t>(S) ? it - S : 0u;
            for (uint32_t i = first; i < it; ++i)
                if (!mbar_drain(&wfull[i % S], (i / S) & 1u, p.err)) break;
        }
        return;
    }

    const int g = lane >> 2;
    const int t = lane & 3;

    if (warp >= NCW) {
        // ------------------------------ staging -------------------------------
        // Warp (j, par) stages activation tile j (rows 8j .. 8j + 7) of the
        // stages in its slots, the whole chunk: lane (g, t) handles row
        // m = 8j + g and, in each k32 block, the 8 codes it holds in the
        // consumers' fragments. Everything it needs across lanes (the row's
        // largest |x| and the bias-term range) reduces inside the quad.
        constexpr int SPT = staging_per_tile(MB, GROUP, LAY);
        const int sw = warp - NCW;
        const int j = sw / SPT;
        const int par = sw % SPT;
        const int m = 8 * j + g;
        // Selector of the XS MMA: column n = g of B belongs to group q = g >> 1
        // of a half chunk, XS (even n, weight 2^j per k slot) or XSc/1024 (odd
        // n, weight 1). k slots 2t + e and 2t + 8 + e of MMA u are the slots
        // (r = 2u, e) and (r = 2u + 1, e) of the unpackers. selq[q] is the
        // selector for group q of the half (zero in the other groups' columns).
        uint32_t selq[4][2][2];
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int u = 0; u < 2; ++u)
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                    const int rr = 2 * u + kk;
                    const uint32_t xs =
                        f16_pow2_bits(slot_shift(BITS, rr, 0)) | (f16_pow2_bits(slot_shift(BITS, rr, 1)) << 16);
                    selq[q][u][kk] = (g >> 1) != q ? 0u : ((g & 1) ? (kF16One | (kF16One << 16)) : xs);
                }
        constexpr int HPC = VPC / 2;                  // k32 blocks per half chunk (groups 0-3 / 4-7)
        // with groups of 32 the raw values of a chunk stay in registers between
        // the two passes; with groups of 64 they are read from shared memory twice
        constexpr bool KEEP = VPC <= 8;

        // Warp par of the tile owns the activation slots f with f % SPT == par:
        // it issues its tile's raw-activation copies (one 3-D TMA box of x per
        // chunk: the tile's 8 rows, refilled with the chunk F items ahead as soon
        // as the staging has read it) and writes its tile's fragments. Every phase of a slot's barriers is
        // therefore awaited, in order, by the one warp that owns the slot (a
        // parity wait may only run one phase ahead of its barrier). x is read
        // only after the preceding work on the stream (which may have produced
        // it) has finished.
        // bytes of one tile copy: the 8-row kernel copies only the call's M rows when
        // M < 8 (rows M..7 of its raw area keep stale values; their fragments, sums
        // and MMA columns are their own and are never stored)
        const uint32_t xtile_bytes = static_cast<uint32_t>((MB == 8 ? min(p.M, 8) : 8) * NBX * 128);
        auto issue_raw = [&](int f, int c) {
            uint64_t* bar = &xfull[f * NT + j];
            if (c < 0 || c >= p.C) {
                record_bad_copy(p.err, p.x, static_cast<uint64_t>(f) << 32 | static_cast<uint32_t>(c), 5u);
                mbar_arrive(bar);   // complete the phase without data
                return;
            }
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(bar, xtile_bytes);
            tma_load_3d(aring + f * ASB + OFF_XR + j * XRT, &P.tmx, 0, c * NBX, 8 * j, bar);
        };
        griddep_wait();
        // The items of this warp's slots are the items it with it % STRIDE == par;
        // it walks them only (warps with par >= STRIDE own no slot).
        constexpr int STRIDE = F <= SPT ? F : SPT;
        static_assert(F <= SPT || F % SPT == 0, "activation slot ownership");
        if (par >= STRIDE) return;
        WorkIter<SWIGLU, TN> lead;   // the item F ahead of the current one
        lead.init(p, s_range);
        uint32_t issued = 0;     // one past the last item whose raw copy this warp issued
        for (int i = 0; i < F && lead.valid; ++i, lead.next(p))
            if (i % STRIDE == par) {
                if (lane == 0) issue_raw(i, lead.c);
                issued = static_cast<uint32_t>(i) + 1u;
            }
        if (XFIRST && lane == 0) mbar_arrive(xissued);

        // After a timed-out wait no further copies are issued; the ones in
        // flight (this warp's items failed .. issued - 1) are drained before the
        // warp exits.
        bool ok = true;
        uint32_t failed = 0;
        WorkIter<SWIGLU, TN> wi;
        wi.init(p, s_range);
        // (the 8-row kernel steps with one add inside a row block; the 16-row
        // kernel, whose staging warps own every other item, measured faster
        // stepping one item at a time)
        if constexpr (MB == 8) {
            wi.advance(p, par);
            lead.advance(p, par);
        } else {
#pragma unroll 1
            for (int k = 0; k < par; ++k) {
                wi.next(p);
                lead.next(p);
            }
        }
        uint32_t it = static_cast<uint32_t>(par);
        for (; wi.valid; it += STRIDE) {
            const int slot = static_cast<int>(it % static_cast<uint32_t>(F));
            const uint32_t phase = (it / static_cast<uint32_t>(F)) & 1u;
            if (ok && !mbar_wait(&xfull[slot * NT + j], phase, p.err, kErrFullWait)) {
                ok = false;
                failed = it;
            }
            uint8_t* st = aring + slot * ASB;
            // refill the slot with the raw activations of the item F ahead (issued
            // after the item is staged: a copy issued while the weight stages fill
            // the copy engine can hold the warp, and the item F ahead is needed
            // only F items later)
            auto refill = [&]() {
                __syncwarp();
                if (ok && lead.valid) {
                    if (lane == 0) issue_raw(slot, lead.c);
                    issued = it + static_cast<uint32_t>(F) + 1u;
                }
            };
            // Tile row g, 64-code block b: 128 bytes at u = g * NBX + b (times 128)
            // of the tile's raw area, with 16-byte piece c stored at piece c ^ (u & 7).
            // Codes past K (and, in the 16-row kernel, rows >= M) arrive from the TMA
            // as zeros.
            auto load_raw = [&](int vb, uint32_t (&v)[4]) {
                const int u = g * NBX + (vb >> 1);
                const uint8_t* rb = st + OFF_XR + j * XRT + u * 128;
                const int key = u & 7;
                if constexpr (BITS == 8) {
                    // codes 4t .. 4t + 3 and 16 + 4t .. 16 + 4t + 3 of the k32 block
                    const int c0 = (vb & 1) * 4 + (t >> 1), c1 = c0 + 2;
                    const uint2 a0 = *reinterpret_cast<const uint2*>(rb + ((c0 ^ key) << 4) + (t & 1) * 8);
                    const uint2 a1 = *reinterpret_cast<const uint2*>(rb + ((c1 ^ key) << 4) + (t & 1) * 8);
                    v[0] = a0.x;
                    v[1] = a0.y;
                    v[2] = a1.x;
                    v[3] = a1.y;
                } else {
                    // codes 8t .. 8t + 7 of the k32 block
                    const uint4 a = *reinterpret_cast<const uint4*>(rb + ((((vb & 1) * 4 + t) ^ key) << 4));
                    v[0] = a.x;
                    v[1] = a.y;
                    v[2] = a.z;
                    v[3] = a.w;
                }
            };
            uint32_t keep[KEEP ? VPC : 1][4];
            // pass 1: largest |x| of row m over the chunk (the lane's codes as a
            // tree, then the quad)
            uint32_t bm[VPC];
#pragma unroll
            for (int vb = 0; vb < VPC; ++vb) {
                uint32_t v[4];
                load_raw(vb, v);
                bm[vb] = bf16x2_absmax(bf16x2_absmax(v[0], v[1]), bf16x2_absmax(v[2], v[3]));
                if constexpr (KEEP) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) keep[vb][e] = v[e];
                }
            }
#pragma unroll
            for (int w2 = VPC / 2; w2 >= 1; w2 /= 2)
#pragma unroll
                for (int i = 0; i < w2; ++i) bm[i] = bf16x2_absmax(bm[i], bm[i + w2]);
            // the fragment area must be free: the consumers are done with the item F before
            if (it >= static_cast<uint32_t>(F))
                mbar_wait_sleep(&fempty[slot], phase ^ 1u, p.err, kErrEmptyWait, 128u);
            const uint32_t mx = bm[0];
            uint32_t mag = max(mx & 0x7FFFu, (mx >> 16) & 0x7FFFu);
            mag = max(mag, __shfl_xor_sync(0xFFFFFFFFu, mag, 1));
            mag = max(mag, __shfl_xor_sync(0xFFFFFFFFu, mag, 2));
            // f puts the chunk's largest |x| of the row in [2^14, 2^15): every
            // f*x*2^-j is below 2^15, and any x within 2^27 of the largest is exact
            int ex = 0;
            if (mag != 0) ex = min(127, max(-100, static_cast<int>(mag >> 7) - 127));
            const float f = pow2f(14 - ex);
            const float rf = pow2f(ex - 14);
            float fs[4][2];
#pragma unroll
            for (int rr = 0; rr < 4; ++rr)
#pragma unroll
                for (int e = 0; e < 2; ++e) fs[rr][e] = f * pow2f(-slot_shift(BITS, rr, e));

            // pass 2: fragments, and f*XS, f*XSc/1024 per group through the selector MMA
            // (accumulator 2h + (vb & 1): half h of the chunk, even/odd blocks)
            float D[4][4];
#pragma unroll
            for (int a = 0; a < 4; ++a) D[a][0] = D[a][1] = D[a][2] = D[a][3] = 0.0f;
#pragma unroll
            for (int vb = 0; vb < VPC; ++vb) {
                uint32_t v[4];
                if constexpr (KEEP) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) v[e] = keep[vb][e];
                } else {
                    load_raw(vb, v);
                }
                uint32_t fr[4];
#pragma unroll
                for (int rr = 0; rr < 4; ++rr) {
                    float v2[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        int wi4, hf;
                        if constexpr (BITS == 8) {
                            // piece rr >> 1, word e, half rr & 1
                            wi4 = 2 * (rr >> 1) + e;
                            hf = rr & 1;
                        } else {
                            const int cc = slot_code(BITS, rr, e);
                            wi4 = cc >> 1;
                            hf = cc & 1;
                        }
                        v2[e] = bf16_half(v[wi4], hf);
                    }
                    // (f * 2^-j, exact: one paired multiply for the two codes)
                    mul_x2(v2[0], v2[1], v2[0], v2[1], fs[rr][0], fs[rr][1]);
                    fr[rr] = f2_to_h2(v2[0], v2[1]);
                }
                *reinterpret_cast<uint4*>(st + OFF_XF + ((vb * NT + j) * 32 + lane) * 16) =
                    make_uint4(fr[0], fr[1], fr[2], fr[3]);
                const int hv = vb / HPC;                      // half chunk
                const int q = (vb % HPC) / VB;                // group within the half
                float (&Da)[4] = D[2 * hv + (vb & 1)];
                mma_f16(Da, fr[0], 0u, fr[1], 0u, selq[q][0][0], selq[q][0][1]);
                mma_f16(Da, fr[2], 0u, fr[3], 0u, selq[q][1][0], selq[q][1][1]);
            }
            // lane (g, t): groups t (half 0) and 4 + t (half 1) of row m
            const float xs0 = (D[0][0] + D[1][0]) * rf, xsc0 = (D[0][1] + D[1][1]) * (rf * 1024.0f);
            const float xs1 = (D[2][0] + D[3][0]) * rf, xsc1 = (D[2][1] + D[3][1]) * (rf * 1024.0f);
            float am = fmaxf(fmaxf(fabsf(xs0), fabsf(xsc0)), fmaxf(fabsf(xs1), fabsf(xsc1)));
            am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, 1));
            am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, 2));
            // sigma puts the largest |XS/sigma|, |XSc/sigma| of the row in [2^13, 2^14)
            int es = 13;
            if (am > 0.0f && am <= 3.0e38f) es = max(-100, static_cast<int>((__float_as_uint(am) >> 23) & 0xFFu) - 127);
            const float rsig = pow2f(13 - es);    // 1 / sigma
            const float sg = pow2f(es - 13);
            uint32_t hi[2], lo[2];
            {
                const float vv[2] = {xs0 * rsig, xs1 * rsig};
                const float ww[2] = {-xsc0 * rsig, -xsc1 * rsig};
#pragma unroll
                for (int hv = 0; hv < 2; ++hv) {
                    const __half vh = __float2half_rn(vv[hv]), wh = __float2half_rn(ww[hv]);
                    const __half vl = __float2half_rn(vv[hv] - __half2float(vh));
                    const __half wl = __float2half_rn(ww[hv] - __half2float(wh));
                    hi[hv] = pack_half2(vh, wh);
                    lo[hv] = pack_half2(vl, wl);
                }
            }
            // groups 4hv + t and 4hv + t + 1 form the bias fragment of lane (g, 2hv + t / 2),
            // stored by the lanes with even t (with groups of 64 both halves' fragments
            // behind one branch: 1.5-2.5 % faster calls than a branch per half, which
            // measured 1 % faster with groups of 32)
            auto bias_frag = [&](int hv) {
                const uint32_t hi_p = __shfl_xor_sync(0xFFFFFFFFu, hi[hv], 1);
                const uint32_t lo_p = __shfl_xor_sync(0xFFFFFFFFu, lo[hv], 1);
                return make_uint4((hi[hv] & 0xFFFFu) | (hi_p << 16), (hi[hv] >> 16) | (hi_p & 0xFFFF0000u),
                                  (lo[hv] & 0xFFFFu) | (lo_p << 16), (lo[hv] >> 16) | (lo_p & 0xFFFF0000u));
            };
            auto xb_at = [&](int hv) {
                return reinterpret_cast<uint4*>(st + OFF_XB + (j * 32 + g * 4 + 2 * hv + (t >> 1)) * 16);
            };
            if constexpr (VB > 1) {
                const uint4 b0 = bias_frag(0), b1 = bias_frag(1);
                if ((t & 1) == 0) {
                    *xb_at(0) = b0;
                    *xb_at(1) = b1;
                }
            } else {
#pragma unroll
                for (int hv = 0; hv < 2; ++hv) {
                    const uint4 b = bias_frag(hv);
                    if ((t & 1) == 0) *xb_at(hv) = b;
                }
            }
            if (t == 0) {
                float* xt = reinterpret_cast<float*>(st + OFF_XT);
                xt[m] = sg;
                xt[MB + m] = rf;
            }
            // the warp's fragment stores, ordered by the warp barrier before one lane's release
            __syncwarp();
            if (lane == 0) mbar_arrive(&sfull[slot]);
            refill();
            if constexpr (MB == 8) {
                wi.advance(p, STRIDE);
                lead.advance(p, STRIDE);
            } else {
#pragma unroll 1
                for (int k = 0; k < STRIDE; ++k) {
                    wi.next(p);
                    lead.next(p);
                }
            }
        }
        if (!ok && lane == 0) {
            for (uint32_t i = failed; i < issued; i += STRIDE) {
                const int f = static_cast<int>(i % static_cast<uint32_t>(F));
                if (!mbar_drain(&xfull[f * NT + j], (i / static_cast<uint32_t>(F)) & 1u, p.err)) break;
            }
        }
        __syncwarp();
        return;
    }

    // -------------------------------- consumers --------------------------------
    // Warp (w, cp) owns the SPW 16-row slabs SPW*w .. SPW*w + SPW - 1 of every
    // row block (slab z: tile rows 16z + g and 16z + g + 8), every group of the
    // chunks in the stage slots of parity cp (all slots when CPAR == 1). The
    // slabs of a warp share its activation fragment loads and give it SPW
    // independent MMA chains.
    constexpr int SPW = consumer_slabs(LAY);
    constexpr int WPP = NCW / CPAR;              // consumer warps per parity
    const int w = warp % WPP;
    const int cp = warp / WPP;
    const int r0 = kSlab * SPW * w + g;          // first slab's row; slab s: r0 + 16 s
    const uint32_t magic = p.unpack_magic;
    const uint32_t sel2 = unpack2_selector(t);   // 2-bit codes only
    const uint32_t ring = smem_u32(smem);
    // Per-lane code addresses of the first slab inside a stage (4- and 8-bit:
    // ldmatrix row addresses; 2-bit: 16-byte chunks of row r0; 3/5/6-bit: the
    // two words of each block of row r0). Row r0 + 8 has the same swizzle,
    // 8 * W further; the slab s rows, 16 * s * W further.
    constexpr int NOFF = BITS == 4 ? (VPC / 2 < 4 ? VPC / 2 : 4)
                       : BITS == 8 ? 4
                       : BITS == 2 ? RB / 16
                       : 2 * VPC;
    int off[NOFF];
    {
        const int lr = kSlab * SPW * w + ((lane >> 3) & 1) * 8 + (lane & 7);   // ldmatrix row of this lane
#pragma unroll
        for (int i = 0; i < NOFF; ++i) {
            if constexpr (BITS == 4) {
                const int b = 2 * i + (lane >> 4);                       // k32 block = 16-byte chunk
                off[i] = lr * 128 + (((b & 7) ^ (lane & 7)) << 4);
            } else if constexpr (BITS == 8) {
                const int k = 2 * i + (lane >> 4);                       // 16-byte chunk (half block)
                off[i] = lr * 128 + (((k & 7) ^ (lane & 7)) << 4);
            } else if constexpr (BITS == 2) {
                off[i] = wtile_off<BITS, GROUP, TN>(r0, 16 * i);
            } else {
                const int vb = i >> 1;
                const int b = vb * BB + 4 * ((BITS * t) >> 2) + 4 * (i & 1);
                // 3-bit lane 3 needs no second word: read its first word again
                const int bb = (BITS == 3 && t == 3 && (i & 1)) ? b - 4 : b;
                off[i] = wtile_off<BITS, GROUP, TN>(r0, bb);
            }
        }
    }
    const uint32_t oddsh = static_cast<uint32_t>(((BITS * t) & 3) * 8);

    int cslot = 0;            // item % S (weight stage), kept incrementally
    uint32_t cphase = 0;      // (item / S) & 1
    int aslot = 0;            // item % F (activation slot)
    uint32_t aphase = 0;      // (item / F) & 1
    // Each output sums its block's items in two halves, the items of even and of
    // odd index (the two consumer parities when there are two; otherwise one
    // warp keeps both sums), added at the end of the block: so row m of an
    // output is bitwise the same whether the 8- or the 16-row kernel made it.
    constexpr int NACC = CPAR == 1 ? 2 : 1;
    // With the 16-row tile (two activation slots) and in the pair layout a warp
    // releases the activation slot with its last block's fragment loads and the
    // stage once it has loaded the bias-term operands, before the last group's
    // and the bias term's arithmetic, so the slot is restaged sooner (16-row calls
    // 2-3.5 % faster, pr1_ref 1 %); with the 8-row tile's narrow and wide layouts
    // the early stage release measured up to 1.7 % slower.
    // (Not the fused gate/up kernel: there the early order spills and its 16-row
    // calls measured 3 % slower.)
    constexpr bool EARLY_RELEASE = (MB == 16 && !SWIGLU) || LAY == kPair;
    float acc[NACC][SPW][NT][4];
    uint32_t ipar = 0;        // item & 1
    WorkIter<SWIGLU, TN> wi;
    wi.init(p, s_range);
    for (; wi.valid; wi.next(p), ipar ^= 1u) {
        if (wi.block_start()) {
#pragma unroll
            for (int a = 0; a < NACC; ++a)
#pragma unroll
                for (int sl = 0; sl < SPW; ++sl)
#pragma unroll
                    for (int jj = 0; jj < NT; ++jj)
#pragma unroll
                        for (int e = 0; e < 4; ++e) acc[a][sl][jj][e] = 0.0f;
        }
        // (a warp whose first slab holds rows of the block computes all of its
        // slabs; rows past the block are not stored)
        const bool active = w * SPW * kSlab < wi.rows;
        const int slot = cslot;
        const int fslot = aslot;
        // (S and F are multiples of CPAR, so both slots have the item's parity)
        const bool mine = CPAR == 1 || slot % CPAR == cp;
        // a timed-out wait is recorded; the warp then stops waiting but keeps the
        // same control flow
        bool released = false;    // (the early release below)
        if (mine) {
        {
            // both first tests before either branch: their latencies overlap
            // (0.5-1.4 % faster calls than one wait after the other)
            const bool wready = mbar_try_wait(&wfull[slot], cphase);
            const bool sready = mbar_try_wait(&sfull[fslot], aphase);
            if (!wready) mbar_wait_slow(&wfull[slot], cphase, p.err, kErrFullWait);
            if (!sready) mbar_wait_slow(&sfull[fslot], aphase, p.err, kErrFullWait);
        }
        if (active) {
            const uint32_t st = ring + static_cast<uint32_t>(slot * WSB);
            const uint32_t at = ring + static_cast<uint32_t>(S * WSB + fslot * ASB);
            const uint32_t b_r0 = st + static_cast<uint32_t>(r0 * 16);   // rows r0 (+128: r0 + 8) of scales, biases
            const uint32_t b_l = at + static_cast<uint32_t>(lane * 16);  // this lane's fragment vectors
            const uint32_t b_t = at + static_cast<uint32_t>(t * 8);      // activation rows 2t, 2t + 1 of the factors
            const int ng = min(kGPC, p.G - wi.c * kGPC);
            // this lane's scales of rows r0 + 16 s and r0 + 16 s + 8 (8 binary16 values each)
            uint32_t s0w[SPW][4], s1w[SPW][4];
            static_for<0, SPW>([&](auto s_c) {
                constexpr int sl = decltype(s_c)::value;
                const uint4 sv0 = lds128_at<OFF_S + 256 * sl>(b_r0);
                const uint4 sv1 = lds128_at<OFF_S + 256 * sl + 128>(b_r0);
                s0w[sl][0] = sv0.x; s0w[sl][1] = sv0.y; s0w[sl][2] = sv0.z; s0w[sl][3] = sv0.w;
                s1w[sl][0] = sv1.x; s1w[sl][1] = sv1.y; s1w[sl][2] = sv1.z; s1w[sl][3] = sv1.w;
            });
            if (ng < kGPC) {
                // groups past the end of K (stale shared memory on the cp.async path):
                // zero their scales so they contribute nothing
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t keep = (2 * i + 1 < ng) ? 0xFFFFFFFFu : (2 * i < ng ? 0x0000FFFFu : 0u);
#pragma unroll
                    for (int sl = 0; sl < SPW; ++sl) {
                        s0w[sl][i] &= keep;
                        s1w[sl][i] &= keep;
                    }
                }
            }
            // code addresses of this chunk (4/8-bit: ldmatrix rows; 2-bit: row r0's 16-byte chunks)
            uint32_t cb[(BITS == 4 || BITS == 8 || BITS == 2) ? NOFF : 1];
            if constexpr (BITS == 4 || BITS == 8 || BITS == 2) {
#pragma unroll
                for (int i = 0; i < NOFF; ++i) cb[i] = st + static_cast<uint32_t>(off[i]);
            }
            float accc[SPW][NT][4];
            uint2 rfa[NT], sga[NT];   // bias-term operands from the slot (early release)
            uint4 bba[NT];
            uint32_t q4[SPW][4];     // 4-bit: ldmatrix words of the current pair of blocks
            uint4 q2a[SPW], q2b[SPW];   // 2-bit: the 16-byte chunk (two blocks) of rows r0, r0 + 8
            static_for<0, kGPC>([&](auto gq_c) {
                constexpr int gq = decltype(gq_c)::value;
                // the group's products. Groups of 32 (one k32 block): two independent
                // MMAs a slab, one per k16 half, added when the group is done. Groups
                // of 64: one chain of four MMAs a slab (measured faster there).
                constexpr bool ONECHAIN = VB > 1;
                float Pg[SPW][NT][2][4];
                static_for<0, VB>([&](auto v_c) {
                    constexpr int v = decltype(v_c)::value;
                    constexpr int vb = gq * VB + v;              // k32 block within the chunk
                    uint4 bf[NT];
                    static_for<0, NT>([&](auto j_c) {
                        constexpr int jj = decltype(j_c)::value;
                        bf[jj] = lds128_at<OFF_XF + (vb * NT + jj) * 512>(b_l);
                    });
                    if constexpr (EARLY_RELEASE && vb == VPC - 1) {
                        // the slot's last reads (the bias-term operands with the last
                        // block's fragments): one lane releases it after the warp barrier
                        static_for<0, NT>([&](auto j_c) {
                            constexpr int jj = decltype(j_c)::value;
                            rfa[jj] = lds64_at<OFF_XT + 4 * (MB + 8 * jj)>(b_t);
                            sga[jj] = lds64_at<OFF_XT + 4 * (8 * jj)>(b_t);
                            bba[jj] = lds128_at<OFF_XB + jj * 512>(b_l);
                        });
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&fempty[fslot]);
                    }
                    static_for<0, SPW>([&](auto s_c) {
                        constexpr int sl = decltype(s_c)::value;
                        constexpr int SO = sl * kSlab * W;       // slab offset inside a weight box
                        uint32_t ra[4], rb[4];
                        if constexpr (BITS == 4) {
                            // one ldmatrix per pair of blocks (rows r0 and r0 + 8 of both)
                            if constexpr ((vb & 1) == 0)
                                ldmatrix_x4_at<(vb >> 3) * (TN * 128) + SO>(cb[(vb >> 1) & 3], q4[sl][0], q4[sl][1],
                                                                             q4[sl][2], q4[sl][3]);
                            unpack4((vb & 1) ? q4[sl][2] : q4[sl][0], ra, magic);
                            unpack4((vb & 1) ? q4[sl][3] : q4[sl][1], rb, magic);
                        } else if constexpr (BITS == 8) {
                            uint32_t d0, d1, d2, d3;
                            ldmatrix_x4_at<(vb >> 2) * (TN * 128) + SO>(cb[vb & 3], d0, d1, d2, d3);
                            unpack8(d0, d2, ra, magic);
                            unpack8(d1, d3, rb, magic);
                        } else if constexpr (BITS == 2) {
                            if constexpr ((vb & 1) == 0) {
                                q2a[sl] = lds128_at<SO>(cb[vb >> 1]);
                                q2b[sl] = lds128_at<SO + 8 * W>(cb[vb >> 1]);
                            }
                            const uint32_t wa = (vb & 1) ? ((t >> 1) ? q2a[sl].w : q2a[sl].z)
                                                         : ((t >> 1) ? q2a[sl].y : q2a[sl].x);
                            const uint32_t wb = (vb & 1) ? ((t >> 1) ? q2b[sl].w : q2b[sl].z)
                                                         : ((t >> 1) ? q2b[sl].y : q2b[sl].x);
                            unpack2(wa, sel2, ra, magic);
                            unpack2(wb, sel2, rb, magic);
                        } else {
                            const uint32_t lo = st + static_cast<uint32_t>(off[2 * vb]);
                            const uint32_t hi = st + static_cast<uint32_t>(off[2 * vb + 1]);
                            const uint32_t lo0 = lds32_at<SO>(lo);
                            const uint32_t hi0 = lds32_at<SO>(hi);
                            const uint32_t lo1 = lds32_at<SO + 8 * W>(lo);
                            const uint32_t hi1 = lds32_at<SO + 8 * W>(hi);
                            unpack_odd<BITS>(lo0, hi0, oddsh, ra, magic);
                            unpack_odd<BITS>(lo1, hi1, oddsh, rb, magic);
                        }
                        static_for<0, NT>([&](auto j_c) {
                            constexpr int jj = decltype(j_c)::value;
                            if constexpr (ONECHAIN) {
                                if constexpr (v == 0)
                                    mma_f16_zc(Pg[sl][jj][0], ra[0], rb[0], ra[1], rb[1], bf[jj].x, bf[jj].y);
                                else
                                    mma_f16(Pg[sl][jj][0], ra[0], rb[0], ra[1], rb[1], bf[jj].x, bf[jj].y);
                                mma_f16(Pg[sl][jj][0], ra[2], rb[2], ra[3], rb[3], bf[jj].z, bf[jj].w);
                            } else if constexpr (v == 0) {
                                mma_f16_zc(Pg[sl][jj][0], ra[0], rb[0], ra[1], rb[1], bf[jj].x, bf[jj].y);
                                mma_f16_zc(Pg[sl][jj][1], ra[2], rb[2], ra[3], rb[3], bf[jj].z, bf[jj].w);
                            } else {
                                mma_f16(Pg[sl][jj][0], ra[0], rb[0], ra[1], rb[1], bf[jj].x, bf[jj].y);
                                mma_f16(Pg[sl][jj][1], ra[2], rb[2], ra[3], rb[3], bf[jj].z, bf[jj].w);
                            }
                        });
                    });
                });
#pragma unroll
                for (int sl = 0; sl < SPW; ++sl) {
                    const float sa =
                        __half2float(__ushort_as_half(static_cast<uint16_t>(s0w[sl][gq >> 1] >> (16 * (gq & 1)))));
                    const float sb =
                        __half2float(__ushort_as_half(static_cast<uint16_t>(s1w[sl][gq >> 1] >> (16 * (gq & 1)))));
#pragma unroll
                    for (int jj = 0; jj < NT; ++jj) {
                        // (elements 0, 1: row r0; 2, 3: row r0 + 8; paired by row)
                        float pg[4];
                        if constexpr (ONECHAIN) {
#pragma unroll
                            for (int e = 0; e < 4; ++e) pg[e] = Pg[sl][jj][0][e];
                        } else {
                            add_x2(pg[0], pg[1], Pg[sl][jj][0][0], Pg[sl][jj][0][1], Pg[sl][jj][1][0], Pg[sl][jj][1][1]);
                            add_x2(pg[2], pg[3], Pg[sl][jj][0][2], Pg[sl][jj][0][3], Pg[sl][jj][1][2], Pg[sl][jj][1][3]);
                        }
                        if constexpr (gq == 0) {
                            mul_x2(accc[sl][jj][0], accc[sl][jj][1], sa, sa, pg[0], pg[1]);
                            mul_x2(accc[sl][jj][2], accc[sl][jj][3], sb, sb, pg[2], pg[3]);
                        } else {
                            fma_x2(accc[sl][jj][0], accc[sl][jj][1], sa, sa, pg[0], pg[1], accc[sl][jj][0],
                                   accc[sl][jj][1]);
                            fma_x2(accc[sl][jj][2], accc[sl][jj][3], sb, sb, pg[2], pg[3], accc[sl][jj][2],
                                   accc[sl][jj][3]);
                        }
                    }
                }
            });
            // bias and offset terms of the chunk, (b | s) x (XS | -XSc) / sigma
            const uint32_t b_r0t = b_r0 + static_cast<uint32_t>(4 * t);
            const uint32_t keep = ng >= kGPC ? 0xFFFFFFFFu
                                : (2 * t + 1 < ng) ? 0xFFFFFFFFu : (2 * t < ng ? 0x0000FFFFu : 0u);
            // one bias-term step: slab sl, tile jj, from its operands
            auto bias_step = [&](auto s_c, auto j_c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint2 rfv,
                                 uint2 sgv, uint4 bb) {
                constexpr int sl = decltype(s_c)::value;
                constexpr int jj = decltype(j_c)::value;
                const float2 rf = make_float2(__uint_as_float(rfv.x), __uint_as_float(rfv.y));
                const float2 sg = make_float2(__uint_as_float(sgv.x), __uint_as_float(sgv.y));
                float Dd[4];
                mma_f16_zc(Dd, a0, a1, a2, a3, bb.x, bb.y);
                mma_f16(Dd, a0, a1, a2, a3, bb.z, bb.w);
                // A = rf * accc + (sg * Dd + A), by pairs (columns 2t, 2t + 1)
                auto add = [&](float (&A)[SPW][NT][4]) {
#pragma unroll
                    for (int h = 0; h < 4; h += 2) {
                        float u0, u1;
                        fma_x2(u0, u1, sg.x, sg.y, Dd[h], Dd[h + 1], A[sl][jj][h], A[sl][jj][h + 1]);
                        fma_x2(A[sl][jj][h], A[sl][jj][h + 1], rf.x, rf.y, accc[sl][jj][h], accc[sl][jj][h + 1],
                               u0, u1);
                    }
                };
                if (NACC == 1 || ipar == 0)
                    add(acc[0]);
                else
                    add(acc[NACC - 1]);
            };
            // (groups past the end of K, stale shared memory on the cp.async path: zeroed)
            if constexpr (EARLY_RELEASE) {
                uint32_t av[SPW][4];
                static_for<0, SPW>([&](auto s_c) {
                    constexpr int sl = decltype(s_c)::value;
                    av[sl][0] = lds32_at<OFF_B + 256 * sl>(b_r0t) & keep;
                    av[sl][1] = lds32_at<OFF_B + 256 * sl + 128>(b_r0t) & keep;
                    av[sl][2] = lds32_at<OFF_S + 256 * sl>(b_r0t) & keep;
                    av[sl][3] = lds32_at<OFF_S + 256 * sl + 128>(b_r0t) & keep;
                });
                // every value the warp reads from the stage is loaded: after the warp
                // barrier one lane releases it (the slot is released already)
                __syncwarp();
                if (lane == 0) mbar_arrive(&wempty[slot]);
                released = true;
                static_for<0, SPW>([&](auto s_c) {
                    constexpr int sl = decltype(s_c)::value;
                    static_for<0, NT>([&](auto j_c) {
                        constexpr int jj = decltype(j_c)::value;
                        bias_step(s_c, j_c, av[sl][0], av[sl][1], av[sl][2], av[sl][3], rfa[jj], sga[jj], bba[jj]);
                    });
                });
            } else {
                static_for<0, SPW>([&](auto s_c) {
                    constexpr int sl = decltype(s_c)::value;
                    const uint32_t a0 = lds32_at<OFF_B + 256 * sl>(b_r0t) & keep;
                    const uint32_t a1 = lds32_at<OFF_B + 256 * sl + 128>(b_r0t) & keep;
                    const uint32_t a2 = lds32_at<OFF_S + 256 * sl>(b_r0t) & keep;
                    const uint32_t a3 = lds32_at<OFF_S + 256 * sl + 128>(b_r0t) & keep;
                    static_for<0, NT>([&](auto j_c) {
                        constexpr int jj = decltype(j_c)::value;
                        bias_step(s_c, j_c, a0, a1, a2, a3, lds64_at<OFF_XT + 4 * (MB + 8 * jj)>(b_t),
                                  lds64_at<OFF_XT + 4 * (8 * jj)>(b_t), lds128_at<OFF_XB + jj * 512>(b_l));
                    });
                });
            }
        }
        if (!released) {
            // every value the warp read from the stage and the slot is in its
            // registers and used; after the warp barrier one lane releases both
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&wempty[slot]);
                mbar_arrive(&fempty[fslot]);
            }
        }
        }
        if (++cslot == S) {
            cslot = 0;
            cphase ^= 1u;
        }
        if (++aslot == F) {
            aslot = 0;
            aphase ^= 1u;
        }
        if constexpr (CPAR == 2) {
            // The next item is the other parity's. While it neither ends this row
            // block nor is followed by a new one (and this item does not end the
            // block either), step over it here: its slots and position only, not
            // a whole visit of the loop.
            if (mine && wi.c + 2 < wi.c1) {
                wi.c += 1;        // the loop step adds the other one
                ipar ^= 1u;
                if (++cslot == S) {
                    cslot = 0;
                    cphase ^= 1u;
                }
                if (++aslot == F) {
                    aslot = 0;
                    aphase ^= 1u;
                }
                continue;
            }
        }

        if (!wi.block_end()) continue;
        if constexpr (NACC == 2) {
            // even items + odd items
#pragma unroll
            for (int sl = 0; sl < SPW; ++sl)
#pragma unroll
                for (int jj = 0; jj < NT; ++jj)
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[0][sl][jj][e] += acc[1][sl][jj][e];
        }
        if constexpr (CPAR > 1) {
            // add the second parity's partial sums in a fixed order: parity 0 + parity 1
            float* sc = combine + (w * SPW * NT * 4) * 32 + lane;
            if (cp == 1 && active) {
#pragma unroll
                for (int sl = 0; sl < SPW; ++sl)
#pragma unroll
                    for (int jj = 0; jj < NT; ++jj)
#pragma unroll
                        for (int e = 0; e < 4; ++e) sc[((sl * NT + jj) * 4 + e) * 32] = acc[0][sl][jj][e];
            }
            named_barrier(1, NCW * 32);
            if (cp == 0 && active) {
#pragma unroll
                for (int sl = 0; sl < SPW; ++sl)
#pragma unroll
                    for (int jj = 0; jj < NT; ++jj)
#pragma unroll
                        for (int e = 0; e < 4; ++e) acc[0][sl][jj][e] += sc[((sl * NT + jj) * 4 + e) * 32];
            }
        }
        if (cp == 0 && active) {
            // this row block's outputs: [M][N] at column n0 of the bank's output
            // (bf16 or fp32), or of its K slice's fp32 partial sums
            const bool partial = p.out_mode == kOutPartial;
            const bool to_bf16 = p.out_mode == kOutBF16;
            void* const out = P.bank[wi.bank].out;
            float* const fbase =
                (partial ? p.partial + static_cast<int64_t>(wi.bank * p.splits + wi.split) * p.M * p.N
                         : static_cast<float*>(out)) + wi.n0;
            __nv_bfloat16* const hbase = static_cast<__nv_bfloat16*>(out) + wi.n0;
            const int mrows = p.M;
#pragma unroll
            for (int sl = 0; sl < SPW; ++sl) {
#pragma unroll
            for (int jj = 0; jj < NT; ++jj) {
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int nl = r0 + kSlab * sl + 8 * hh;
                    if (nl >= wi.rows) continue;
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int mm = 8 * jj + 2 * t + e;
                        if (mm >= mrows) continue;
                        const int64_t idx = static_cast<int64_t>(mm) * p.N + nl;
                        float v = acc[0][sl][jj][2 * hh + e];
                        if constexpr (SWIGLU) {
                            if (!partial) {
                                // gate pass: keep the fp32 gate; up pass: the same thread
                                // wrote this (m, n) gate in the gate pass of this row block
                                float* const g = p.gate + wi.n0 + idx;
                                if (wi.bank == 0) {
                                    *g = v;
                                    continue;
                                }
                                const float gv = *g;
                                v = gv / (1.0f + expf(-gv)) * v;
                            }
                        }
                        if (to_bf16)
                            hbase[idx] = __float2bfloat16_rn(v);
                        else
                            fbase[idx] = v;
                    }
                }
            }
            }
        }
        if constexpr (CPAR > 1) named_barrier(1, NCW * 32);   // the combine scratch is free again
    }
}

// ---------------------------------------------------------------------------
// 2. Split-K reduce: out = sum_{s=0..S-1} partial[s] in slice order.
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
        uint8_t* out = codes + n * K + vb * 32;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t v = (r[q] >> (16 * h)) & 0xFFFFu;
                const int j = slot_shift(BITS, q, h);
                const uint32_t mant = v & 0x3FFu;
                const bool okv = (v & 0xFC00u) == 0x6400u && (mant & ((1u << j) - 1u)) == 0 && (mant >> j) < (1u << BITS);
                out[block_code(BITS, t, q, h)] = okv ? static_cast<uint8_t>(mant >> j) : static_cast<uint8_t>(0xFF);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Host-side launch helpers (defined per code width in qmm_inst_b*.cu).
// ---------------------------------------------------------------------------
struct LaunchCfg {
    int mb;            // 8 or 16
    int lay;           // consumer layout (kNarrow, kWide: 8-row kernel only, kPair)
    int ctas;
    int smem;
    cudaStream_t stream;
};

// Set the dynamic shared-memory limit of one format's main kernels for one row
// tile and consumer layout (every bank capacity).
template <int BITS>
cudaError_t configure_kernels(int group, int mb, int lay, int smem_bytes);

// Weight-box width for a format (host side, for encoding tensor maps).
inline int weight_box_width(int bits, int group) { return wbox_width(bits, group); }
template <int BITS>
cudaError_t launch_forward(int group, const LaunchCfg& L, const MainParams<1>* single, const MainParams<kMaxBanks>* banked,
                           const MainParams<2>* fused);
template <int BITS>
cudaError_t launch_unpack(const uint32_t* w, int64_t K, int64_t N, uint8_t* codes, cudaStream_t stream);

cudaError_t launch_reduce(const ReduceParams& rp, int64_t elems, cudaStream_t stream);

}  // namespace qmmk
