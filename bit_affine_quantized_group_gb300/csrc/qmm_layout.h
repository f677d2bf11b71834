// Layout constants of the qmm kernels, shared by the host dispatch and the
// device code (both sides of the library; nothing here is used by the oracle).
//
// Work decomposition (one main-kernel CTA per SM):
//   * K is cut into chunks of kGPC = 8 scale groups. A CTA walks its rows in
//     row blocks of up to consumer_rows(layout) weight rows (kTN = 128, or 64
//     in the pair layout); one pipeline stage holds one chunk of one row
//     block: the packed code bytes of those rows (TMA tensor boxes) and their
//     8 scales and 8 biases (TMA boxes). A separate ring of activation slots
//     holds, per work item, the raw bfloat16 activation rows of the chunk (one
//     TMA box per 8-row tile) and the chunk's staged activation fragments.
//   * Warp roles: consumer_warps() consumer warps (warp (w, p) owns
//     consumer_slabs(layout) 16-row slabs of every row block, all 8 groups of
//     every chunk, in the stage slots of parity p when there are two consumer
//     parities; the two parities' partial sums are added at the end of the row
//     block), staging_warps activation-staging warps (warp (j, p) turns the
//     raw activations of 8-row tile j into tensor-core fragments in the
//     activation slots it owns) and one weight-copy-issuing producer warp.
//   * Inside a slab the contraction runs on tensor cores with
//     mma.m16n8k16: A = 16 weight rows x 16 codes (unpacked to the exact
//     binary16 values 1024 + q * 2^j), B = 16 codes x 8 activation rows (x
//     times a power-of-two range factor, times 2^-j, in binary16), fp32
//     accumulators. One k32 block of codes feeds two such MMAs.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define QMM_HD __host__ __device__ __forceinline__
#else
#define QMM_HD inline
#endif

namespace qmmk {

constexpr int kGPC = 8;            // scale groups per chunk (pipeline stage)
constexpr int kTN = 128;           // weight rows per row block
constexpr int kSlab = 16;          // rows per MMA slab
constexpr int kSlabs = kTN / kSlab; // 16-row slabs per row block
constexpr int kMaxStages = 8;
// Weight stages the producer issues before it lets the first activation copies
// of the call go ahead of the rest (see the producer in qmm_kernels.cuh).
constexpr int kStagesBeforeX = 2;
// Dynamic shared memory a CTA may opt into on sm_100-class GPUs (GB300: 227 KB).
constexpr int kSmemOptin = 232448;
// Bytes after the mbarriers and the combine scratch for the CTA's work range.
constexpr int kRangeBytes = 32;
constexpr int kReduceThreads = 256;

QMM_HD constexpr int round_up(int v, int a) { return (v + a - 1) / a * a; }
QMM_HD constexpr int log2i(int v) { return v <= 1 ? 0 : 1 + log2i(v / 2); }

// 8-row activation tiles of an MB-row kernel (MB = 8 or 16).
QMM_HD constexpr int n8_tiles(int mb) { return mb / 8; }
// Consumer warps, in one of three layouts, 8 warps each:
//   * narrow: one 16-row slab a warp, every work item (128 rows an item);
//   * wide (8-row kernel only): two slabs a warp (two independent MMA chains
//     sharing the activation fragment loads) in two parities, parity p taking
//     the items in the stage slots of parity p (128 rows an item). It pays when
//     a CTA's row blocks fill most of the 8 slabs and the pipeline keeps
//     several stages per parity;
//   * pair: one slab a warp in two parities, two items in flight; its row
//     blocks (and weight stages) are 64 rows.
// Every layout sums a block's even- and odd-index items apart and adds the two
// at the end, so they all give the same bits.
constexpr int kNarrow = 0;
constexpr int kWide = 1;
constexpr int kPair = 2;
QMM_HD constexpr int consumer_slabs(int lay) { return lay == kWide ? 2 : 1; }
QMM_HD constexpr int consumer_parities(int lay) { return lay == kNarrow ? 1 : 2; }
QMM_HD constexpr int consumer_warps() { return kSlabs; }
// Rows of a row block: the rows one work item covers.
QMM_HD constexpr int consumer_rows(int lay) {
    return kSlab * consumer_slabs(lay) * consumer_warps() / consumer_parities(lay);
}
// Staging warps: staging_per_tile per 8-row activation tile, warp p of a tile
// owning the activation slots s with s % staging_per_tile == p. The 8-row
// kernel takes six, or three in the wide layout with groups of 32: there the raw
// activations of a chunk stay in registers between the staging passes, three
// warps keep up with the consumers, and a CTA of 12 warps (three a scheduler)
// leaves 168 registers a thread instead of 128 (5120 x 17408 calls at 8 rows
// 0.8 % faster with 4-bit codes, 2.7 % with 5-bit, 6.7 % with 6-bit; with groups
// of 64 and in the other layouts three staging warps measured 1-15 % slower).
// The 16-row kernel takes two per tile.
QMM_HD constexpr int staging_per_tile(int mb, int group, int lay) {
    return mb == 8 ? (group == 32 && lay == kWide ? 3 : 6) : 2;
}
QMM_HD constexpr int staging_warps(int mb, int group, int lay) {
    return staging_per_tile(mb, group, lay) * n8_tiles(mb);
}
QMM_HD constexpr int main_threads(int mb, int group, int lay) {
    return (consumer_warps() + staging_warps(mb, group, lay) + 1) * 32;
}
// F activation slots suit spt staging warps a tile when every warp owns whole
// slots: F at most spt, or a multiple of it.
QMM_HD constexpr bool slots_fit(int f, int spt) { return f <= spt || f % spt == 0; }

// k32 blocks per scale group and per chunk.
QMM_HD constexpr int vblocks_per_group(int group) { return group / 32; }
QMM_HD constexpr int vblocks_per_chunk(int group) { return kGPC * vblocks_per_group(group); }
// Codes of one row in a full chunk.
QMM_HD constexpr int chunk_codes(int group) { return kGPC * group; }
// Bytes of one weight row that one k32 block consumes.
QMM_HD constexpr int vblock_bytes(int bits) { return 4 * bits; }
// Packed bytes of one weight row in a full chunk.
QMM_HD constexpr int chunk_row_bytes(int bits, int group) { return kGPC * group * bits / 8; }
// The weight tile of a stage arrives as TMA boxes of kTN rows x W bytes, W the
// widest of 128/64/32 that divides the chunk row, stored with the matching
// shared-memory swizzle (16-byte chunk c of row r lands at c ^ f(r)), so every
// box row is one full-line request and the consumers' reads hit distinct banks.
QMM_HD constexpr int wbox_width(int bits, int group) {
    return chunk_row_bytes(bits, group) % 128 == 0 ? 128 : (chunk_row_bytes(bits, group) % 64 == 0 ? 64 : 32);
}
QMM_HD constexpr int wbox_count(int bits, int group) { return chunk_row_bytes(bits, group) / wbox_width(bits, group); }

// Staged activations of a chunk, written by the staging warps into the stage:
// MMA B fragments (one 16-byte vector per lane per k32 block per 8-row tile),
// the bias-term fragments (one 16-byte vector per lane per tile), and two
// factors per activation row (the bias-term range factor sigma and 1/f, f the
// x range factor).
QMM_HD constexpr int xfrag_bytes(int group, int mb) { return vblocks_per_chunk(group) * n8_tiles(mb) * 512; }
QMM_HD constexpr int xbias_bytes(int mb) { return n8_tiles(mb) * 512; }
QMM_HD constexpr int xstaged_bytes(int group, int mb) {
    return round_up(xfrag_bytes(group, mb) + xbias_bytes(mb) + 2 * mb * 4, 128);
}

// Raw activations of one chunk, per 8-row tile one 3-D TMA box of x viewed as
// [M rows][K/64 blocks][64 codes]: [MB/8][8][chunk_codes/64][128 bytes], each
// 128-byte line stored with the 128-byte swizzle (so the staging warps' 16-byte
// reads of 8 different rows fall in different banks); the 16-row kernel's rows
// >= M arrive as zeros, the 8-row kernel copies only M rows when M < 8.
QMM_HD constexpr int xraw_bytes(int group, int mb) { return 2 * chunk_codes(group) * mb; }

// Weight stage (one chunk of one row block of consumer_rows(lay) rows:
// kTN, or 64 for the pair layout; 1024-byte aligned, the swizzle atom):
// packed codes, scales, biases.
QMM_HD constexpr int stage_weight_bytes(int bits, int group, int lay) {
    return consumer_rows(lay) * chunk_row_bytes(bits, group);
}
QMM_HD constexpr int stage_sb_bytes(int lay) { return consumer_rows(lay) * 16; }   // 8 binary16 values per row
QMM_HD constexpr int wstage_bytes(int bits, int group, int lay) {
    return round_up(stage_weight_bytes(bits, group, lay) + 2 * stage_sb_bytes(lay), 1024);
}
// Activation slot (one chunk): raw activations (1024-byte aligned) and the
// staged fragments.
QMM_HD constexpr int aslot_bytes(int group, int mb) { return round_up(xraw_bytes(group, mb) + xstaged_bytes(group, mb), 1024); }

// Scratch for adding the second consumer parity's partial sums at the end of
// a row block (wide and pair layouts): [slab][tile][4][32 lanes] floats.
QMM_HD constexpr int combine_bytes(int mb, int lay) {
    return consumer_parities(lay) > 1 ? consumer_rows(lay) / kSlab * n8_tiles(mb) * 4 * 32 * 4 : 0;
}

// Dynamic shared memory of the main kernel with S weight stages and F
// activation slots: the stages, the slots, two mbarriers per weight stage
// (landed, consumed), per activation slot one per tile (raw landed) and two
// more (staged, consumed), the combine scratch, the CTA's work range and one
// more mbarrier (first activation copies issued).
// 1024 bytes of slack let the kernel align its rings to 1024.
QMM_HD constexpr int main_smem_bytes(int bits, int group, int mb, int lay, int S, int F) {
    return 1024 + S * wstage_bytes(bits, group, lay) + F * aslot_bytes(group, mb) + (2 * S + (2 + n8_tiles(mb)) * F) * 8 +
           combine_bytes(mb, lay) + kRangeBytes + 8;
}
// The most weight stages (<= kMaxStages) that fit kSmemOptin next to F
// activation slots, a multiple of the consumer parities (each parity owns the
// stages of its parity); 0 if fewer than two fit.
QMM_HD constexpr int weight_stages_for(int bits, int group, int mb, int lay, int F) {
    return (main_smem_bytes(bits, group, mb, lay, 8, F) <= kSmemOptin   ? 8
          : main_smem_bytes(bits, group, mb, lay, 7, F) <= kSmemOptin ? 7
          : main_smem_bytes(bits, group, mb, lay, 6, F) <= kSmemOptin ? 6
          : main_smem_bytes(bits, group, mb, lay, 5, F) <= kSmemOptin ? 5
          : main_smem_bytes(bits, group, mb, lay, 4, F) <= kSmemOptin ? 4
          : main_smem_bytes(bits, group, mb, lay, 3, F) <= kSmemOptin ? 3
          : main_smem_bytes(bits, group, mb, lay, 2, F) <= kSmemOptin ? 2
                                                                        : 0) /
           consumer_parities(lay) * consumer_parities(lay);
}
// Activation slots: a multiple of the consumer parities, and either at most
// the staging warps per tile or a multiple of them (each warp owns whole
// slots). The 8-row kernel takes the larger choice that still leaves four
// weight stages; the 16-row kernel, whose slots are twice as large, takes two
// and gives the room to weight stages (measured faster than four slots).
QMM_HD constexpr int act_slots(int bits, int group, int mb, int lay) {
    return mb == 8 ? (weight_stages_for(bits, group, mb, lay, 6) >= 4 ? 6
                      : weight_stages_for(bits, group, mb, lay, 4) >= 4 && slots_fit(4, staging_per_tile(mb, group, lay))
                          ? 4
                          : 2)
                   : 2;
}
QMM_HD constexpr int stage_count(int bits, int group, int mb, int lay) {
    return weight_stages_for(bits, group, mb, lay, act_slots(bits, group, mb, lay));
}
QMM_HD constexpr int main_smem_bytes(int bits, int group, int mb, int lay) {
    return main_smem_bytes(bits, group, mb, lay, stage_count(bits, group, mb, lay), act_slots(bits, group, mb, lay));
}

}  // namespace qmmk
