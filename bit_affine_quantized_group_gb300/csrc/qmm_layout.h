// Layout constants of the qmm kernels, shared by the host dispatch and the
// device code (both sides of the library; nothing here is used by the oracle).
//
// Work decomposition (one main-kernel CTA per SM):
//   * K is cut into chunks of kGPC = 8 scale groups; one pipeline stage holds
//     one chunk for a row block of up to kTN = 128 weight rows: the packed
//     code bytes of those rows (TMA tensor boxes), their 8 scales and 8 biases
//     (TMA boxes), and the staged activation fragments of the chunk (one bulk
//     copy).
//   * A row block is 8 slabs of 16 rows. There are 8 consumer warps and one
//     producer warp. Consumer warp w owns slabs (w % 4) and (w % 4) + 4 and
//     the groups 4*(w / 4) .. 4*(w / 4) + 3 of every chunk, so each slab pair
//     is split between two warps along K; their partial sums are added in a
//     fixed order through a small shared-memory scratch at the end of the row
//     block.
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
constexpr int kSlabPairs = 4;      // consumer warps along the rows
constexpr int kKParts = 2;         // consumer warps along K (halves of a chunk)
constexpr int kNCW = kSlabPairs * kKParts;   // consumer warps
constexpr int kSPW = 2;            // slabs per consumer warp
constexpr int kGroupsPerWarp = kGPC / kKParts;
constexpr int kThreads = (kNCW + 1) * 32;
constexpr int kMaxStages = 8;
constexpr int kXprepThreads = 256;
constexpr int kReduceThreads = 256;

QMM_HD constexpr int round_up(int v, int a) { return (v + a - 1) / a * a; }

// k32 blocks per scale group.
QMM_HD constexpr int vblocks_per_group(int bits, int group) { return (void)bits, group / 32; }
QMM_HD constexpr int vblocks_per_chunk(int bits, int group) {
    return kGPC * vblocks_per_group(bits, group);
}
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
QMM_HD constexpr int log2i(int v) { return v <= 1 ? 0 : 1 + log2i(v / 2); }

// Staged activations, per chunk: MMA B fragments (one 16-byte vector per lane
// per k32 block per 8-row tile), the bias-term fragments, and two factors per
// activation row (the bias-term range factor and 1/f, f the x range factor).
QMM_HD constexpr int n8_tiles(int mb) { return mb / 8; }
QMM_HD constexpr int xprep_frag_bytes(int bits, int group, int mb) {
    return vblocks_per_chunk(bits, group) * n8_tiles(mb) * 512;
}
QMM_HD constexpr int xprep_bias_bytes(int mb) { return n8_tiles(mb) * 512; }
QMM_HD constexpr int xprep_chunk_bytes(int bits, int group, int mb) {
    return round_up(xprep_frag_bytes(bits, group, mb) + xprep_bias_bytes(mb) + 2 * mb * 4, 128);
}

// One pipeline stage in shared memory (1024-byte aligned: the swizzle atom).
QMM_HD constexpr int stage_weight_bytes(int bits, int group) { return kTN * chunk_row_bytes(bits, group); }
QMM_HD constexpr int stage_sb_bytes() { return kTN * 16; }   // 8 binary16 values per row
QMM_HD constexpr int stage_bytes(int bits, int group, int mb) {
    return round_up(stage_weight_bytes(bits, group) + 2 * stage_sb_bytes() + xprep_chunk_bytes(bits, group, mb), 1024);
}

// Scratch for adding the two K halves of every slab pair at a row block's end.
QMM_HD constexpr int reduce_scratch_bytes(int mb) { return kSlabPairs * kSPW * n8_tiles(mb) * 4 * 32 * 4; }
// Dynamic shared memory of the main kernel with `stages` pipeline stages.
// (1024 bytes of slack let the kernel align its stage ring to 1024.)
QMM_HD constexpr int main_smem_bytes(int bits, int group, int mb, int stages) {
    return 1024 + stages * stage_bytes(bits, group, mb) + stages * 16 + reduce_scratch_bytes(mb);
}


}  // namespace qmmk
