// Host-side helpers shared by qmm_api.cu and qmm_noalloc.cu (see qmm_host.h).
#include "qmm_host.h"

#include <cudaTypedefs.h>

#include <mutex>

namespace qmmk {

int stages_for(int bits, int group, int mb, int lay, int optin) {
    if (lay == kWide && mb != 8) return 0;
    const int st = stage_count(bits, group, mb, lay);
    return (st >= 2 && main_smem_bytes(bits, group, mb, lay) <= optin) ? st : 0;
}

// The pair layout keeps two items in flight with one slab a warp, but covers
// only 64 rows an item: it serves calls whose longest CTA range has at most
// four slabs, where the narrow layout would put one item at a time on at most
// four warps. A wide consumer warp owns two slabs of each row block: with CTA
// row ranges of fewer than 96 rows some wide warps would idle while others
// carry two slabs, and with fewer than four weight stages each parity would
// wait for its own refills; the narrow layout (every warp on every item) is
// then faster.
int consumer_layout(int bits, int group, int mb, int64_t rows_total, int64_t ctas, bool single, int optin) {
    if (ctas < 1) return kNarrow;
    const int64_t slabs = (rows_total + kSlab - 1) / kSlab;
    const int64_t longest = (slabs + ctas - 1) / ctas * kSlab;
    if (single && longest <= consumer_rows(kPair) && stages_for(bits, group, mb, kPair, optin) >= 2) return kPair;
    if (mb == 8 && stages_for(bits, group, 8, kWide, optin) >= 4 && rows_total / ctas >= 96) return kWide;
    return kNarrow;
}

int chunk_count(int64_t K, int group) { return static_cast<int>((K / group + kGPC - 1) / kGPC); }

// Per-CTA cost model, fitted on GB300 to the 4-bit group-64 K=17408 N=5120
// projection over 1, 2, 4 and 8 slices: a CTA pays, per row block of up to 128
// rows, one pass over its slice's chunks (chunk bytes at about 28 GB/s per SM)
// plus about 2 us of restart, and slicing adds about 3.7 us for the partial
// sums and their reduce. The work is cut evenly over (bank, slice, row) space,
// so when the CTA count is not a multiple of the bank-slice segments some CTA
// ranges straddle two segments and pay one more row block. A slice may be a
// single chunk.
int auto_split_count(int64_t K, int64_t N, int bits, int group, int64_t banks, int num_sms, int cap) {
    const int C = chunk_count(K, group);
    const double chunk_us = kTN * (chunk_row_bytes(bits, group) + 4.0 * kGPC) / 28e3;
    const double row_block_us = 2.0;
    const double split_us = 3.7;
    int best = 1;
    double best_cost = 0.0;
    for (int s = 1; s <= cap; ++s) {
        if (s > C) break;
        const int64_t rows_total = banks * s * N;
        int64_t ctas = (rows_total + kSlab - 1) / kSlab;
        if (ctas > num_sms) ctas = num_sms;
        const int64_t rows_per_cta = (rows_total + ctas - 1) / ctas;
        int64_t blocks = (rows_per_cta + kTN - 1) / kTN;
        if (ctas % (banks * s) != 0) ++blocks;
        const int per_slice = (C + s - 1) / s;
        // CTA ranges of at most four slabs take the pair layout (two items in
        // flight), measured 10-22 % faster per chunk than one item at a time
        const int64_t slabs = (rows_total + kSlab - 1) / kSlab;
        const bool pair = banks == 1 && (slabs + ctas - 1) / ctas * kSlab <= consumer_rows(kPair);
        const double cost = blocks * (per_slice * chunk_us * (pair ? 0.8 : 1.0) + row_block_us) +
                            (s > 1 ? split_us : 0.0);
        if (s == 1 || cost < best_cost) {
            best = s;
            best_cost = cost;
        }
    }
    return best;
}

cudaError_t configure_format(int bits, int group, int mb, int lay, int smem_bytes) {
    switch (bits) {
        case 2: return configure_kernels<2>(group, mb, lay, smem_bytes);
        case 3: return configure_kernels<3>(group, mb, lay, smem_bytes);
        case 4: return configure_kernels<4>(group, mb, lay, smem_bytes);
        case 5: return configure_kernels<5>(group, mb, lay, smem_bytes);
        case 6: return configure_kernels<6>(group, mb, lay, smem_bytes);
        case 8: return configure_kernels<8>(group, mb, lay, smem_bytes);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_format(int bits, int group, const LaunchCfg& L, const MainParams<1>* single,
                          const MainParams<kMaxBanks>* banked, const MainParams<2>* fused) {
    switch (bits) {
        case 2: return launch_forward<2>(group, L, single, banked, fused);
        case 3: return launch_forward<3>(group, L, single, banked, fused);
        case 4: return launch_forward<4>(group, L, single, banked, fused);
        case 5: return launch_forward<5>(group, L, single, banked, fused);
        case 6: return launch_forward<6>(group, L, single, banked, fused);
        case 8: return launch_forward<8>(group, L, single, banked, fused);
        default: return cudaErrorInvalidValue;
    }
}

namespace {
// cuTensorMapEncodeTiled, fetched once from the driver through the runtime.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}
}  // namespace

bool encode_weight_map(const void* w, int64_t K, int64_t N, int bits, int group, int rows, CUtensorMap* out) {
    auto enc = tensor_map_encoder();
    if (enc == nullptr) return false;
    const int W = wbox_width(bits, group);
    const cuuint64_t row_bytes = static_cast<cuuint64_t>(K * bits / 8);
    const cuuint64_t dims[2] = {row_bytes, static_cast<cuuint64_t>(N)};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(W), static_cast<cuuint32_t>(rows)};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapSwizzle sw = W == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                           : (W == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
    return enc(out, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(w), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_sb_map(const void* a, int64_t G, int64_t N, int rows, CUtensorMap* out) {
    auto enc = tensor_map_encoder();
    if (enc == nullptr) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(G), static_cast<cuuint64_t>(N)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(G) * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kGPC), static_cast<cuuint32_t>(rows)};
    const cuuint32_t estr[2] = {1, 1};
    return enc(out, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(a), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

void set_slice_bounds(MainHeader& h) {
    for (int s = 0; s <= kMaxSplits; ++s)
        h.cb[s] = s <= h.splits ? static_cast<int>(static_cast<int64_t>(s) * h.C / h.splits) : h.C;
}

bool encode_x_map(const void* x, int M, int64_t K, int group, int mb, CUtensorMap* out) {
    auto enc = tensor_map_encoder();
    if (enc == nullptr || M < 1 || K % 64 != 0) return false;
    const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(K / 64), static_cast<cuuint64_t>(M)};
    const cuuint64_t strides[2] = {128, static_cast<cuuint64_t>(K) * 2};
    // one 8-row tile; the 8-row kernel copies only the call's M rows (its rows >= M
    // are never stored, and every row's staging and MMA column is its own)
    const cuuint32_t rows = (mb == 8 && M < 8) ? static_cast<cuuint32_t>(M) : 8u;
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(chunk_codes(group) / 64), rows};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(out, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(x), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace qmmk
