// Host-side helpers shared by the plan path (qmm_api.cu) and the no-allocation
// entry point (qmm_noalloc.cu): pipeline depth, kernel configuration and
// launch dispatch by code width, and TMA tensor-map encoding of the weights,
// scales and biases. Not part of the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "qmm_kernels.cuh"

namespace qmmk {

// The format's pipeline depth (stage_count, fixed at compile time) for a row
// tile and consumer layout when its main-kernel shared memory fits `optin`
// bytes; 0 otherwise (also for the wide layout of the 16-row tile).
int stages_for(int bits, int group, int mb, int lay, int optin);

// Consumer layout (kNarrow, kWide, kPair) of a call's main kernel over
// rows_total flattened rows on `ctas` CTAs; `single`: one projection (the
// pair layout is compiled for those only).
int consumer_layout(int bits, int group, int mb, int64_t rows_total, int64_t ctas, bool single, int optin);

// 8-group chunks along K.
int chunk_count(int64_t K, int group);

// The chunk bounds of the header's K slices (h.cb, from h.C and h.splits).
void set_slice_bounds(MainHeader& h);

// Automatic K-slice count (1..cap) for `banks` projections of K x N in one
// format on `num_sms` SMs, from a per-CTA cost model (see qmm_host.cu).
int auto_split_count(int64_t K, int64_t N, int bits, int group, int64_t banks, int num_sms, int cap);

// Set the main kernels' dynamic shared-memory limit for one format, row tile
// and consumer layout.
cudaError_t configure_format(int bits, int group, int mb, int lay, int smem_bytes);

// Launch the main kernel of one format (exactly one of the parameter blocks is non-null).
cudaError_t launch_format(int bits, int group, const LaunchCfg& L, const MainParams<1>* single,
                          const MainParams<kMaxBanks>* banked, const MainParams<2>* fused);

// Packed codes as uint8 [N][K*bits/8], box `rows` rows (the consumer layout's
// block rows) x W bytes with the W-byte swizzle.
bool encode_weight_map(const void* w, int64_t K, int64_t N, int bits, int group, int rows, CUtensorMap* out);
// Scales or biases as uint16 [N][G], box `rows` rows x 8 values, unswizzled.
bool encode_sb_map(const void* a, int64_t G, int64_t N, int rows, CUtensorMap* out);
// Activations x [M][K] bfloat16 (16-byte aligned, K % 64 == 0) viewed as
// [M][K/64][64], box 64 x (codes per chunk / 64) x 8 rows (M rows for the 8-row
// kernel when M < 8), 128-byte swizzle.
bool encode_x_map(const void* x, int M, int64_t K, int group, int mb, CUtensorMap* out);

}  // namespace qmmk
