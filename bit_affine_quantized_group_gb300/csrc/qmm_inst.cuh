// Per-code-width launchers. Each qmm_inst_b<BITS>.cu includes this file with
// QMM_INST_BITS defined, so the four widths compile as separate units.
#pragma once

#include "qmm_kernels.cuh"

namespace qmmk {

namespace {
template <int BITS, int GROUP, int MB, int CAP, int LAY>
cudaError_t configure_cap(int smem_bytes) {
    return cudaFuncSetAttribute(qmm_main_kernel<BITS, GROUP, MB, CAP, LAY>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                smem_bytes);
}

// The pair layout is compiled for single projections only; banked and fused
// calls use the narrow or wide layout.
template <int BITS, int GROUP, int MB, int LAY>
cudaError_t configure_one(int smem_bytes) {
    cudaError_t e = configure_cap<BITS, GROUP, MB, 1, LAY>(smem_bytes);
    if constexpr (LAY == kPair) {
        return e;
    } else {
        if (e != cudaSuccess) return e;
        e = configure_cap<BITS, GROUP, MB, 2, LAY>(smem_bytes);
        if (e != cudaSuccess) return e;
        return configure_cap<BITS, GROUP, MB, kMaxBanks, LAY>(smem_bytes);
    }
}

template <int BITS, int GROUP, int MB, int CAP, int LAY>
cudaError_t launch_one(const LaunchCfg& L, const MainParams<CAP>& mp) {
    // The main kernel is a programmatic dependent of whatever precedes it on the
    // stream: it is scheduled as soon as that work allows (its CTAs take SMs as
    // the preceding grid's CTAs leave them) and streams weights at once; its
    // staging warps wait (griddepcontrol.wait) for that work to finish before
    // they read x.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(L.ctas));
    cfg.blockDim = dim3(main_threads(MB, GROUP, LAY));
    cfg.dynamicSmemBytes = static_cast<size_t>(L.smem);
    cfg.stream = L.stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, qmm_main_kernel<BITS, GROUP, MB, CAP, LAY>, mp);
}

template <int BITS, int GROUP, int MB, int LAY>
cudaError_t launch_cap(const LaunchCfg& L, const MainParams<1>* single, const MainParams<kMaxBanks>* banked,
                       const MainParams<2>* fused) {
    if (single) return launch_one<BITS, GROUP, MB, 1, LAY>(L, *single);
    if constexpr (LAY == kPair) {
        return cudaErrorInvalidValue;
    } else {
        if (fused) return launch_one<BITS, GROUP, MB, 2, LAY>(L, *fused);
        return launch_one<BITS, GROUP, MB, kMaxBanks, LAY>(L, *banked);
    }
}

template <int BITS, int GROUP>
cudaError_t configure_group(int mb, int lay, int smem_bytes) {
    if (mb == 16) {
        if (lay == kNarrow) return configure_one<BITS, GROUP, 16, kNarrow>(smem_bytes);
        if (lay == kPair) return configure_one<BITS, GROUP, 16, kPair>(smem_bytes);
        return cudaErrorInvalidValue;
    }
    if (lay == kNarrow) return configure_one<BITS, GROUP, 8, kNarrow>(smem_bytes);
    if (lay == kWide) return configure_one<BITS, GROUP, 8, kWide>(smem_bytes);
    if (lay == kPair) return configure_one<BITS, GROUP, 8, kPair>(smem_bytes);
    return cudaErrorInvalidValue;
}

template <int BITS, int GROUP>
cudaError_t launch_group(const LaunchCfg& L, const MainParams<1>* single, const MainParams<kMaxBanks>* banked,
                         const MainParams<2>* fused) {
    if (L.mb == 16) {
        if (L.lay == kNarrow) return launch_cap<BITS, GROUP, 16, kNarrow>(L, single, banked, fused);
        if (L.lay == kPair) return launch_cap<BITS, GROUP, 16, kPair>(L, single, banked, fused);
        return cudaErrorInvalidValue;
    }
    if (L.lay == kNarrow) return launch_cap<BITS, GROUP, 8, kNarrow>(L, single, banked, fused);
    if (L.lay == kWide) return launch_cap<BITS, GROUP, 8, kWide>(L, single, banked, fused);
    if (L.lay == kPair) return launch_cap<BITS, GROUP, 8, kPair>(L, single, banked, fused);
    return cudaErrorInvalidValue;
}
}  // namespace

template <>
cudaError_t configure_kernels<QMM_INST_BITS>(int group, int mb, int lay, int smem_bytes) {
    constexpr int B = QMM_INST_BITS;
    if (group == 32) return configure_group<B, 32>(mb, lay, smem_bytes);
    if (group == 64) return configure_group<B, 64>(mb, lay, smem_bytes);
    return cudaErrorInvalidValue;
}

template <>
cudaError_t launch_forward<QMM_INST_BITS>(int group, const LaunchCfg& L, const MainParams<1>* single,
                                          const MainParams<kMaxBanks>* banked, const MainParams<2>* fused) {
    constexpr int B = QMM_INST_BITS;
    if (group == 32) return launch_group<B, 32>(L, single, banked, fused);
    if (group == 64) return launch_group<B, 64>(L, single, banked, fused);
    return cudaErrorInvalidValue;
}

template <>
cudaError_t launch_unpack<QMM_INST_BITS>(const uint32_t* w, int64_t K, int64_t N, uint8_t* codes,
                                          cudaStream_t stream) {
    constexpr int B = QMM_INST_BITS;
    const int64_t vbk = K / 32;
    const int64_t total = N * vbk * 4;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 65535) blocks = 65535;
    if (blocks < 1) blocks = 1;
    qmm_unpack_kernel<B><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(w, K, N, codes);
    return cudaGetLastError();
}

}  // namespace qmmk
