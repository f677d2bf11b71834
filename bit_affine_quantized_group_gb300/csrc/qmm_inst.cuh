// Per-code-width launchers. Each qmm_inst_b<BITS>.cu includes this file with
// QMM_INST_BITS defined, so the four widths compile as separate units.
#pragma once

#include "qmm_kernels.cuh"

namespace qmmk {

namespace {
template <int BITS, int GROUP, int MB, bool WIDE>
cudaError_t configure_one(int smem_bytes) {
    cudaError_t e = cudaFuncSetAttribute(qmm_main_kernel<BITS, GROUP, MB, 1, WIDE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(qmm_main_kernel<BITS, GROUP, MB, 2, WIDE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem_bytes);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(qmm_main_kernel<BITS, GROUP, MB, kMaxBanks, WIDE>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
}

template <int BITS, int GROUP, int MB, int CAP, bool WIDE>
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
    cfg.blockDim = dim3(main_threads(MB));
    cfg.dynamicSmemBytes = static_cast<size_t>(L.smem);
    cfg.stream = L.stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, qmm_main_kernel<BITS, GROUP, MB, CAP, WIDE>, mp);
}

template <int BITS, int GROUP, int MB, bool WIDE>
cudaError_t launch_cap(const LaunchCfg& L, const MainParams<1>* single, const MainParams<kMaxBanks>* banked,
                       const MainParams<2>* fused) {
    if (single) return launch_one<BITS, GROUP, MB, 1, WIDE>(L, *single);
    if (fused) return launch_one<BITS, GROUP, MB, 2, WIDE>(L, *fused);
    return launch_one<BITS, GROUP, MB, kMaxBanks, WIDE>(L, *banked);
}

template <int BITS, int GROUP>
cudaError_t configure_group(int mb, bool wide, int smem_bytes) {
    if (mb == 16) return wide ? cudaErrorInvalidValue : configure_one<BITS, GROUP, 16, false>(smem_bytes);
    return wide ? configure_one<BITS, GROUP, 8, true>(smem_bytes) : configure_one<BITS, GROUP, 8, false>(smem_bytes);
}

template <int BITS, int GROUP>
cudaError_t launch_group(const LaunchCfg& L, const MainParams<1>* single, const MainParams<kMaxBanks>* banked,
                         const MainParams<2>* fused) {
    if (L.mb == 16)
        return L.wide ? cudaErrorInvalidValue : launch_cap<BITS, GROUP, 16, false>(L, single, banked, fused);
    return L.wide ? launch_cap<BITS, GROUP, 8, true>(L, single, banked, fused)
                  : launch_cap<BITS, GROUP, 8, false>(L, single, banked, fused);
}
}  // namespace

template <>
cudaError_t configure_kernels<QMM_INST_BITS>(int group, int mb, bool wide, int smem_bytes) {
    constexpr int B = QMM_INST_BITS;
    if (group == 32) return configure_group<B, 32>(mb, wide, smem_bytes);
    if (group == 64) return configure_group<B, 64>(mb, wide, smem_bytes);
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
