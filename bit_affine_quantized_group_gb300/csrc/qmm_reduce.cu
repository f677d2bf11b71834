// Split-K reduce kernel: out[bank][m][n] = sum over slices s = 0..S-1, in that
// order, of the fp32 partials (vmlx-swift PR #565, "JANGH split-K verify tile"
// commit: K slices write FP32 partials which are then summed). For the fused
// gate/up projection it writes silu(gate sum) * (up sum) to the one output.
#include "qmm_kernels.cuh"

namespace qmmk {

__global__ void __launch_bounds__(kReduceThreads) qmm_splitk_reduce_kernel(const __grid_constant__ ReduceParams p) {
    // the next kernel on the stream may be scheduled now; the partials of the
    // main kernel are complete and visible after the wait
    griddep_launch_dependents();
    griddep_wait();
    const int64_t per_bank = static_cast<int64_t>(p.M) * p.N;
    const int64_t total = per_bank * (p.swiglu ? 1 : p.banks);
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t bank = i / per_bank;
        const int64_t e = i - bank * per_bank;
        const float* src = p.partial + bank * p.splits * per_bank + e;
        float s = src[0];
        for (int sp = 1; sp < p.splits; ++sp) s += src[sp * per_bank];
        if (p.swiglu) {
            // fused gate/up: bank 0 holds the gate slices, bank 1 the up slices
            const float* usrc = p.partial + p.splits * per_bank + e;
            float u = usrc[0];
            for (int sp = 1; sp < p.splits; ++sp) u += usrc[sp * per_bank];
            s = s / (1.0f + expf(-s)) * u;
        }
        if (p.out_bf16)
            static_cast<__nv_bfloat16*>(p.out[bank])[e] = __float2bfloat16_rn(s);
        else
            static_cast<float*>(p.out[bank])[e] = s;
    }
}

cudaError_t launch_reduce(const ReduceParams& rp, int64_t elems, cudaStream_t stream) {
    int64_t blocks = (elems + kReduceThreads - 1) / kReduceThreads;
    if (blocks > 4096) blocks = 4096;
    if (blocks < 1) blocks = 1;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(kReduceThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, qmm_splitk_reduce_kernel, rp);
}

}  // namespace qmmk
