// qmm_forward_noalloc: the single-projection forward for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at the point
// where they run a projection: code that runs while another component owns the
// device allocator, real-time or embedded loops that forbid allocation after
// start-up, and plug-in hosts that expose only the tensors they pass in. For
// them this entry point needs no plan and no workspace: the per-call
// activation staging that qmm_forward keeps in its plan's workspace lives in a
// file-scope device array instead, reserved when the library is loaded and
// held by every GPU that loads it until the process exits.
//
// The kernels are the ones qmm_forward launches; only where their scratch
// lives differs. Split-K is not offered here (splits is always 1), so no
// partial sums need storage.
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "../../include/qmm.h"
#include "qmm_kernels.cuh"

using namespace qmmk;

namespace {

// First 256 bytes: the kernels' error word; then the staged activations.
constexpr size_t kErrArea = 256;
static_assert(QMM_NOALLOC_SCRATCH_BYTES % 256 == 0, "scratch size");

}  // namespace

// The scratch itself. In host code this name is only a stand-in: its device
// address comes from cudaGetSymbolAddress, once per device, with that device current.
static __device__ __align__(256) uint8_t g_noalloc_scratch[QMM_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;

struct DeviceSetup {
    bool ready;
    uint8_t* scratch;         // device address of g_noalloc_scratch on this device
    int num_sms;
    int optin;
    uint32_t configured;      // bit (bits_index * 4 + group_index * 2 + mb_index): kernel attributes set
};

DeviceSetup g_dev[kMaxDevices];
std::mutex g_mutex;

int bits_index(int bits) { return bits == 2 ? 4 : bits == 3 ? 5 : bits == 4 ? 0 : bits == 5 ? 1 : bits == 6 ? 2 : 3; }

cudaError_t configure_format(int bits, int group, int mb, int smem) {
    switch (bits) {
        case 2: return configure_kernels<2>(group, mb, smem);
        case 3: return configure_kernels<3>(group, mb, smem);
        case 4: return configure_kernels<4>(group, mb, smem);
        case 5: return configure_kernels<5>(group, mb, smem);
        case 6: return configure_kernels<6>(group, mb, smem);
        default: return configure_kernels<8>(group, mb, smem);
    }
}

cudaError_t launch_format(int bits, int group, const LaunchCfg& L, const MainParams<1>* mp) {
    switch (bits) {
        case 2: return launch_forward<2>(group, L, mp, nullptr, nullptr);
        case 3: return launch_forward<3>(group, L, mp, nullptr, nullptr);
        case 4: return launch_forward<4>(group, L, mp, nullptr, nullptr);
        case 5: return launch_forward<5>(group, L, mp, nullptr, nullptr);
        case 6: return launch_forward<6>(group, L, mp, nullptr, nullptr);
        default: return launch_forward<8>(group, L, mp, nullptr, nullptr);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
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

// Same tensor-map shapes the plan path uses: codes as uint8 [N][K*bits/8] in
// kTN x W swizzled boxes; scales/biases as uint16 [N][K/group] in kTN x 8 boxes.
bool encode_maps(const qmm_desc& d, const void* w, const void* s, const void* b, bool sb_tma, CUtensorMap* mw,
                 CUtensorMap* ms, CUtensorMap* mb) {
    auto enc = encoder();
    if (enc == nullptr) return false;
    const int W = wbox_width(d.bits, d.group);
    const cuuint64_t row_bytes = static_cast<cuuint64_t>(d.K * d.bits / 8);
    const cuuint64_t wdims[2] = {row_bytes, static_cast<cuuint64_t>(d.N)};
    const cuuint64_t wstr[1] = {row_bytes};
    const cuuint32_t wbox[2] = {static_cast<cuuint32_t>(W), static_cast<cuuint32_t>(kTN)};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapSwizzle sw = W == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                           : (W == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
    if (enc(mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(w), wdims, wstr, wbox, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    if (!sb_tma) return true;
    const cuuint64_t G = static_cast<cuuint64_t>(d.K / d.group);
    const cuuint64_t sdims[2] = {G, static_cast<cuuint64_t>(d.N)};
    const cuuint64_t sstr[1] = {G * 2};
    const cuuint32_t sbox[2] = {static_cast<cuuint32_t>(kGPC), static_cast<cuuint32_t>(kTN)};
    for (int i = 0; i < 2; ++i) {
        if (enc(i == 0 ? ms : mb, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(i == 0 ? s : b), sdims, sstr,
                sbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    return true;
}

}  // namespace

extern "C" int qmm_forward_noalloc(const void* x_bf16, int M, const uint32_t* packed_w, const uint16_t* scales_f16,
                                   const uint16_t* biases_f16, int64_t K, int64_t N, int bits, int group,
                                   int out_dtype, void* out, void* stream) {
    // 1. Host-only checks, identical to qmm_forward's (with splits = 1, one bank).
    qmm_desc d;
    std::memset(&d, 0, sizeof(d));
    d.K = K;
    d.N = N;
    d.bits = bits;
    d.group = group;
    d.max_M = QMM_MAX_ROWS;
    d.out_dtype = out_dtype;
    d.splits = 1;
    d.max_banks = 1;
    const int v = qmm_validate_desc(&d);
    if (v != QMM_OK) return v;
    const int chk = qmm_check_forward_args(&d, x_bf16, M, 1, &packed_w, &scales_f16, &biases_f16, K, N, bits, group,
                                           &out);
    if (chk != QMM_OK) return chk;
    if (M == 0) return QMM_OK;

    // 2. The staged activations must fit the static scratch.
    const int mb = M > 8 ? 16 : 8;
    const int G = static_cast<int>(K / group);
    const int C = (G + kGPC - 1) / kGPC;
    const size_t xprep_bytes = static_cast<size_t>(C) * xprep_chunk_bytes(bits, group, mb);
    if (kErrArea + xprep_bytes > QMM_NOALLOC_SCRATCH_BYTES) return QMM_ERR_SCRATCH_LIMIT;

    // 3. Once per device (with that device current): the scratch's device
    //    address, device limits, and the kernels' shared-memory attribute.
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QMM_ERR_CUDA;
    const uint32_t cfg_bit = 1u << (bits_index(bits) * 4 + (group == 64 ? 2 : 0) + (mb == 16 ? 1 : 0));
    DeviceSetup ds;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        DeviceSetup& s = g_dev[dev];
        if (!s.ready) {
            void* ptr = nullptr;
            if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) return QMM_ERR_CUDA;
            int sms = 0, optin = 0;
            if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return QMM_ERR_CUDA;
            if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
                return QMM_ERR_CUDA;
            s.scratch = static_cast<uint8_t*>(ptr);
            s.num_sms = sms;
            s.optin = optin;
            s.configured = 0;
            s.ready = true;
        }
        int stages = (s.optin - 2048 - reduce_scratch_bytes(mb)) / (stage_bytes(bits, group, mb) + 16);
        if (stages > kMaxStages) stages = kMaxStages;
        if (stages < 2) return QMM_ERR_UNSUPPORTED;
        if (!(s.configured & cfg_bit)) {
            if (configure_format(bits, group, mb, main_smem_bytes(bits, group, mb, stages)) != cudaSuccess)
                return QMM_ERR_CUDA;
            s.configured |= cfg_bit;
        }
        ds = s;
    }
    int stages = (ds.optin - 2048 - reduce_scratch_bytes(mb)) / (stage_bytes(bits, group, mb) + 16);
    if (stages > kMaxStages) stages = kMaxStages;

    // 4. Launch the same kernels qmm_forward launches, pointed at the scratch.
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // the error word must start at zero for this call (the staging area is fully rewritten)
    if (cudaMemsetAsync(ds.scratch, 0, sizeof(uint32_t), st) != cudaSuccess) return QMM_ERR_CUDA;

    MainParams<1> mp;
    std::memset(&mp, 0, sizeof(mp));
    MainHeader& h = mp.h;
    h.xprep = ds.scratch + kErrArea;
    h.partial = nullptr;
    h.err = reinterpret_cast<uint32_t*>(ds.scratch);
    h.N = N;
    h.K = K;
    h.row_bytes = K * bits / 8;
    h.G = G;
    h.C = C;
    h.splits = 1;
    h.M = M;
    h.stages = stages;
    h.out_mode = out_dtype == QMM_OUT_F32 ? kOutF32 : kOutBF16;
    h.sb_tma = (G % 8 == 0) ? 1 : 0;
    h.sb_vec16 = h.sb_tma;
    h.unpack_magic = kF16x2_1024;
    h.banks = 1;
    h.xprep_bytes = static_cast<int64_t>(xprep_bytes);
    h.rows_total = N;
    mp.bank[0].w = packed_w;
    mp.bank[0].s = scales_f16;
    mp.bank[0].b = biases_f16;
    mp.bank[0].out = out;
    if (!encode_maps(d, packed_w, scales_f16, biases_f16, h.sb_tma != 0, &mp.tmw[0], &mp.tms[0], &mp.tmb[0]))
        return QMM_ERR_CUDA;

    int64_t ctas = (N + kSlab - 1) / kSlab;
    if (ctas > ds.num_sms) ctas = ds.num_sms;
    LaunchCfg L;
    L.x = static_cast<const uint16_t*>(x_bf16);
    L.M = M;
    L.mb = mb;
    L.ctas = static_cast<int>(ctas);
    L.smem = main_smem_bytes(bits, group, mb, stages);
    L.stream = st;
    return launch_format(bits, group, L, &mp) == cudaSuccess ? QMM_OK : QMM_ERR_CUDA;
}
