// qmm_forward_noalloc: the single-projection forward for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at the point
// where they run a projection: code that runs while another component owns the
// device allocator, real-time or embedded loops that forbid allocation after
// start-up, and plug-in hosts that expose only the tensors they pass in. For
// them this entry point needs no plan and no workspace: the device scratch
// that qmm_forward keeps in its plan's workspace (the kernels' error word and
// the fp32 partial sums of K-sliced projections) lives in a file-scope device
// array instead, reserved when the library is loaded and held by every GPU
// that loads it until the process exits.
//
// The kernels are the ones qmm_forward launches; only where their scratch
// lives differs. The K-slice count is the one an automatic plan would choose,
// lowered until the partial sums fit the array (one slice needs none).
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "../../include/qmm.h"
#include "qmm_host.h"

using namespace qmmk;

namespace {

// First 256 bytes: the kernels' error word; then the split-K partial sums.
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
    uint64_t configured;      // bit (bits_index * 8 + group_index * 4 + 3 * (16-row tile) + layout): attributes set
};

DeviceSetup g_dev[kMaxDevices];
std::mutex g_mutex;

int bits_index(int bits) { return bits == 2 ? 4 : bits == 3 ? 5 : bits == 4 ? 0 : bits == 5 ? 1 : bits == 6 ? 2 : 3; }

}  // namespace

extern "C" int qmm_forward_noalloc(const void* x_bf16, int M, const uint32_t* packed_w, const uint16_t* scales_f16,
                                   const uint16_t* biases_f16, int64_t K, int64_t N, int bits, int group,
                                   int out_dtype, void* out, void* stream) {
    // 1. Host-only checks, identical to qmm_forward's (one bank).
    qmm_desc d;
    std::memset(&d, 0, sizeof(d));
    d.K = K;
    d.N = N;
    d.bits = bits;
    d.group = group;
    d.max_M = QMM_MAX_ROWS;
    d.out_dtype = out_dtype;
    d.splits = 0;
    d.max_banks = 1;
    const int v = qmm_validate_desc(&d);
    if (v != QMM_OK) return v;
    const int chk = qmm_check_forward_args(&d, x_bf16, M, 1, &packed_w, &scales_f16, &biases_f16, K, N, bits, group,
                                           &out);
    if (chk != QMM_OK) return chk;
    if (M == 0) return QMM_OK;

    // 2. Once per device (with that device current): the scratch's device
    //    address, device limits, and the kernels' shared-memory attribute.
    const int mb = M > 8 ? 16 : 8;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QMM_ERR_CUDA;
    DeviceSetup ds;
    int stages = 0;
    int lay = kNarrow;
    int splits = 1;
    const int C = chunk_count(K, group);
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
        // 3. K slices: the automatic choice, lowered until the partial sums fit;
        //    then the consumer layout, as qmm_forward chooses it.
        int cap = C;
        if (cap > 8) cap = 8;
        splits = auto_split_count(K, N, bits, group, 1, s.num_sms, cap);
        const size_t per_split = static_cast<size_t>(M) * static_cast<size_t>(N) * sizeof(float);
        while (splits > 1 && kErrArea + static_cast<size_t>(splits) * per_split > QMM_NOALLOC_SCRATCH_BYTES) --splits;
        const int64_t rows = static_cast<int64_t>(splits) * N;
        int64_t ctas = (rows + kSlab - 1) / kSlab;
        if (ctas > s.num_sms) ctas = s.num_sms;
        lay = consumer_layout(bits, group, mb, rows, ctas, true, s.optin);
        stages = stages_for(bits, group, mb, lay, s.optin);
        if (stages < 2) return QMM_ERR_UNSUPPORTED;
        const int layout = (mb == 16 ? 3 : 0) + lay;
        const uint64_t cfg_bit = 1ull << (bits_index(bits) * 8 + (group == 64 ? 4 : 0) + layout);
        if (!(s.configured & cfg_bit)) {
            if (configure_format(bits, group, mb, lay, main_smem_bytes(bits, group, mb, lay)) != cudaSuccess)
                return QMM_ERR_CUDA;
            s.configured |= cfg_bit;
        }
        ds = s;
    }

    // 4. Launch the kernels qmm_forward launches, pointed at the scratch.
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // the error word must start at zero for this call
    if (cudaMemsetAsync(ds.scratch, 0, sizeof(uint32_t), st) != cudaSuccess) return QMM_ERR_CUDA;

    MainParams<1> mp;
    std::memset(&mp, 0, sizeof(mp));
    MainHeader& h = mp.h;
    h.x = static_cast<const uint16_t*>(x_bf16);
    h.partial = reinterpret_cast<float*>(ds.scratch + kErrArea);
    h.err = reinterpret_cast<uint32_t*>(ds.scratch);
    h.N = N;
    h.K = K;
    h.G = static_cast<int>(K / group);
    h.C = C;
    h.splits = splits;
    set_slice_bounds(h);
    h.M = M;
    h.out_mode = splits > 1 ? kOutPartial : (out_dtype == QMM_OUT_F32 ? kOutF32 : kOutBF16);
    h.sb_tma = (h.G % 8 == 0) ? 1 : 0;
    h.unpack_magic = kF16x2_1024;
    h.banks = 1;
    h.rows_total = static_cast<int64_t>(splits) * N;
    mp.bank[0].w = packed_w;
    mp.bank[0].s = scales_f16;
    mp.bank[0].b = biases_f16;
    mp.bank[0].out = out;
    const int rows = consumer_rows(lay);   // weight and scale boxes: one row block
    if (!encode_weight_map(packed_w, K, N, bits, group, rows, &mp.tmw[0])) return QMM_ERR_CUDA;
    if (!encode_x_map(x_bf16, M, K, group, mb, &mp.tmx)) return QMM_ERR_CUDA;
    if (h.sb_tma &&
        (!encode_sb_map(scales_f16, h.G, N, rows, &mp.tms[0]) || !encode_sb_map(biases_f16, h.G, N, rows, &mp.tmb[0])))
        return QMM_ERR_CUDA;

    int64_t ctas = (h.rows_total + kSlab - 1) / kSlab;
    if (ctas > ds.num_sms) ctas = ds.num_sms;
    LaunchCfg L;
    L.mb = mb;
    L.lay = lay;
    L.ctas = static_cast<int>(ctas);
    L.smem = main_smem_bytes(bits, group, mb, lay);
    L.stream = st;
    if (launch_format(bits, group, L, &mp, nullptr, nullptr) != cudaSuccess) return QMM_ERR_CUDA;
    if (splits > 1) {
        ReduceParams rp;
        std::memset(&rp, 0, sizeof(rp));
        rp.partial = h.partial;
        rp.N = N;
        rp.M = M;
        rp.splits = splits;
        rp.banks = 1;
        rp.out_bf16 = out_dtype == QMM_OUT_BF16 ? 1 : 0;
        rp.out[0] = out;
        if (launch_reduce(rp, static_cast<int64_t>(M) * N, st) != cudaSuccess) return QMM_ERR_CUDA;
    }
    return QMM_OK;
}
