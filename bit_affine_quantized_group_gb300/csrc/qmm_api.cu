// C ABI of the qmm library: descriptor validation, plans, and the forward
// dispatch. Declarations and the contract are in include/qmm.h.
#include <cuda_runtime.h>

#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <unordered_map>

#include "../../include/qmm.h"
#include "qmm_host.h"

using namespace qmmk;

static_assert(QMM_MAX_BANKS == kMaxBanks, "bank table size");
static_assert(QMM_MAX_SPLITS == kMaxSplits, "K-slice bound table size");

struct qmm_plan {
    qmm_desc d;
    int device;
    int num_sms;
    int optin;           // opt-in shared memory per CTA
    int splits;
    int C;
    int G;
    int stages[6];       // index 3 * (M > 8) + layout (kNarrow, kWide, kPair); 0: not usable
    int smem[6];
    uint8_t* ws;
    size_t ws_bytes;
    bool owns_ws;
    uint32_t* err;       // device error word (start of the workspace)
    float* partial;
    // TMA tensor maps already encoded for a given base pointer (weights, scales,
    // biases), for row blocks of kTN rows [0] and of the pair layout's rows [1]
    std::unordered_map<const void*, CUtensorMap> wmaps[2], smaps[2], bmaps[2];
};

namespace {

constexpr size_t kErrBytes = 256;

// Index into the plan's stages/smem of the main kernel that a call of M rows
// over rows_total flattened rows (banks x slices x N) launches; `single`: one
// projection.
int layout_index(const struct qmm_plan* p, int M, int64_t rows_total, bool single) {
    const int base = M > 8 ? 3 : 0;
    int64_t ctas = (rows_total + kSlab - 1) / kSlab;
    if (ctas > p->num_sms) ctas = p->num_sms;
    const int lay = consumer_layout(p->d.bits, p->d.group, M > 8 ? 16 : 8, rows_total, ctas, single, p->optin);
    return p->stages[base + lay] != 0 ? base + lay : base + kNarrow;
}

int chunks_of(const qmm_desc* d) {
    const int64_t G = d->K / d->group;
    return static_cast<int>((G + kGPC - 1) / kGPC);
}

// Largest K-slice count a plan for d may use (the automatic choice never exceeds it).
int splits_cap(const qmm_desc* d) {
    if (d->splits > 0) return d->splits;
    int c = chunks_of(d);
    if (c > 8) c = 8;
    return c;
}

int auto_splits(const qmm_desc* d, int num_sms) {
    return auto_split_count(d->K, d->N, d->bits, d->group, d->max_banks > 0 ? d->max_banks : 1, num_sms,
                            splits_cap(d));
}


size_t partial_region_bytes(const qmm_desc* d, int splits) {
    // unsliced plans with two or more banks keep room for the fused gate/up
    // projection's fp32 gate results ([max_M][N])
    if (splits <= 1) return d->max_banks >= 2 ? static_cast<size_t>(d->max_M) * d->N * sizeof(float) : 0;
    return static_cast<size_t>(d->max_banks) * splits * d->max_M * static_cast<size_t>(d->N) * sizeof(float);
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Cached lookup; the cache is cleared when it grows past a few thousand pointers.
bool tensor_map_for(struct qmm_plan* p, std::unordered_map<const void*, CUtensorMap>& cache, const void* ptr, bool weights,
                    int rows, CUtensorMap* out) {
    auto it = cache.find(ptr);
    if (it != cache.end()) {
        *out = it->second;
        return true;
    }
    CUtensorMap m;
    if (!(weights ? encode_weight_map(ptr, p->d.K, p->d.N, p->d.bits, p->d.group, rows, &m)
                  : encode_sb_map(ptr, p->G, p->d.N, rows, &m)))
        return false;
    if (cache.size() >= 4096) cache.clear();
    cache.emplace(ptr, m);
    *out = m;
    return true;
}

}  // namespace

extern "C" {

const char* qmm_status_string(int status) {
    switch (status) {
        case QMM_OK: return "QMM_OK";
        case QMM_ERR_INVALID_ARG: return "QMM_ERR_INVALID_ARG: invalid argument";
        case QMM_ERR_UNSUPPORTED: return "QMM_ERR_UNSUPPORTED: format or shape not supported";
        case QMM_ERR_PLAN_MISMATCH: return "QMM_ERR_PLAN_MISMATCH: K/N/bits/group differ from the plan";
        case QMM_ERR_CUDA: return "QMM_ERR_CUDA: CUDA runtime error";
        case QMM_ERR_ALLOC: return "QMM_ERR_ALLOC: allocation failed";
        case QMM_ERR_TIMEOUT: return "QMM_ERR_TIMEOUT: a kernel gave up a bounded wait";
        case QMM_ERR_SCRATCH_LIMIT: return "QMM_ERR_SCRATCH_LIMIT: the call needs more than the static scratch";
        default: return "unknown qmm status";
    }
}

int qmm_validate_desc(const qmm_desc* d) {
    if (d == nullptr) return QMM_ERR_INVALID_ARG;
    if (d->K <= 0 || d->N <= 0 || d->group <= 0 || d->bits <= 0) return QMM_ERR_INVALID_ARG;
    if (d->K > (1LL << 24) || d->N > (1LL << 30)) return QMM_ERR_INVALID_ARG;
    if (d->K % d->group != 0) return QMM_ERR_INVALID_ARG;
    if (d->max_M < 1 || d->max_M > QMM_MAX_ROWS) return QMM_ERR_INVALID_ARG;
    if (d->out_dtype != QMM_OUT_F32 && d->out_dtype != QMM_OUT_BF16) return QMM_ERR_INVALID_ARG;
    if (d->splits < 0 || d->splits > QMM_MAX_SPLITS) return QMM_ERR_INVALID_ARG;
    if (d->max_banks < 1 || d->max_banks > QMM_MAX_BANKS) return QMM_ERR_INVALID_ARG;
    if (d->bits < 2 || d->bits > 8 || d->bits == 7) return QMM_ERR_UNSUPPORTED;
    if (d->group != 32 && d->group != 64) return QMM_ERR_UNSUPPORTED;
    if ((d->K * d->bits) % 128 != 0) return QMM_ERR_UNSUPPORTED;
    if ((d->K / d->group) % 2 != 0) return QMM_ERR_UNSUPPORTED;
    if (d->splits > chunks_of(d)) return QMM_ERR_UNSUPPORTED;
    return QMM_OK;
}

size_t qmm_workspace_bytes(const qmm_desc* d) {
    if (qmm_validate_desc(d) != QMM_OK) return 0;
    return kErrBytes + partial_region_bytes(d, splits_cap(d));
}

int qmm_plan(qmm_plan_t** plan, const qmm_desc* d, void* workspace, size_t ws_bytes) {
    if (plan == nullptr) return QMM_ERR_INVALID_ARG;
    *plan = nullptr;
    const int v = qmm_validate_desc(d);
    if (v != QMM_OK) return v;
    const size_t need = qmm_workspace_bytes(d);
    if (workspace != nullptr && (ws_bytes < need || !aligned(workspace, 256))) return QMM_ERR_INVALID_ARG;

    int dev = 0, sms = 0, optin = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return QMM_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return QMM_ERR_CUDA;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return QMM_ERR_CUDA;

    struct qmm_plan* p = new (std::nothrow) struct qmm_plan();
    if (p == nullptr) return QMM_ERR_ALLOC;
    p->d = *d;
    p->device = dev;
    p->num_sms = sms;
    p->C = chunks_of(d);
    p->G = static_cast<int>(d->K / d->group);
    p->splits = d->splits > 0 ? d->splits : auto_splits(d, sms);
    if (p->splits > splits_cap(d)) p->splits = splits_cap(d);

    p->optin = optin;
    for (int i = 0; i < 6; ++i) {
        p->stages[i] = 0;
        p->smem[i] = 0;
    }
    for (int i = 0; i < 6; ++i) {
        const int mb = i >= 3 ? 16 : 8;
        const int lay = i % 3;
        if (mb == 16 && d->max_M <= 8) continue;
        const int st = stages_for(d->bits, d->group, mb, lay, optin);
        if (st < 2) {
            if (lay != kNarrow) continue;   // the narrow layout serves every call
            delete p;
            return QMM_ERR_UNSUPPORTED;
        }
        p->stages[i] = st;
        p->smem[i] = main_smem_bytes(d->bits, d->group, mb, lay);
        if (configure_format(d->bits, d->group, mb, lay, p->smem[i]) != cudaSuccess) {
            delete p;
            return QMM_ERR_CUDA;
        }
    }

    if (workspace == nullptr) {
        void* ws = nullptr;
        if (cudaMalloc(&ws, need) != cudaSuccess) {
            delete p;
            return QMM_ERR_ALLOC;
        }
        p->ws = static_cast<uint8_t*>(ws);
        p->ws_bytes = need;
        p->owns_ws = true;
    } else {
        p->ws = static_cast<uint8_t*>(workspace);
        p->ws_bytes = ws_bytes;
        p->owns_ws = false;
    }
    p->err = reinterpret_cast<uint32_t*>(p->ws);
    p->partial = reinterpret_cast<float*>(p->ws + kErrBytes);
    if (cudaMemsetAsync(p->ws, 0, kErrBytes, 0) != cudaSuccess || cudaStreamSynchronize(0) != cudaSuccess) {
        if (p->owns_ws) cudaFree(p->ws);
        delete p;
        return QMM_ERR_CUDA;
    }
    *plan = p;
    return QMM_OK;
}

int qmm_plan_get_info(const qmm_plan_t* p, qmm_plan_info* info) {
    if (p == nullptr || info == nullptr) return QMM_ERR_INVALID_ARG;
    info->splits = p->splits;
    info->chunks = p->C;
    const int64_t rows = static_cast<int64_t>(p->splits) * p->d.N;
    const int l8 = layout_index(p, 1, rows, true);
    const int l16 = p->d.max_M > 8 ? layout_index(p, 16, rows, true) : 3;
    info->stages[0] = p->stages[l8];
    info->stages[1] = p->stages[l16];
    info->smem_bytes[0] = p->smem[l8];
    info->smem_bytes[1] = p->smem[l16];
    info->num_sms = p->num_sms;
    info->device = p->device;
    info->workspace_bytes = static_cast<int64_t>(p->ws_bytes);
    return QMM_OK;
}

int qmm_check_forward_args(const qmm_desc* d, const void* x_bf16, int M, int n_banks,
                           const uint32_t* const* packed_w, const uint16_t* const* scales_f16,
                           const uint16_t* const* biases_f16, int64_t K, int64_t N, int bits, int group,
                           void* const* out) {
    if (d == nullptr) return QMM_ERR_INVALID_ARG;
    if (K != d->K || N != d->N || bits != d->bits || group != d->group) return QMM_ERR_PLAN_MISMATCH;
    if (M < 0 || M > d->max_M) return QMM_ERR_INVALID_ARG;
    if (n_banks < 1 || n_banks > d->max_banks) return QMM_ERR_INVALID_ARG;
    if (packed_w == nullptr || scales_f16 == nullptr || biases_f16 == nullptr || out == nullptr)
        return QMM_ERR_INVALID_ARG;
    if (M == 0) return QMM_OK;
    if (x_bf16 == nullptr || !aligned(x_bf16, 16)) return QMM_ERR_INVALID_ARG;
    const size_t sb_align = ((d->K / d->group) % 8 == 0) ? 16 : 4;
    const size_t out_align = d->out_dtype == QMM_OUT_F32 ? 4 : 2;
    for (int i = 0; i < n_banks; ++i) {
        if (packed_w[i] == nullptr || !aligned(packed_w[i], 16)) return QMM_ERR_INVALID_ARG;
        if (scales_f16[i] == nullptr || !aligned(scales_f16[i], sb_align)) return QMM_ERR_INVALID_ARG;
        if (biases_f16[i] == nullptr || !aligned(biases_f16[i], sb_align)) return QMM_ERR_INVALID_ARG;
        if (out[i] == nullptr || !aligned(out[i], out_align)) return QMM_ERR_INVALID_ARG;
    }
    return QMM_OK;
}

namespace {

// Shared body of the banked and the fused gate/up entry points. With swiglu,
// n_banks is 2 (gate, up) and out[1] is the one output.
int forward_impl(const qmm_plan_t* p, const void* x_bf16, int M, int n_banks, const uint32_t* const* packed_w,
                 const uint16_t* const* scales_f16, const uint16_t* const* biases_f16, int64_t K, int64_t N,
                 int bits, int group, void* const* out, void* stream, bool swiglu) {
    if (p == nullptr) return QMM_ERR_INVALID_ARG;
    const int chk = qmm_check_forward_args(&p->d, x_bf16, M, n_banks, packed_w, scales_f16, biases_f16, K, N,
                                           bits, group, out);
    if (chk != QMM_OK) return chk;
    if (M == 0) return QMM_OK;

    const int64_t rows_total = static_cast<int64_t>(swiglu ? 1 : n_banks) * p->splits * N;
    const int mi = layout_index(p, M, rows_total, !swiglu && n_banks == 1);
    if (p->stages[mi] == 0) return QMM_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    struct qmm_plan* mp_plan = const_cast<struct qmm_plan*>(p);   // the tensor-map caches are plan-owned scratch

    MainHeader h;
    std::memset(&h, 0, sizeof(h));
    h.x = static_cast<const uint16_t*>(x_bf16);
    h.partial = p->partial;
    h.err = p->err;
    h.N = N;
    h.K = K;
    h.G = p->G;
    h.C = p->C;
    h.splits = p->splits;
    set_slice_bounds(h);
    h.M = M;
    h.out_mode = p->splits > 1 ? kOutPartial : (p->d.out_dtype == QMM_OUT_F32 ? kOutF32 : kOutBF16);
    h.sb_tma = (p->G % 8 == 0) ? 1 : 0;
    h.unpack_magic = kF16x2_1024;
    h.banks = n_banks;
    h.gate = swiglu ? p->partial : nullptr;
    h.rows_total = rows_total;

    int64_t ctas = (h.rows_total + kSlab - 1) / kSlab;
    if (ctas > p->num_sms) ctas = p->num_sms;
    LaunchCfg L;
    L.mb = mi >= 3 ? 16 : 8;
    L.lay = mi % 3;
    const int rows = consumer_rows(L.lay);           // weight and scale boxes: one row block
    const int mc = rows == kTN ? 0 : 1;
    L.ctas = static_cast<int>(ctas);
    L.smem = p->smem[mi];
    L.stream = st;

    CUtensorMap xmap;
    if (!encode_x_map(x_bf16, M, K, group, L.mb, &xmap)) return QMM_ERR_CUDA;
    auto fill = [&](auto& mp) -> bool {
        mp.h = h;
        mp.tmx = xmap;
        for (int i = 0; i < n_banks; ++i) {
            mp.bank[i].w = packed_w[i];
            mp.bank[i].s = scales_f16[i];
            mp.bank[i].b = biases_f16[i];
            mp.bank[i].out = out[i];
            if (!tensor_map_for(mp_plan, mp_plan->wmaps[mc], packed_w[i], true, rows, &mp.tmw[i])) return false;
            if (h.sb_tma) {
                if (!tensor_map_for(mp_plan, mp_plan->smaps[mc], scales_f16[i], false, rows, &mp.tms[i])) return false;
                if (!tensor_map_for(mp_plan, mp_plan->bmaps[mc], biases_f16[i], false, rows, &mp.tmb[i])) return false;
            }
        }
        return true;
    };
    cudaError_t le;
    if (swiglu) {
        MainParams<2> mp2;
        std::memset(&mp2, 0, sizeof(mp2));
        if (!fill(mp2)) return QMM_ERR_CUDA;
        le = launch_format(bits, group, L, nullptr, nullptr, &mp2);
    } else if (n_banks == 1) {
        MainParams<1> mp1;
        std::memset(&mp1, 0, sizeof(mp1));
        if (!fill(mp1)) return QMM_ERR_CUDA;
        le = launch_format(bits, group, L, &mp1, nullptr, nullptr);
    } else {
        static thread_local MainParams<kMaxBanks> mpb;   // 25 KB: kept off the stack
        std::memset(&mpb, 0, sizeof(mpb));
        if (!fill(mpb)) return QMM_ERR_CUDA;
        le = launch_format(bits, group, L, nullptr, &mpb, nullptr);
    }
    if (le != cudaSuccess) return QMM_ERR_CUDA;

    if (p->splits > 1) {
        ReduceParams rp;
        std::memset(&rp, 0, sizeof(rp));
        rp.partial = p->partial;
        rp.N = N;
        rp.M = M;
        rp.splits = p->splits;
        rp.banks = n_banks;
        rp.swiglu = swiglu ? 1 : 0;
        rp.out_bf16 = p->d.out_dtype == QMM_OUT_BF16 ? 1 : 0;
        for (int i = 0; i < n_banks; ++i) rp.out[i] = out[i];
        if (swiglu) rp.out[0] = out[1];
        if (launch_reduce(rp, static_cast<int64_t>(swiglu ? 1 : n_banks) * M * N, st) != cudaSuccess)
            return QMM_ERR_CUDA;
    }
    return QMM_OK;
}

}  // namespace

int qmm_forward_banked(const qmm_plan_t* p, const void* x_bf16, int M, int n_banks,
                       const uint32_t* const* packed_w, const uint16_t* const* scales_f16,
                       const uint16_t* const* biases_f16, int64_t K, int64_t N, int bits, int group,
                       void* const* out, void* stream) {
    return forward_impl(p, x_bf16, M, n_banks, packed_w, scales_f16, biases_f16, K, N, bits, group, out, stream,
                        false);
}

int qmm_forward_swiglu(const qmm_plan_t* p, const void* x_bf16, int M, const uint32_t* w_gate,
                       const uint16_t* s_gate, const uint16_t* b_gate, const uint32_t* w_up, const uint16_t* s_up,
                       const uint16_t* b_up, int64_t K, int64_t N, int bits, int group, void* out, void* stream) {
    if (p == nullptr) return QMM_ERR_INVALID_ARG;
    if (p->d.max_banks < 2) return QMM_ERR_INVALID_ARG;   // the gate results live in the bank workspace
    const uint32_t* w[2] = {w_gate, w_up};
    const uint16_t* sc[2] = {s_gate, s_up};
    const uint16_t* bi[2] = {b_gate, b_up};
    void* o[2] = {out, out};
    return forward_impl(p, x_bf16, M, 2, w, sc, bi, K, N, bits, group, o, stream, true);
}

int qmm_forward(const qmm_plan_t* p, const void* x_bf16, int M, const uint32_t* packed_w,
                const uint16_t* scales_f16, const uint16_t* biases_f16, int64_t K, int64_t N, int bits, int group,
                void* out, void* stream) {
    return qmm_forward_banked(p, x_bf16, M, 1, &packed_w, &scales_f16, &biases_f16, K, N, bits, group, &out,
                              stream);
}

int qmm_unpack_codes(const uint32_t* packed_w, int64_t K, int64_t N, int bits, uint8_t* codes, void* stream) {
    if (bits < 2 || bits > 8 || bits == 7) return QMM_ERR_UNSUPPORTED;
    if (K <= 0 || N < 0 || K % 32 != 0 || K > (1LL << 24)) return QMM_ERR_INVALID_ARG;
    if (N == 0) return QMM_OK;
    if (packed_w == nullptr || codes == nullptr || !aligned(packed_w, 4)) return QMM_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    switch (bits) {
        case 2: e = launch_unpack<2>(packed_w, K, N, codes, st); break;
        case 3: e = launch_unpack<3>(packed_w, K, N, codes, st); break;
        case 4: e = launch_unpack<4>(packed_w, K, N, codes, st); break;
        case 5: e = launch_unpack<5>(packed_w, K, N, codes, st); break;
        case 6: e = launch_unpack<6>(packed_w, K, N, codes, st); break;
        default: e = launch_unpack<8>(packed_w, K, N, codes, st); break;
    }
    return e == cudaSuccess ? QMM_OK : QMM_ERR_CUDA;
}

int qmm_plan_error(const qmm_plan_t* p, uint32_t* flags) {
    if (p == nullptr || flags == nullptr) return QMM_ERR_INVALID_ARG;
    uint32_t v = 0;
    if (cudaMemcpy(&v, p->err, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return QMM_ERR_CUDA;
    if (v != 0 && cudaMemset(p->err, 0, sizeof(v)) != cudaSuccess) return QMM_ERR_CUDA;
    *flags = v;
    return v == 0 ? QMM_OK : QMM_ERR_TIMEOUT;
}

void qmm_destroy(qmm_plan_t* p) {
    if (p == nullptr) return;
    if (p->owns_ws && p->ws != nullptr) cudaFree(p->ws);
    delete p;
}

}  // extern "C"
