/*
 * qmm.h -- C ABI of the GB300 (sm_103a) group-wise affine-quantized
 * multi-row matmul.
 *
 * The operation (vmlx-swift PR #565 "Enable bundle-aware Qwen speculation and
 * dense mixed JANGH loading", LaneQMM commit: matmul over raw affine codes with
 * the dequant applied after the dot product, "C += s*P + b*XS"):
 *
 *   y[m,n] = sum_g ( s[n,g] * P[m,n,g] + b[n,g] * XS[m,g] )
 *   P[m,n,g] = sum_{k in g} x[m,k] * q[n,k]      XS[m,g] = sum_{k in g} x[m,k]
 *
 * which equals x . W^T with W[n,k] = s[n,k/group] * q[n,k] + b[n,k/group].
 * It serves decode (M = 1) and speculative-decoding verification (M = 2..16
 * rows; same page, LaneQMM and qwen_qmv_rows_full commits: weight words, scales
 * and biases are read once for all rows).
 *
 * Data layout (all row-major, all owned by the caller):
 *   x       [M, K]          bfloat16 activations
 *   w       [N, K*bits/32]  uint32 words; row n holds q[n, 0..K-1] as an
 *                           LSB-first bit stream: bit j of code k is bit
 *                           (k*bits + j) mod 32 of word (k*bits + j) / 32.
 *                           5- and 6-bit codes may straddle two words.
 *   scales  [N, K/group]    IEEE binary16
 *   biases  [N, K/group]    IEEE binary16
 *   out     [M, N]          float32 or bfloat16 (round to nearest even),
 *                           overwritten (never accumulated into).
 *
 * Supported formats: bits in {2, 3, 4, 5, 6, 8}, group in {32, 64}, 1 <= M <= 16.
 * (2-bit tensors are in use beside 4/8-bit ones per "Qwen3.8 Flash Next
 * performance and parity receipt", MTPLX logic review, and the "JANGH split-K
 * verify tile" commit tests 2/4/8-bit codes; 3-bit follows the same stream.)
 * Requirements checked before any launch: K % group == 0; K*bits % 128 == 0
 * (every packed row starts on a 16-byte boundary); K/group even (so K is a
 * multiple of 64); x, packed weights, scales and biases 16-byte aligned
 * device pointers (x is read with tensor-memory-access copies); out a
 * naturally aligned device pointer.
 *
 * Split-K (same page, commit "JANGH split-K verify tile": K is sliced across
 * the grid, FP32 partials are written and then summed): with splits S > 1 the
 * K range is cut into S slices on 8-group chunk boundaries (uneven slices
 * allowed), each slice writes float32 partials into the plan's workspace and a
 * second kernel sums them in slice order 0..S-1, so results are deterministic
 * run to run but not bitwise equal to S = 1 (the page's contract: not
 * bitwise, covered by tolerance tests).
 *
 * Banked mode (same page, qwen_qmv_rows_full commit: 36 projection banks in
 * one dispatch) runs several projections that share x in one launch.
 *
 * Conventions:
 *   - Every function returns a qmm_status (0 = QMM_OK) and never throws.
 *   - qmm_forward / qmm_forward_banked / qmm_forward_swiglu are asynchronous on `stream` (a
 *     cudaStream_t passed as void*, NULL = legacy default stream); they never
 *     allocate and never synchronize. Errors in arguments are reported before
 *     anything is launched. Launch failures return QMM_ERR_CUDA.
 *   - A plan (and its workspace) must be used by one stream at a time.
 *   - All device pointers must stay valid until the stream work completes.
 */
#ifndef QMM_H
#define QMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
enum {
    QMM_OK = 0,
    QMM_ERR_INVALID_ARG = 1,   /* NULL/misaligned pointer, out-of-range value */
    QMM_ERR_UNSUPPORTED = 2,   /* well-formed request this library does not implement */
    QMM_ERR_PLAN_MISMATCH = 3, /* K/N/bits/group differ from the plan's */
    QMM_ERR_CUDA = 4,          /* a CUDA runtime call failed (no device, launch error) */
    QMM_ERR_ALLOC = 5,         /* host or device allocation failed in qmm_plan */
    QMM_ERR_TIMEOUT = 6,       /* a kernel gave up a bounded wait (qmm_plan_error) */
    QMM_ERR_SCRATCH_LIMIT = 7  /* reserved (no longer returned: qmm_forward_noalloc lowers its K slices to fit) */
};

/* Output element types. */
enum { QMM_OUT_F32 = 0, QMM_OUT_BF16 = 1 };

#define QMM_MAX_ROWS 16
#define QMM_MAX_BANKS 64
#define QMM_MAX_SPLITS 16

/* Problem descriptor fixed at plan time. */
typedef struct qmm_desc {
    int64_t K;          /* reduction length (codes per weight row) */
    int64_t N;          /* output columns (weight rows) */
    int32_t bits;       /* code width: 2, 3, 4, 5, 6 or 8 */
    int32_t group;      /* codes per scale/bias group: 32 or 64 */
    int32_t max_M;      /* largest M forward will be called with, 1..16 */
    int32_t out_dtype;  /* QMM_OUT_F32 or QMM_OUT_BF16 */
    int32_t splits;     /* 0 = choose automatically, else 1..16 K slices */
    int32_t max_banks;  /* largest n_banks for qmm_forward_banked, 1..64 */
} qmm_desc;

/* What a plan decided (for reporting and tests). */
typedef struct qmm_plan_info {
    int32_t splits;          /* K slices used by every forward call */
    int32_t chunks;          /* 8-group chunks along K */
    int32_t stages[2];       /* weight-pipeline depth of the main kernel a single-projection call
                                of M <= 8 rows uses, and of the one for 9 <= M <= 16 */
    int32_t smem_bytes[2];   /* dynamic shared memory per CTA, same order */
    int32_t num_sms;         /* streaming multiprocessors on the plan's device */
    int32_t device;          /* CUDA device ordinal the plan was made on */
    int64_t workspace_bytes; /* device workspace the plan uses */
} qmm_plan_info;

typedef struct qmm_plan qmm_plan_t;

/*
 * Validate a descriptor on the host (no CUDA call). Returns QMM_OK,
 * QMM_ERR_INVALID_ARG (malformed: NULL, K % group != 0, out-of-range
 * max_M/out_dtype/splits/max_banks) or QMM_ERR_UNSUPPORTED (well formed but
 * outside this library: other bit widths or group sizes, K*bits % 128 != 0,
 * K/group odd, splits greater than the number of 8-group chunks).
 */
int qmm_validate_desc(const qmm_desc* d);

/*
 * Device workspace a plan for `d` needs (bytes; 0 if d is invalid): a
 * 256-byte error word plus split-K partials for max_banks * splits * max_M * N
 * floats (splits = 0 is sized for the largest automatic choice,
 * min(8, chunks) with chunks = ceil(K / group / 8)). Lets the caller
 * (e.g. PyTorch's allocator) own it.
 */
size_t qmm_workspace_bytes(const qmm_desc* d);

/*
 * Create a plan on the current CUDA device. Validates `d`, queries the device
 * (SM count, shared memory), picks splits when d->splits == 0, and configures
 * the kernels. If `workspace` is NULL the plan cudaMallocs its own workspace of
 * qmm_workspace_bytes(d) bytes (freed by qmm_destroy); otherwise `workspace`
 * must be a device pointer, 256-byte aligned, of at least ws_bytes >=
 * qmm_workspace_bytes(d) bytes, owned by the caller and not used by anything
 * else while the plan is in use. On failure *plan is set to NULL.
 */
int qmm_plan(qmm_plan_t** plan, const qmm_desc* d, void* workspace, size_t ws_bytes);

/* Copy out what the plan decided. */
int qmm_plan_get_info(const qmm_plan_t* p, qmm_plan_info* info);

/*
 * Host-only check of forward arguments against a descriptor, exactly as
 * qmm_forward_banked performs it before launching (n_banks arrays of device
 * pointers; qmm_forward is the n_banks == 1 case). No CUDA call. Returns
 * QMM_OK, QMM_ERR_INVALID_ARG (NULL or misaligned pointer, M < 0,
 * M > max_M, n_banks out of range) or QMM_ERR_PLAN_MISMATCH.
 */
int qmm_check_forward_args(const qmm_desc* d, const void* x_bf16, int M, int n_banks,
                           const uint32_t* const* packed_w, const uint16_t* const* scales_f16,
                           const uint16_t* const* biases_f16, int64_t K, int64_t N, int bits,
                           int group, void* const* out);

/*
 * y = qmm(x, w, scales, biases) for one projection. M = 0 is a no-op that
 * returns QMM_OK. K, N, bits and group must equal the plan's
 * (QMM_ERR_PLAN_MISMATCH otherwise); M must be <= the plan's max_M.
 * Launches, in stream order: the main kernel (it streams the weights, stages
 * the activations and computes the projection) and, when the plan's
 * splits > 1, the split-K reduce kernel.
 *
 * Ordering: x is read only after the work issued before the call on the
 * stream has finished, and out is written after that too. The packed weights,
 * scales and biases are streamed from the start (programmatic dependent
 * launch), possibly while that earlier work still runs: they must not be
 * written by work issued just before the call (weights are normally written
 * once, at load time; synchronize the stream or record/wait an event in
 * between otherwise). The same holds for every forward entry point.
 */
int qmm_forward(const qmm_plan_t* p, const void* x_bf16, int M, const uint32_t* packed_w,
                const uint16_t* scales_f16, const uint16_t* biases_f16, int64_t K, int64_t N,
                int bits, int group, void* out, void* stream);

/*
 * n_banks projections of the same shape and format that share x, in one
 * launch of the main kernel. packed_w, scales_f16, biases_f16 and out are HOST
 * arrays of n_banks device pointers (copied into the kernel parameters; the
 * arrays may be reused as soon as the call returns). 1 <= n_banks <= the
 * plan's max_banks (<= 64). Each bank's result equals qmm_forward on that bank
 * with the same plan.
 */
int qmm_forward_banked(const qmm_plan_t* p, const void* x_bf16, int M, int n_banks,
                       const uint32_t* const* packed_w, const uint16_t* const* scales_f16,
                       const uint16_t* const* biases_f16, int64_t K, int64_t N, int bits,
                       int group, void* const* out, void* stream);

/*
 * Fused gate/up projection with a SwiGLU epilogue ("Qwen3.8 Flash Next
 * performance and parity receipt": the exact fused projection promoted over
 * separate gate and up projections):
 *   out[m, n] = silu(gate[m, n]) * up[m, n],   silu(g) = g / (1 + exp(-g)),
 * where gate and up are the qmm_forward results of (w_gate, s_gate, b_gate)
 * and (w_up, s_up, b_up) on the same x, both N x K in the plan's format. One
 * launch of the main kernel computes both: every CTA runs each of its row
 * blocks for the gate and then for the up weights, keeping the fp32 gate
 * values in the plan's workspace. The plan must have max_banks >= 2 (else
 * QMM_ERR_INVALID_ARG). With splits > 1 both projections write fp32 slice
 * partials and the reduce kernel applies the epilogue to the slice sums.
 * Pointers and argument checks as for qmm_forward; out is [M, N] in the
 * plan's output type.
 */
int qmm_forward_swiglu(const qmm_plan_t* p, const void* x_bf16, int M, const uint32_t* w_gate,
                       const uint16_t* s_gate, const uint16_t* b_gate, const uint32_t* w_up,
                       const uint16_t* s_up, const uint16_t* b_up, int64_t K, int64_t N, int bits,
                       int group, void* out, void* stream);

/*
 * Diagnostic: run the main kernel's in-register code unpacking on packed
 * weights and write the decoded codes, codes[n*K + k] = q[n,k] (uint8, device
 * pointer, N*K bytes). A code whose unpacked binary16 image is not the exact
 * value 1024 + q * 2^j (j the code's mantissa shift) is written as 0xFF.
 * Asynchronous on `stream`.
 */
int qmm_unpack_codes(const uint32_t* packed_w, int64_t K, int64_t N, int bits, uint8_t* codes,
                     void* stream);

/*
 * Read (synchronously) and clear the plan's device error word. Sets *flags to
 * 0 when every kernel since the last call finished normally; nonzero when a
 * kernel gave up a bounded wait (its output is then incomplete) and returns
 * QMM_ERR_TIMEOUT in that case.
 */
int qmm_plan_error(const qmm_plan_t* p, uint32_t* flags);

/*
 * Size of the device scratch qmm_forward_noalloc keeps in a static device
 * array (held by every GPU that loads this library until the process exits).
 */
#define QMM_NOALLOC_SCRATCH_BYTES (4u << 20)

/*
 * qmm_forward without a plan and without any allocation, for callers that
 * cannot call cudaMalloc when they run a projection (code that runs while
 * another component owns the device allocator, loops that forbid allocation
 * after start-up, plug-in hosts that only hand over their tensors). The pages
 * describe no counterpart: this is a deployment variant of qmm_forward.
 *
 * Same arguments, data layout and kernels as qmm_forward, with the output
 * type given directly (QMM_OUT_F32 or QMM_OUT_BF16). The device scratch that
 * qmm_forward keeps in its plan's workspace (the kernels' error word and the
 * fp32 partial sums of K slices) lives in a static device array of
 * QMM_NOALLOC_SCRATCH_BYTES. The K-slice count is the one an automatic plan
 * would choose, lowered until 256 + slices * M * N * 4 bytes fit the array
 * (one slice needs no partials), so every supported shape runs; results are
 * bitwise those of qmm_forward with a plan of that slice count. Nothing is
 * allocated: no cudaMalloc, no cudaFree, no allocating library routine.
 *
 * The first call on a device (with that device current) looks up the
 * scratch's device address and sets the kernels' shared-memory limit; make
 * that first call before any stream capture. Every call on a device shares the
 * one scratch array and overwrites it, so calls whose executions overlap on
 * the GPU (different streams, or concurrent host threads) race: serialize
 * them. Device-side timeouts are recorded only in the scratch and not
 * reported; use qmm_forward for that.
 */
int qmm_forward_noalloc(const void* x_bf16, int M, const uint32_t* packed_w, const uint16_t* scales_f16,
                        const uint16_t* biases_f16, int64_t K, int64_t N, int bits, int group, int out_dtype,
                        void* out, void* stream);

/* Free the plan and any workspace it allocated. NULL is accepted. */
void qmm_destroy(qmm_plan_t* p);

/* Static description of a status code; never NULL. */
const char* qmm_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* QMM_H */
