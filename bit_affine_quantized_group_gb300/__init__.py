"""GB300 (sm_103a) group-wise affine-quantized multi-row matmul.

Thin ctypes binding of the C ABI in ``include/qmm.h`` (``libqmm.so`` in this
directory). It only marshals arguments: every step of the computation runs in
the library's CUDA kernels. PyTorch is used for device memory and streams.

    import bit_affine_quantized_group_gb300 as qmm
    plan = qmm.Plan(K=5120, N=17408, bits=4, group=32, max_M=16, out_dtype="bf16")
    qmm.forward(plan, x, w, s, b, out)        # tensors on the plan's device

The library is built by ``bit_affine_quantized_group_gb300._build`` (nvcc for
sm_103a). There is no fallback: if the library is missing, the first call
raises ImportError.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libqmm.so")

QMM_OK = 0
QMM_ERR_INVALID_ARG = 1
QMM_ERR_UNSUPPORTED = 2
QMM_ERR_PLAN_MISMATCH = 3
QMM_ERR_CUDA = 4
QMM_ERR_ALLOC = 5
QMM_ERR_TIMEOUT = 6
QMM_ERR_SCRATCH_LIMIT = 7
NOALLOC_SCRATCH_BYTES = 4 << 20
QMM_OUT_F32 = 0
QMM_OUT_BF16 = 1
MAX_ROWS = 16
MAX_BANKS = 64
MAX_SPLITS = 16

# Every entry point declared in include/qmm.h.
EXPORTS = (
    "qmm_validate_desc", "qmm_workspace_bytes", "qmm_plan", "qmm_plan_get_info",
    "qmm_check_forward_args", "qmm_forward", "qmm_forward_banked", "qmm_unpack_codes",
    "qmm_plan_error", "qmm_destroy", "qmm_status_string", "qmm_forward_noalloc", "qmm_forward_swiglu",
)


class QmmDesc(ctypes.Structure):
    _fields_ = [("K", ctypes.c_int64), ("N", ctypes.c_int64), ("bits", ctypes.c_int32),
                ("group", ctypes.c_int32), ("max_M", ctypes.c_int32), ("out_dtype", ctypes.c_int32),
                ("splits", ctypes.c_int32), ("max_banks", ctypes.c_int32)]


class QmmPlanInfo(ctypes.Structure):
    _fields_ = [("splits", ctypes.c_int32), ("chunks", ctypes.c_int32), ("stages", ctypes.c_int32 * 2),
                ("smem_bytes", ctypes.c_int32 * 2), ("num_sms", ctypes.c_int32), ("device", ctypes.c_int32),
                ("workspace_bytes", ctypes.c_int64)]


class QmmError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"qmm CUDA library not built ({LIB_PATH} missing); run "
                          "`python -m bit_affine_quantized_group_gb300._build` (needs nvcc, sm_103a)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    pp = ctypes.POINTER(ctypes.c_void_p)
    lib.qmm_validate_desc.argtypes = [ctypes.POINTER(QmmDesc)]
    lib.qmm_workspace_bytes.argtypes = [ctypes.POINTER(QmmDesc)]
    lib.qmm_workspace_bytes.restype = sz
    lib.qmm_plan.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(QmmDesc), vp, sz]
    lib.qmm_plan_get_info.argtypes = [vp, ctypes.POINTER(QmmPlanInfo)]
    lib.qmm_check_forward_args.argtypes = [ctypes.POINTER(QmmDesc), vp, i32, i32, pp, pp, pp, i64, i64, i32, i32, pp]
    lib.qmm_forward.argtypes = [vp, vp, i32, vp, vp, vp, i64, i64, i32, i32, vp, vp]
    lib.qmm_forward_banked.argtypes = [vp, vp, i32, i32, pp, pp, pp, i64, i64, i32, i32, pp, vp]
    lib.qmm_forward_swiglu.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp, vp, i64, i64, i32, i32, vp, vp]
    lib.qmm_unpack_codes.argtypes = [vp, i64, i64, i32, vp, vp]
    lib.qmm_forward_noalloc.argtypes = [vp, i32, vp, vp, vp, i64, i64, i32, i32, i32, vp, vp]
    lib.qmm_plan_error.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
    lib.qmm_destroy.argtypes = [vp]
    lib.qmm_destroy.restype = None
    lib.qmm_status_string.argtypes = [i32]
    lib.qmm_status_string.restype = ctypes.c_char_p
    for name in EXPORTS:
        if name not in ("qmm_workspace_bytes", "qmm_destroy", "qmm_status_string"):
            getattr(lib, name).restype = i32
    return lib


_LIB = None


def _lib() -> ctypes.CDLL:
    """The loaded libqmm.so (loaded on first use; ImportError if it was never built)."""
    global _LIB
    if _LIB is None:
        _LIB = _load()
    return _LIB


def __getattr__(name):
    if name == "lib":
        return _lib()
    raise AttributeError(name)


def status_string(status: int) -> str:
    return _lib().qmm_status_string(int(status)).decode()


def _out_code(out_dtype) -> int:
    if out_dtype in ("f32", "float32", QMM_OUT_F32):
        return QMM_OUT_F32
    if out_dtype in ("bf16", "bfloat16", QMM_OUT_BF16):
        return QMM_OUT_BF16
    try:
        import torch
        if out_dtype is torch.float32:
            return QMM_OUT_F32
        if out_dtype is torch.bfloat16:
            return QMM_OUT_BF16
    except ImportError:
        pass
    raise ValueError(f"unsupported out_dtype {out_dtype!r}")


def make_desc(K, N, bits, group, max_M=16, out_dtype="bf16", splits=0, max_banks=1) -> QmmDesc:
    return QmmDesc(int(K), int(N), int(bits), int(group), int(max_M), _out_code(out_dtype), int(splits),
                   int(max_banks))


def validate_desc(desc: QmmDesc) -> int:
    return int(_lib().qmm_validate_desc(ctypes.byref(desc)))


def workspace_bytes(desc: QmmDesc) -> int:
    return int(_lib().qmm_workspace_bytes(ctypes.byref(desc)))


def _stream_handle(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


class Plan:
    """A qmm plan (qmm_plan / qmm_destroy). By default its workspace is a
    PyTorch-allocated device buffer (so PyTorch's allocator owns the memory);
    pass ``torch_workspace=False`` to let the library cudaMalloc it."""

    def __init__(self, K, N, bits, group, max_M=16, out_dtype="bf16", splits=0, max_banks=1,
                 torch_workspace: bool = True, device=None):
        import torch
        self.desc = make_desc(K, N, bits, group, max_M, out_dtype, splits, max_banks)
        st = validate_desc(self.desc)
        if st != QMM_OK:
            raise QmmError(st, "qmm_validate_desc")
        self.K, self.N, self.bits, self.group = int(K), int(N), int(bits), int(group)
        self.max_M, self.max_banks = int(max_M), int(max_banks)
        self.out_dtype = torch.float32 if self.desc.out_dtype == QMM_OUT_F32 else torch.bfloat16
        self._handle = ctypes.c_void_p()
        self.workspace = None
        dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        with torch.cuda.device(dev):
            if torch_workspace:
                nbytes = workspace_bytes(self.desc)
                self.workspace = torch.empty(nbytes + 256, dtype=torch.uint8, device=dev)
                base = self.workspace.data_ptr()
                aligned = (base + 255) // 256 * 256
                st = _lib().qmm_plan(ctypes.byref(self._handle), ctypes.byref(self.desc), ctypes.c_void_p(aligned),
                                  ctypes.c_size_t(nbytes))
            else:
                st = _lib().qmm_plan(ctypes.byref(self._handle), ctypes.byref(self.desc), None, ctypes.c_size_t(0))
        if st != QMM_OK:
            raise QmmError(st, "qmm_plan")
        self.device = dev

    @property
    def handle(self):
        return self._handle

    def info(self) -> dict:
        inf = QmmPlanInfo()
        st = _lib().qmm_plan_get_info(self._handle, ctypes.byref(inf))
        if st != QMM_OK:
            raise QmmError(st, "qmm_plan_get_info")
        return {"splits": inf.splits, "chunks": inf.chunks, "stages": list(inf.stages),
                "smem_bytes": list(inf.smem_bytes), "num_sms": inf.num_sms, "device": inf.device,
                "workspace_bytes": inf.workspace_bytes}

    def error_flags(self) -> int:
        v = ctypes.c_uint32(0)
        st = _lib().qmm_plan_error(self._handle, ctypes.byref(v))
        if st not in (QMM_OK, QMM_ERR_TIMEOUT):
            raise QmmError(st, "qmm_plan_error")
        return int(v.value)

    def close(self):
        if self._handle is not None and self._handle.value:
            _lib().qmm_destroy(self._handle)
            self._handle = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _ptr(t) -> int:
    return int(t.data_ptr()) if t is not None else 0


def forward(plan: Plan, x, w, s, b, out, stream=None) -> None:
    """out[M, N] = qmm(x[M, K], w, s, b) via qmm_forward (asynchronous on `stream`)."""
    M = int(x.shape[0]) if x.dim() == 2 else 1
    st = _lib().qmm_forward(plan.handle, ctypes.c_void_p(_ptr(x)), M, ctypes.c_void_p(_ptr(w)),
                         ctypes.c_void_p(_ptr(s)), ctypes.c_void_p(_ptr(b)), plan.K, plan.N, plan.bits,
                         plan.group, ctypes.c_void_p(_ptr(out)), ctypes.c_void_p(_stream_handle(stream)))
    if st != QMM_OK:
        raise QmmError(st, "qmm_forward")


def _ptr_array(ts):
    arr = (ctypes.c_void_p * len(ts))()
    for i, t in enumerate(ts):
        arr[i] = _ptr(t)
    return arr


def forward_banked(plan: Plan, x, ws, ss, bs, outs, stream=None) -> None:
    """One launch for len(ws) projections sharing x (qmm_forward_banked)."""
    n = len(ws)
    M = int(x.shape[0]) if x.dim() == 2 else 1
    st = _lib().qmm_forward_banked(plan.handle, ctypes.c_void_p(_ptr(x)), M, n, _ptr_array(ws), _ptr_array(ss),
                                _ptr_array(bs), plan.K, plan.N, plan.bits, plan.group, _ptr_array(outs),
                                ctypes.c_void_p(_stream_handle(stream)))
    if st != QMM_OK:
        raise QmmError(st, "qmm_forward_banked")


def forward_swiglu(plan: Plan, x, w_gate, s_gate, b_gate, w_up, s_up, b_up, out, stream=None) -> None:
    """out[M, N] = silu(qmm(x, gate weights)) * qmm(x, up weights) in one main-kernel
    launch (qmm_forward_swiglu; the plan needs max_banks >= 2)."""
    M = int(x.shape[0]) if x.dim() == 2 else 1
    vp = ctypes.c_void_p
    st = _lib().qmm_forward_swiglu(plan.handle, vp(_ptr(x)), M, vp(_ptr(w_gate)), vp(_ptr(s_gate)),
                                   vp(_ptr(b_gate)), vp(_ptr(w_up)), vp(_ptr(s_up)), vp(_ptr(b_up)), plan.K,
                                   plan.N, plan.bits, plan.group, vp(_ptr(out)), vp(_stream_handle(stream)))
    if st != QMM_OK:
        raise QmmError(st, "qmm_forward_swiglu")


def check_forward_args(desc: QmmDesc, x_ptr: int, M: int, w_ptrs, s_ptrs, b_ptrs, K, N, bits, group,
                       out_ptrs) -> int:
    """Host-only argument check (qmm_check_forward_args); pointers are plain integers."""
    def arr(ps):
        if ps is None:
            return None
        a = (ctypes.c_void_p * len(ps))()
        for i, p in enumerate(ps):
            a[i] = p
        return a
    n = len(w_ptrs) if w_ptrs is not None else 1
    return int(_lib().qmm_check_forward_args(ctypes.byref(desc), ctypes.c_void_p(x_ptr), int(M), n, arr(w_ptrs),
                                          arr(s_ptrs), arr(b_ptrs), int(K), int(N), int(bits), int(group),
                                          arr(out_ptrs)))


def unpack_codes(w, K: int, N: int, bits: int, stream=None):
    """Run the kernels' in-register unpacking on packed words; returns uint8 [N, K]."""
    import torch
    codes = torch.empty((N, K), dtype=torch.uint8, device=w.device)
    st = _lib().qmm_unpack_codes(ctypes.c_void_p(_ptr(w)), int(K), int(N), int(bits), ctypes.c_void_p(_ptr(codes)),
                              ctypes.c_void_p(_stream_handle(stream)))
    if st != QMM_OK:
        raise QmmError(st, "qmm_unpack_codes")
    return codes
