"""GPU-test helpers: move seeded numpy inputs to the device, run the library
through the C ABI (via the ctypes binding), bring results back as float64."""
from __future__ import annotations

import numpy as np


def dev_tensors(inp, bank: int = 0, device: str = "cuda"):
    import torch
    x = torch.from_numpy(np.ascontiguousarray(inp.x).view(np.int16)).to(device).view(torch.bfloat16)
    w = torch.from_numpy(np.ascontiguousarray(inp.words[bank]).view(np.int32)).to(device)
    s = torch.from_numpy(np.ascontiguousarray(inp.scales[bank]).view(np.int16)).to(device).view(torch.float16)
    b = torch.from_numpy(np.ascontiguousarray(inp.biases[bank]).view(np.int16)).to(device).view(torch.float16)
    return x, w, s, b


def to_f64(t) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def run_forward(plan, x, w, s, b, M: int, out=None):
    import torch
    import bit_affine_quantized_group_gb300 as q
    if out is None:
        out = torch.empty((M, plan.N), dtype=plan.out_dtype, device=x.device)
    q.forward(plan, x[:M], w, s, b, out)
    torch.cuda.synchronize()
    return out


def check(y_gpu: np.ndarray, y_ref: np.ndarray, out_dtype: str):
    from tests._helpers import check_bf16, check_f32
    if out_dtype == "f32":
        return check_f32(y_gpu, y_ref)
    return check_bf16(y_gpu, y_ref)
