"""Helpers of the GPU tests: device tensors from generated arrays and reads
of the library's state through dllm_state_copy."""
import numpy as np
import torch

from denoising_step_kv_gb300 import _lib as K
from denoising_step_kv_gb300.loop import to_device

BF16_RTOL, BF16_ATOL = 2e-2, 1e-3      # bf16 outputs and probabilities
F32_TOL = 1e-5                          # fp32 workload


def tol(w):
    return (BF16_RTOL, BF16_ATOL) if w.dtype == "bf16" else (F32_TOL, F32_TOL)


def to_f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def read_field(c, field, layer, shape, dtype):
    n = K.state_size(c, field, layer)
    if dtype == "bf16":
        host = torch.empty(n // 2, dtype=torch.int16)
        K.dllm_state_copy(c, field, layer, host, False)
        return host.view(torch.bfloat16).float().numpy().astype(np.float64).reshape(shape)
    tdt = {"f32": torch.float32, "i32": torch.int32, "u8": torch.uint8}[dtype]
    host = torch.empty(n // torch.empty(0, dtype=tdt).element_size(), dtype=tdt)
    K.dllm_state_copy(c, field, layer, host, False)
    out = host.numpy()
    return (out.astype(np.float64) if dtype == "f32" else out).reshape(shape)


def write_field(c, field, layer, arr, dtype):
    if dtype == "bf16":
        from workloads.generate import f32_to_bf16_bits
        host = torch.from_numpy(f32_to_bf16_bits(np.asarray(arr, np.float32)).view(np.int16).reshape(-1).copy())
    elif dtype == "f32":
        host = torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32).reshape(-1))
    elif dtype == "i32":
        host = torch.from_numpy(np.ascontiguousarray(arr, dtype=np.int32).reshape(-1))
    else:
        host = torch.from_numpy(np.ascontiguousarray(arr, dtype=np.uint8).reshape(-1))
    K.dllm_state_copy(c, field, layer, host, True)


def cache_fields(w):
    return "bf16" if w.dtype == "bf16" else "f32"


def close(a, b, w):
    rtol, atol = tol(w)
    return np.allclose(a, b, rtol=rtol, atol=atol)


def max_err(a, b):
    return float(np.max(np.abs(np.asarray(a) - np.asarray(b)))) if np.size(a) else 0.0
