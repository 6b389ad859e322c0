"""Helpers of the GPU tests: device tensors from generated arrays and reads
of the library's state through dllm_state_copy."""
import functools

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


def worst(a, b, w):
    """(count over tolerance, got, want) at the element farthest past it."""
    rtol, atol = tol(w)
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    ex = np.abs(a - b) - (atol + rtol * np.abs(b))
    i = np.unravel_index(np.argmax(ex), ex.shape)
    return int(np.sum(ex > 0)), float(a[i]), float(b[i]), tuple(int(x) for x in i)


def max_err(a, b):
    return float(np.max(np.abs(np.asarray(a) - np.asarray(b)))) if np.size(a) else 0.0


def kv_index(B, L, H, DH, esize):
    """Element index, in a layer's tiled Q/K/V cache, of the logical element
    [b, pos, h, e] (the layout include/dllm_kv.h documents for the Q/K/V
    fields: per (sequence, head) block of Lp rows, 64-row tiles of 128-byte
    sub-tile rows, 16-byte chunk c of row r at chunk c ^ (r % 8))."""
    Lp = -(-L // 64) * 64
    row_bytes = DH * esize
    b = np.arange(B)[:, None, None, None]
    pos = np.arange(L)[None, :, None, None]
    h = np.arange(H)[None, None, :, None]
    e = np.arange(DH)[None, None, None, :]
    per = 16 // esize
    chunk, within = e // per, (e % per) * esize
    sub, cc, r = chunk >> 3, chunk & 7, pos & 63
    off = ((b * H + h) * Lp + (pos & ~63)) * row_bytes + sub * 8192 + r * 128 + ((cc ^ (r & 7)) << 4) + within
    return off // esize


def _kv_shape(w):
    if w.streaming:
        return 1, w.sink + w.window
    return w.batch, w.seq_len


def read_kv(c, field, layer, w):
    """Q/K/V cache of a layer as [B, L, H, dh] float64 (streaming: [1, S+W, H, dh])."""
    B, L = _kv_shape(w)
    esize = 2 if w.dtype == "bf16" else 4
    n = K.state_size(c, field, layer) // esize
    flat = read_field(c, field, layer, (n,), "bf16" if w.dtype == "bf16" else "f32")
    return flat[kv_index(B, L, w.n_heads, w.head_dim, esize)]


def write_kv(c, field, layer, w, arr):
    """Write a [B, L, H, dh] array into a layer's tiled Q/K/V cache (zeros elsewhere)."""
    B, L = _kv_shape(w)
    esize = 2 if w.dtype == "bf16" else 4
    n = K.state_size(c, field, layer) // esize
    flat = np.zeros(n, dtype=np.float64)
    flat[kv_index(B, L, w.n_heads, w.head_dim, esize)] = np.asarray(arr, dtype=np.float64).reshape(B, L, w.n_heads, w.head_dim)
    write_field(c, field, layer, flat, "bf16" if w.dtype == "bf16" else "f32")


@functools.lru_cache(maxsize=8)
def _kv_idx(B, L, H, dh, esize, seqs):
    return torch.from_numpy(kv_index(B, L, H, dh, esize)[list(seqs)].reshape(-1))


def read_kv_seqs(c, field, layer, w, seqs):
    """Q/K/V of `layer` for the sequences `seqs` only, as [len(seqs), L, H,
    dh] float64 (one read of the whole field, then only those rows decoded)."""
    esize = 2 if w.dtype == "bf16" else 4
    n = K.state_size(c, field, layer) // esize
    host = torch.empty(n, dtype=torch.int16 if esize == 2 else torch.float32)
    K.dllm_state_copy(c, field, layer, host, False)
    vals = host[_kv_idx(w.batch, w.seq_len, w.n_heads, w.head_dim, esize, tuple(seqs))]
    vals = vals.view(torch.bfloat16) if esize == 2 else vals
    return vals.double().numpy().reshape(len(seqs), w.seq_len, w.n_heads, w.head_dim)
