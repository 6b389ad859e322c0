"""Oracle model arithmetic (fp64) for the cached denoising step.

Sources, cited by page title and section:
  [LaCache]  "LaCache: Exact Caching and Precision-Adaptive Inference for
             Diffusion Large Language Models" (gist.science summary), sections
             "Problem statement" and "Methodology 1. LSM": a semi-autoregressive
             masked denoiser whose token-level operators are embedding lookup,
             normalisation, QKV projection and RoPE, followed by bidirectional
             attention over the full context.
  [SWD]      "Stable Window Decoding" page (wmrh.cn/news/51151), section 3.1:
             softmax over the vocabulary, top-1 token and its probability.
  [FlashdLLM] "I/O-aware KV cache and self-verifying parallel decoding"
             (bjdmk.com.cn/news/5926815), section 3.1: per-position entropy of
             the output distribution, normalised by its maximum.

Readings where the pages are silent (each also listed in the design notes):
  * normalisation = RMSNorm without affine weights, eps 1e-6, before the QKV
    projection, before the LM head and before the FFN;
  * RoPE = rotate-half pairing (i, i + dh/2), angle pos * theta^(-2i/dh);
  * the mask id never wins: its logit is -inf, so softmax and entropy range
    over the other V-1 ids;
  * argmax ties go to the lowest index;
  * FFN = W2 . GELU(W1 . RMSNorm(h)) with exact (erf) GELU, no biases.
"""
import numpy as np
from scipy.special import erf as _erf


def bf16_bits_to_f64(u16):
    """bf16 bit patterns (uint16) -> float64 values (exact)."""
    u = np.asarray(u16, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def _round_bf16(x):
    """Round fp64 values to the nearest bf16 value (ties to even), as fp64.

    bf16 keeps 8 significant bits, so the fp64 significand (53 bits) is rounded
    at bit 45 of the IEEE-754 bit pattern.
    """
    x = np.ascontiguousarray(x, dtype=np.float64)
    u = x.view(np.uint64)
    drop = np.uint64(45)
    half = np.uint64(1) << np.uint64(44)
    odd = (u >> drop) & np.uint64(1)
    r = (u + (half - np.uint64(1)) + odd) & ~((np.uint64(1) << drop) - np.uint64(1))
    return r.view(np.float64)


def round_store(x, dtype):
    """The value the GPU path keeps when it stores ``x`` in ``dtype``."""
    if dtype == "bf16":
        return _round_bf16(x)
    if dtype == "f32":
        return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)
    raise ValueError(dtype)


def rms_scale(x, eps=1e-6):
    """1 / sqrt(mean(x^2) + eps) over the last axis (RMSNorm, no affine)."""
    x = np.asarray(x, dtype=np.float64)
    return 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)


def rope(x, pos, theta=10000.0):
    """Rotary position embedding applied after the projection ([LaCache] LSM:
    "QKV projection and RoPE" are token-level operators).

    x: [..., H, dh]; pos: integer array broadcastable to x.shape[:-2].
    Pair (i, i + dh/2) is rotated by angle pos * theta^(-2i/dh).
    """
    x = np.asarray(x, dtype=np.float64)
    dh = x.shape[-1]
    half = dh // 2
    inv_freq = theta ** (-(2.0 * np.arange(half, dtype=np.float64)) / dh)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * inv_freq        # [..., half]
    c = np.cos(ang)[..., None, :]                                       # [..., 1, half]
    s = np.sin(ang)[..., None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def project_qkv(x, w_qkv, pos, n_heads, dtype, theta=10000.0, eps=1e-6):
    """Token-level operators of one layer for a set of rows ([LaCache] LSM,
    "RoPECache": normalised hidden state after QKV projection and RoPE).

    x: [n, d] layer input rows; w_qkv: [3d, d]; pos: [n] positions.
    Returns (q, k, v), each [n, H, dh], rounded to the storage type.
    """
    x = np.asarray(x, dtype=np.float64)
    n, d = x.shape
    dh = d // n_heads
    y = (x * rms_scale(x, eps)) @ np.asarray(w_qkv, dtype=np.float64).T   # [n, 3d]
    q = y[:, :d].reshape(n, n_heads, dh)
    k = y[:, d:2 * d].reshape(n, n_heads, dh)
    v = y[:, 2 * d:].reshape(n, n_heads, dh)
    q = rope(q, pos, theta)
    k = rope(k, pos, theta)
    return round_store(q, dtype), round_store(k, dtype), round_store(v, dtype)


def attention(q, k, v):
    """Bidirectional attention, no causal mask ([LaCache] problem statement:
    tokens of a block are updated together using the full context).

    q: [nq, H, dh]; k, v: [nk, H, dh].  Returns O: [nq, H, dh] (fp64, unrounded).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    dh = q.shape[-1]
    s = np.einsum("qhd,khd->hqk", q, k) / np.sqrt(dh)
    s = s - s.max(axis=-1, keepdims=True)
    p = np.exp(s)
    p /= p.sum(axis=-1, keepdims=True)
    return np.einsum("hqk,khd->qhd", p, v)


def attention_partial(q, k, v):
    """Online-softmax state of queries q over the keys k, v ([LaCache] LSM,
    FACache: the running maximum m, the normaliser l and the unnormalised
    accumulator O~ of a FlashAttention pass over those keys).

    q: [nq, H, dh]; k, v: [nk, H, dh] (nk may be 0).  Returns
    (m [H, nq], l [H, nq], O~ [nq, H, dh]) with O~ = sum_k e^(s_k - m) v_k,
    l = sum_k e^(s_k - m), s = q.k / sqrt(dh); an empty key set gives
    m = -inf, l = 0, O~ = 0.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    nq, H, dh = q.shape
    if len(k) == 0:
        return np.full((H, nq), -np.inf), np.zeros((H, nq)), np.zeros((nq, H, dh))
    s = np.einsum("qhd,khd->hqk", q, k) / np.sqrt(dh)
    m = s.max(axis=-1)
    p = np.exp(s - m[..., None])
    return m, p.sum(axis=-1), np.einsum("hqk,khd->qhd", p, v)


def merge_partials(parts):
    """Combine online-softmax states of one set of queries over disjoint key
    sets into the attention output over their union:
    O = sum_i e^(m_i - M) O~_i / sum_i e^(m_i - M) l_i, M = max_i m_i."""
    M = np.max(np.stack([m for m, _, _ in parts]), axis=0)             # [H, nq]
    num = 0.0
    den = 0.0
    for m, l, o in parts:
        w = np.where(np.isneginf(m), 0.0, np.exp(m - np.where(np.isneginf(M), 0.0, M)))
        den = den + w * l
        num = num + np.transpose(w)[:, :, None] * o
    return num / np.transpose(den)[:, :, None]


def out_proj(o, w_o, x, dtype):
    """Residual stream after attention: h = x + O . W_o^T (O stored first)."""
    o = round_store(np.asarray(o, dtype=np.float64).reshape(len(x), -1), dtype)
    return round_store(np.asarray(x, dtype=np.float64) + o @ np.asarray(w_o, dtype=np.float64).T, dtype)


def gelu(x):
    """Exact GELU: x/2 * (1 + erf(x / sqrt 2))."""
    return 0.5 * x * (1.0 + _erf(x / np.sqrt(2.0)))


def ffn(h, w1, w2, dtype, eps=1e-6):
    """h + W2 . GELU(W1 . RMSNorm(h)); the GELU output is stored before W2."""
    h = np.asarray(h, dtype=np.float64)
    f = round_store(gelu((h * rms_scale(h, eps)) @ np.asarray(w1, dtype=np.float64).T), dtype)
    return round_store(h + f @ np.asarray(w2, dtype=np.float64).T, dtype)


def lm_head_conf(h, w_lm, mask_id, eps=1e-6):
    """Per row: argmax, top-1 probability and entropy of softmax(RMSNorm(h) W_lm^T)
    with the mask id excluded ([SWD] 3.1: top-1 token and its probability;
    [FlashdLLM] 3.1: entropy of the position's distribution).

    Returns (argmax int32 [n], p1 [n], entropy [n], margin [n]) where margin is
    the gap between the two largest logits.
    """
    h = np.asarray(h, dtype=np.float64)
    logits = (h * rms_scale(h, eps)) @ np.asarray(w_lm, dtype=np.float64).T   # [n, V]
    keep = np.ones(logits.shape[1], dtype=bool)
    keep[mask_id] = False
    lg = logits[:, keep]
    ids = np.nonzero(keep)[0]
    j = np.argmax(lg, axis=1)                       # first occurrence = lowest id
    m = lg[np.arange(len(lg)), j]
    z = lg - m[:, None]
    e = np.exp(z)
    S = e.sum(axis=1)
    A = (e * z).sum(axis=1)
    p1 = 1.0 / S
    ent = np.log(S) - A / S
    top2 = np.partition(lg, -2, axis=1)[:, -2] if lg.shape[1] > 1 else m
    return ids[j].astype(np.int32), p1, ent, m - top2
