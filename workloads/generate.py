"""Seeded synthetic inputs shared by the CPU oracle and the GPU path.

Every array is drawn from ``numpy.random.default_rng([seed, stream_id])`` so a
matrix can be regenerated on its own.  Weights are N(0, 0.02) drawn in fp32; a
bf16 workload stores them as bf16 bit patterns (uint16, round-to-nearest-even of
the fp32 draw).  Tokens: the mask id is 0; prompt ids are uniform in [1, 255]
(tiny workload) or Zipf(1.1) ranks over ids 1..V-1, P(k) proportional to
k^-1.1; generation slots hold the mask id.

No arithmetic of the denoising method lives here: only random draws and their
storage encoding.
"""
import numpy as np

STD = 0.02

# stream ids: one independent generator per array
_S_EMBED, _S_LM, _S_TOK, _S_STREAM = 1, 2, 3, 4
_S_QKV, _S_O, _S_W1, _S_W2 = 10, 11, 12, 13   # + 16 * layer


def f32_to_bf16_bits(a):
    """fp32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def _rng(seed, sid):
    return np.random.default_rng([seed, sid])


def _normal(w, sid, shape, scale=1.0):
    x = _rng(w.seed, sid).standard_normal(size=shape, dtype=np.float32)
    x *= np.float32(STD * scale)
    if w.dtype == "bf16":
        return f32_to_bf16_bits(x)
    return x


def embed(w):
    """Embedding table [V][d]."""
    return _normal(w, _S_EMBED, (w.vocab, w.d_model))


def w_lm(w):
    """LM-head weight [V][d] (times the workload's lm_scale)."""
    return _normal(w, _S_LM, (w.vocab, w.d_model), w.lm_scale)


def w_qkv(w, layer=0):
    """Fused projection [3d][d]: rows [0,d) give q, [d,2d) k, [2d,3d) v."""
    return _normal(w, _S_QKV + 16 * layer, (3 * w.d_model, w.d_model))


def w_o(w, layer=0):
    """Attention output projection [d][d]."""
    return _normal(w, _S_O + 16 * layer, (w.d_model, w.d_model))


def w_ffn1(w, layer=0):
    return _normal(w, _S_W1 + 16 * layer, (w.ffn, w.d_model))


def w_ffn2(w, layer=0):
    return _normal(w, _S_W2 + 16 * layer, (w.d_model, w.ffn))


def _draw_ids(w, rng, n):
    if w.tokens == "uniform255":
        return rng.integers(1, 256, size=n, dtype=np.int64).astype(np.int32)
    ranks = np.arange(1, w.vocab, dtype=np.float64)
    p = ranks ** (-w.zipf_a)
    p /= p.sum()
    return (rng.choice(w.vocab - 1, size=n, p=p) + 1).astype(np.int32)


def prompt_tokens(w):
    """tok[B][L] int32: prompt ids followed by mask ids in the generation slots."""
    rng = _rng(w.seed, _S_TOK)
    tok = np.full((w.batch, w.seq_len), w.mask_id, dtype=np.int32)
    tok[:, :w.n_prompt] = _draw_ids(w, rng, w.batch * w.n_prompt).reshape(w.batch, w.n_prompt)
    return tok


def stream_tokens(w):
    """Token stream [stream_len] int32 for the attention-sink workload."""
    return _draw_ids(w, _rng(w.seed, _S_STREAM), w.stream_len)


def model(w):
    """All weights of a workload as a dict of arrays."""
    m = {"embed": embed(w)}
    if w.streaming:
        m["w_qkv"] = [w_qkv(w, 0)]
        return m
    m["w_lm"] = w_lm(w)
    m["w_qkv"] = [w_qkv(w, l) for l in range(w.n_layers)]
    m["w_o"] = [w_o(w, l) for l in range(w.n_layers)]
    if w.ffn:
        m["w1"] = [w_ffn1(w, l) for l in range(w.n_layers)]
        m["w2"] = [w_ffn2(w, l) for l in range(w.n_layers)]
    return m


# --- seeded inputs for single-kernel tests --------------------------------------------
def normal(seed, shape, std=1.0, dtype="bf16"):
    """N(0, std^2) array in the storage encoding of ``dtype`` (bf16 bits or fp32)."""
    x = np.random.default_rng([seed, 99]).standard_normal(size=shape, dtype=np.float32) * np.float32(std)
    return f32_to_bf16_bits(x) if dtype == "bf16" else x


def integers(seed, lo, hi, shape):
    """Uniform int32 in [lo, hi)."""
    return np.random.default_rng([seed, 98]).integers(lo, hi, size=shape).astype(np.int32)


def uniform(seed, lo, hi, shape):
    """Uniform fp32 in [lo, hi)."""
    return np.random.default_rng([seed, 97]).uniform(lo, hi, size=shape).astype(np.float32)


def choice(seed, n, k):
    """k distinct sorted ints from [0, n)."""
    return np.sort(np.random.default_rng([seed, 96]).choice(n, size=k, replace=False)).astype(np.int32)
