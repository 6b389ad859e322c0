"""Attention-sink stream (GPU) against the oracle: every token's attention
output, and the ring's Q/K/V contents after the stream (exactly the S + W
positions the oracle's sink + rolling cache holds, each at its ring slot)."""
import numpy as np
import pytest
import torch

import oracle as O
from denoising_step_kv_gb300 import _lib as K
from denoising_step_kv_gb300 import loop
from gpu_util import close, max_err, read_kv
from workloads import configs as C
from workloads import generate as G

pytestmark = pytest.mark.gpu


def _run(w, n_tokens=None, preproject=True):
    m = G.model(w)
    stream = G.stream_tokens(w)
    gen = loop.StreamGenerator(w, {k: loop.to_device(v) for k, v in m.items()}, preproject=preproject)
    try:
        gen.tok.copy_(torch.from_numpy(stream))
        out = gen.run(n_tokens).float().cpu().numpy()
        assert K.dllm_cache_check(gen.cache) == 0
        ring = [read_kv(gen.cache, f, 0, w)[0] for f in (K.FIELD_Q, K.FIELD_K, K.FIELD_V)]
    finally:
        gen.close()
    return m, stream, out, ring


def _slot(p, S, W):
    return p if p < S else S + (p - S) % W


@pytest.mark.parametrize("preproject", [True, False])
@pytest.mark.parametrize("name", ["tiny_sink_f32", "mid_sink"])
def test_stream_every_token(name, preproject):
    """Each token's row projected up front and copied into its slot, or
    projected by its own step."""
    w = C.get(name)
    m, stream, out, ring = _run(w, preproject=preproject)
    W64 = O.weights_f64(w, m)
    ref, held = O.run_stream(w, W64, stream)
    for n in range(w.stream_len):
        assert close(out[n], ref[n].reshape(-1), w), (name, n, max_err(out[n], ref[n].reshape(-1)))
    # ring contents after the last token: the held positions, each at its slot
    last = held[w.stream_len - 1]
    assert len(last) == w.sink + w.window
    pos = np.array(last)
    q, k, v = O.project_qkv(W64["embed"][stream[pos]], W64["w_qkv"][0], pos, w.n_heads, w.dtype,
                            w.rope_theta, w.rms_eps)
    slots = [_slot(p, w.sink, w.window) for p in last]
    assert sorted(slots) == list(range(w.sink + w.window))
    for got, want in zip(ring, (q, k, v)):
        want = O.round_store(want, w.dtype)
        assert close(got[slots], want, w), (name, max_err(got[slots], want))


def test_stream_prefix_before_wrap():
    """Tokens before the ring fills: the cache holds positions 0..n only."""
    w = C.get("mid_sink")
    n_tok = w.sink + 7
    m, stream, out, _ = _run(w, n_tok)
    ref, _ = O.run_stream(w, O.weights_f64(w, m), stream, n_tokens=n_tok)
    for n in range(n_tok):
        assert close(out[n], ref[n].reshape(-1), w), (n, max_err(out[n], ref[n].reshape(-1)))
    assert not np.any(out[n_tok:])


def test_sink_ring_full_size_sampled():
    """The 32768-token stream through S=4 + W=4092 at d=4096, 32 heads x 128:
    sampled tokens (first, around the first wrap, the last) against the
    oracle, which projects only the positions their caches hold."""
    w = C.get("sink_ring")
    m, stream, out, _ = _run(w)
    sample = [0, 3, 4, 4094, 4095, 4096, 4097, 8190, 32767]
    ref, held = O.run_stream(w, O.weights_f64(w, m), stream, sample=sample)
    for n in sample:
        assert len(held[n]) == min(n + 1, w.sink + w.window)
        assert close(out[n], ref[n].reshape(-1), w), (n, max_err(out[n], ref[n].reshape(-1)))


def test_stream_cache_ignores_block_len():
    """Streaming mode holds one history counter per sequence whatever
    block_len says: handle creation and reset clear only that, so a large
    block_len leaves every guard intact."""
    from dataclasses import replace
    w = replace(C.get("mid_sink"), block_len=1000)
    c = K.dllm_cache_init(K.make_cfg(w))
    try:
        assert K.dllm_cache_check(c) == 0
        K.dllm_cache_reset(c)
        assert K.dllm_cache_check(c) == 0
        assert K.state_size(c, K.FIELD_HIST_N) == 4 * w.batch
    finally:
        K.dllm_cache_free(c)
