"""The attention with the kept softmax state of the unchanged key tiles
(GPU, "LaCache" FACache) against the oracle: the kernel on written caches
(rebuild, reuse, a changed query token, a changed window row), whole
generations of the single-layer workloads, and the 8B-shaped layer's first
block sampled."""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle as O
from denoising_step_kv_gb300 import _lib as K
from denoising_step_kv_gb300 import loop
from gpu_util import close, i32, read_field, tol, worst, write_field, write_kv
from workloads import configs as C
from workloads import generate as G

pytestmark = pytest.mark.gpu


def _rebuilt(c):
    return int(read_field(c, K.FIELD_FA_REBUILT, 0, (1,), "i32")[0])


@pytest.mark.parametrize("name", ["mid_bf16", "mid_bf16_dh64", "big_rows"])
def test_facache_kernel_rebuild_reuse_and_invalidation(name):
    w = C.get(name)
    B, L, H, dh, d, blk, q0 = w.batch, w.seq_len, w.n_heads, w.head_dim, w.d_model, w.block_len, w.n_prompt
    rnd = lambda s: O.round_store(G.normal(s, (B, L, H, dh), 1.0, "f32").astype(np.float64), w.dtype)
    q, k, v = rnd(61), rnd(62), rnd(63)
    tok_w = G.integers(64, 1, w.vocab, (B, L))
    c = K.dllm_cache_init(K.make_cfg(w, facache=True))

    def run():
        out = torch.zeros(B * blk, d, dtype=torch.bfloat16, device="cuda")
        K.block_attn(c, 0, q0, blk, out)
        assert K.dllm_cache_check(c) == 0
        return out.float().cpu().numpy().astype(np.float64).reshape(B, blk, d)

    def want(qq, kk, vv):
        return np.stack([O.round_store(O.attention(qq[b, q0:q0 + blk], kk[b], vv[b]).reshape(blk, d), w.dtype)
                         for b in range(B)])

    try:
        for f, a in ((K.FIELD_Q, q), (K.FIELD_K, k), (K.FIELD_V, v)):
            write_kv(c, f, 0, w, a)
        write_field(c, K.FIELD_TOK_W, 0, tok_w, "i32")
        o1 = run()                                      # first call: every state rebuilt
        assert close(o1, want(q, k, v), w), worst(o1, want(q, k, v), w)
        assert _rebuilt(c) == B * H
        o2 = run()                                      # same key: window tiles only, merged with the state
        assert close(o2, want(q, k, v), w), worst(o2, want(q, k, v), w)
        assert _rebuilt(c) == B * H
        # a new value in a window row is read (the window is streamed every call)
        k2, v2 = k.copy(), v.copy()
        r = min(L - 1, q0 + blk)                       # inside [q0 - R, q0 + blk + R)
        k2[:, r] = rnd(65)[:, r]
        v2[:, r] = rnd(66)[:, r]
        write_kv(c, K.FIELD_K, 0, w, k2)
        write_kv(c, K.FIELD_V, 0, w, v2)
        o3 = run()
        assert close(o3, want(q, k2, v2), w), worst(o3, want(q, k2, v2), w)
        assert _rebuilt(c) == B * H
        # a changed query token in sequence B-1 (with its new Q) rebuilds that sequence only
        q3 = q.copy()
        q3[B - 1, q0 + 1] = rnd(67)[B - 1, q0 + 1]
        tok3 = tok_w.copy()
        tok3[B - 1, q0 + 1] += 1
        write_kv(c, K.FIELD_Q, 0, w, q3)
        write_field(c, K.FIELD_TOK_W, 0, tok3, "i32")
        o4 = run()
        assert close(o4, want(q3, k2, v2), w), worst(o4, want(q3, k2, v2), w)
        assert _rebuilt(c) == B * H + H
        # a reset forgets every state
        K.dllm_cache_reset(c)
        for f, a in ((K.FIELD_Q, q3), (K.FIELD_K, k2), (K.FIELD_V, v2)):
            write_kv(c, f, 0, w, a)
        write_field(c, K.FIELD_TOK_W, 0, tok3, "i32")
        o5 = run()
        assert close(o5, want(q3, k2, v2), w)
        assert _rebuilt(c) == B * H
    finally:
        K.dllm_cache_free(c)


def _ambiguous(rec, w):
    amb = rec["margin"] <= 1e-2
    for b in range(w.batch):
        for j in range(w.block_len):
            ps = rec["swd"].p[b][j]
            if len(ps) == w.swd_K and abs(float(np.mean(ps)) - w.swd_tau) < 1e-3:
                amb[b, j] = True
    return amb


@pytest.mark.parametrize("name", ["mid_bf16", "mid_bf16_dh64", "mid_bf16_sharp", "big_rows"])
def test_facache_generation(name):
    """A whole generation with the kept state against the oracle's FACache
    loop (equal to its plain loop, pinned): outputs, confidences and the
    trajectory until an ambiguous position; the device's rebuild count
    equals the oracle's rebuilds times the heads."""
    w = C.get(name)
    m = G.model(w)
    tok0 = G.prompt_tokens(w)
    trace = O.run_dense(w, O.weights_f64(w, m), tok0, facache=True)
    gen = loop.DenseGenerator(w, {k: loop.to_device(v) for k, v in m.items()}, facache=True)
    B, L, blk, d = w.batch, w.seq_len, w.block_len, w.d_model
    got = []

    def grab(t, q0, s):
        got.append(dict(argmax=gen.argmax.cpu().numpy().reshape(B, blk), p1=gen.p1.cpu().numpy().reshape(B, blk),
                        ent=gen.ent.cpu().numpy().reshape(B, blk), tok=gen.tok.cpu().numpy().copy(),
                        o=gen.o.float().cpu().numpy().reshape(B, blk, d), rebuilt=_rebuilt(gen.cache),
                        rows=gen.rows.cpu().numpy()[:int(gen.n_rows.item())].copy()))

    gen.tok_in.copy_(torch.from_numpy(tok0))
    try:
        gen.run(on_step=grab)
        assert K.dllm_cache_check(gen.cache) == 0
    finally:
        gen.close()
    rtol, atol = tol(w)
    compared, n_rebuilt = 0, 0
    for rec, g in zip(trace, got):
        t = rec["t"]
        assert close(g["o"], rec["o"], w), (name, t, "o", worst(g["o"], rec["o"], w))
        assert np.allclose(g["p1"], rec["p1"], rtol=rtol, atol=atol), (name, t, "p1")
        assert np.allclose(g["ent"], rec["ent"], rtol=rtol, atol=atol), (name, t, "ent")
        amb = _ambiguous(rec, w)
        assert np.array_equal(g["argmax"][~amb], rec["argmax"][~amb]), (name, t, "argmax")
        if np.any(g["argmax"][amb] != rec["argmax"][amb]):
            break
        n_rebuilt += len(rec["fa_rebuilt"]) * w.n_heads
        assert g["rebuilt"] == n_rebuilt, (name, t, "rebuilds", g["rebuilt"], n_rebuilt)
        assert np.array_equal(g["tok"], rec["tok"]), (name, t, "tok")
        assert np.array_equal(g["rows"], rec["rows_next"]), (name, t, "rows")
        compared += 1
    assert compared >= 1 or np.any(trace[0]["margin"] <= 1e-2), (name, compared)


def test_facache_8b_shaped_first_block_sampled():
    """The 8B-shaped layer at full batch for its first block (32 steps, the
    state rebuilt once per sequence and head, then reused): every step's
    attention output and confidences of sequences 2 and 6 against the oracle
    on the GPU's own caches and hidden states."""
    w = C.get("8b_shaped")
    m = G.model(w)
    tok0 = G.prompt_tokens(w)
    B, L, blk, d, H = w.batch, w.seq_len, w.block_len, w.d_model, w.n_heads
    seqs = [2, 6]
    gen = loop.DenseGenerator(w, {k: loop.to_device(v) for k, v in m.items()}, facache=True)
    got = []
    from gpu_util import read_kv_seqs

    def grab(t, q0, s):
        if t % 8 == 0 or t == w.steps_per_block - 1:
            got.append(dict(t=t, q0=q0, o=gen.o.float().cpu().numpy().reshape(B, blk, d),
                            h=gen.h.float().cpu().numpy().reshape(B, blk, d),
                            p1=gen.p1.cpu().numpy().reshape(B, blk), ent=gen.ent.cpu().numpy().reshape(B, blk),
                            qkv=[read_kv_seqs(gen.cache, f, 0, w, seqs) for f in (K.FIELD_Q, K.FIELD_K, K.FIELD_V)],
                            rebuilt=_rebuilt(gen.cache)))

    gen.tok_in.copy_(torch.from_numpy(tok0))
    try:
        gen.run(on_step=grab, n_steps=w.steps_per_block)
        assert K.dllm_cache_check(gen.cache) == 0
    finally:
        gen.close()
    W64 = O.weights_f64(replace(w, batch=1), {"w_lm": m["w_lm"]})
    rtol, atol = tol(w)
    for g in got:
        assert g["rebuilt"] == B * H, (g["t"], g["rebuilt"])      # once per (sequence, head), at the block start
        q0 = g["q0"]
        for si, b in enumerate(seqs):
            qg, kg, vg = (a[si] for a in g["qkv"])
            o_want = O.round_store(O.attention(qg[q0:q0 + blk], kg, vg).reshape(blk, d), w.dtype)
            assert close(g["o"][b], o_want, w), (g["t"], b, "o", worst(g["o"][b], o_want, w))
            am, p1, ent, margin = O.lm_head_conf(g["h"][b].astype(np.float64), W64["w_lm"], w.mask_id, w.rms_eps)
            assert np.allclose(g["p1"][b], p1, rtol=rtol, atol=atol), (g["t"], b, "p1")
            assert np.allclose(g["ent"][b], ent, rtol=rtol, atol=atol), (g["t"], b, "ent")
