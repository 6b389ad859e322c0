"""The multi-layer denoiser (GPU) against the oracle: attention for a row
list, the active-row gather, the FFN, and free-running generations of a
3-layer model with the stability mask gating every layer's refresh (the
per-layer element-wise comparison runs teacher-forced in test_gpu_layers)."""
import numpy as np
import pytest
import torch

import oracle as O
from denoising_step_kv_gb300 import _lib as K
from denoising_step_kv_gb300 import loop
from denoising_step_kv_gb300.loop import to_device
from gpu_util import close, i32, max_err, read_field, tol, write_kv
from workloads import configs as C
from workloads import generate as G

pytestmark = pytest.mark.gpu


def _row_sets(B, L):
    every = np.arange(B * L)
    return {
        "all": every,                                        # several 128-query tiles per sequence
        "one_seq": every[L:L + min(L, 150)],                 # sequence 0 has no rows
        "sparse": np.sort(G.choice(31, B * L, min(B * L - 1, 77))),
        "single": np.array([B * L - 1]),
        "empty": np.array([], dtype=np.int64),
    }


@pytest.mark.parametrize("name", ["mid_multi", "big_rows", "mid_bf16"])
@pytest.mark.parametrize("which", ["all", "one_seq", "sparse", "single", "empty"])
def test_block_attn_rows(name, which):
    w = C.get(name)
    B, L, H, dh, d = w.batch, w.seq_len, w.n_heads, w.head_dim, w.d_model
    rnd = lambda s: O.round_store(G.normal(s, (B, L, H, dh), 1.0, "f32").astype(np.float64), w.dtype)
    q, k, v = rnd(41), rnd(42), rnd(43)
    rows = _row_sets(B, L)[which]
    layer = w.n_layers - 1
    c = K.dllm_cache_init(K.make_cfg(w))
    try:
        for f, a in ((K.FIELD_Q, q), (K.FIELD_K, k), (K.FIELD_V, v)):
            write_kv(c, f, layer, w, a)
        out = torch.full((B * L + 1, d), 7.0, dtype=torch.bfloat16, device="cuda")
        rows_d = torch.zeros(B * L, dtype=torch.int32, device="cuda")
        if len(rows):
            rows_d[:len(rows)] = i32(rows)
        K.block_attn_rows(c, layer, rows_d, i32([len(rows)]), out)
        assert K.dllm_cache_check(c) == 0
        got = out.float().cpu().numpy().astype(np.float64)
        for i, r in enumerate(rows):
            b, p = divmod(int(r), L)
            want = O.round_store(O.attention(q[b, p][None], k[b], v[b])[0], w.dtype).reshape(-1)
            assert close(got[i], want, w), (name, which, i, max_err(got[i], want))
        assert np.all(got[len(rows):] == 7.0)          # nothing written past the list
    finally:
        K.dllm_cache_free(c)


def test_active_rows_gather():
    w = C.get("mid_multi")
    B, L, d, blk, q0 = w.batch, w.seq_len, w.d_model, w.block_len, w.n_prompt
    rows = np.sort(np.concatenate([b * L + np.arange(q0 - 3, q0 + blk + 2) for b in range(B)] + [np.array([5, L + 7])]))
    src = torch.arange(len(rows) * d, dtype=torch.float32, device="cuda").reshape(len(rows), d).to(torch.bfloat16)
    c = K.dllm_cache_init(K.make_cfg(w))
    try:
        dst = torch.zeros(B * blk, d, dtype=torch.bfloat16, device="cuda")
        rows_d = torch.zeros(B * L, dtype=torch.int32, device="cuda")
        rows_d[:len(rows)] = i32(rows)
        K.active_rows(c, src, rows_d, i32([len(rows)]), q0, blk, dst)
        assert K.dllm_cache_check(c) == 0
        for b in range(B):
            for j in range(blk):
                i = int(np.searchsorted(rows, b * L + q0 + j))
                assert torch.equal(dst[b * blk + j], src[i])
        # a missing row: error bit and a zero row
        K.active_rows(c, src, rows_d, i32([len(rows)]), q0 + blk, 3, dst)
        assert K.dllm_cache_error_word(c) & K.ERR_ROW
    finally:
        K.dllm_cache_free(c)


@pytest.mark.parametrize("n", [None, 37, 200])
def test_ffn_gelu(n):
    w = C.get("mid_multi")
    m = G.model(w)
    W = O.weights_f64(w, m)
    B, L, d = w.batch, w.seq_len, w.d_model
    M = B * L
    x = G.normal(51, (M, d), 1.0, "bf16")
    c = K.dllm_cache_init(K.make_cfg(w))
    try:
        h = to_device(x)
        out = torch.zeros_like(h)
        if n is None:
            K.ffn_gelu(c, h, to_device(m["w1"][1]), to_device(m["w2"][1]), w.ffn, M, None, out)
            rows = M
        else:
            K.ffn_gelu(c, h, to_device(m["w1"][1]), to_device(m["w2"][1]), w.ffn, 0, i32([n]), out)
            rows = n
        assert K.dllm_cache_check(c) == 0
        want = O.ffn(O.bf16_bits_to_f64(x)[:rows], W["w1"][1], W["w2"][1], w.dtype, w.rms_eps)
        got = out.float().cpu().numpy().astype(np.float64)[:rows]
        assert close(got, want, w), max_err(got, want)
    finally:
        K.dllm_cache_free(c)


# A stability decision whose mean top-1 probability lies within the
# probability tolerance at tau (1e-3 absolute + 2e-2 relative) of tau may go
# either way after three bf16 layers; the teacher-forced test of
# test_gpu_layers compares every decision exactly on the GPU's own inputs.
def p_band(tau):
    return 1e-3 + 2e-2 * tau


def _ambiguous(rec, w):
    """Active positions whose argmax (top-2 margin <= 1e-2) or stability
    decision (mean top-1 probability within p_band(tau) of tau) may differ."""
    band = p_band(w.swd_tau)
    amb = rec["margin"] <= 1e-2
    for b in range(w.batch):
        for j in range(w.block_len):
            ps = rec["swd"].p[b][j]
            if len(ps) == w.swd_K and abs(float(np.mean(ps)) - w.swd_tau) < band:
                amb[b, j] = True
    return amb


@pytest.mark.parametrize("name", ["mid_multi", "mid_multi_sharp"])
def test_layer_stack_generation(name):
    """Free-running generation of the 3-layer model: every step's confidences
    (the oracle's LM head on the GPU's hidden states, element-wise) and,
    until a position whose argmax margin is <= 1e-2 or whose mean top-1
    probability lies within the probability tolerance of tau could part the
    trajectories, tokens, stability, the row list and every layer's
    versions, bit for bit."""
    w = C.get(name)
    m = G.model(w)
    tok0 = G.prompt_tokens(w)
    trace = O.run_dense(w, O.weights_f64(w, m), tok0)
    gen = loop.LayerStackGenerator(w, {k: to_device(v) for k, v in m.items()})
    B, L, blk, d, nl = w.batch, w.seq_len, w.block_len, w.d_model, w.n_layers
    got = []

    def grab(t, q0, s):
        got.append(dict(argmax=gen.argmax.cpu().numpy().reshape(B, blk), p1=gen.p1.cpu().numpy().reshape(B, blk),
                        ent=gen.ent.cpu().numpy().reshape(B, blk), tok=gen.tok.cpu().numpy().copy(),
                        o=gen.o.float().cpu().numpy().reshape(B, blk, d), h=gen.h.float().cpu().numpy().reshape(B, blk, d),
                        rows=gen.rows.cpu().numpy()[:int(gen.n_rows.item())].copy(),
                        version=read_field(gen.cache, K.FIELD_VERSION, 0, (nl, B, L), "i32"),
                        stable=read_field(gen.cache, K.FIELD_STABLE, 0, (B, L), "u8").astype(bool)))

    gen.tok_in.copy_(torch.from_numpy(tok0))
    try:
        gen.run(on_step=grab)
        assert K.dllm_cache_check(gen.cache) == 0
    finally:
        gen.close()
    rtol, atol = tol(w)
    W64 = O.weights_f64(w, m)
    compared = 0
    for rec, g in zip(trace, got):
        t = rec["t"]
        # the LM head and confidences: the oracle's on the GPU's own hidden states
        am, p1, ent, margin = O.lm_head_conf(g["h"].reshape(B * blk, d).astype(np.float64), W64["w_lm"],
                                             w.mask_id, w.rms_eps)
        assert np.allclose(g["p1"].reshape(-1), p1, rtol=rtol, atol=atol), (name, t, "p1")
        assert np.allclose(g["ent"].reshape(-1), ent, rtol=rtol, atol=atol), (name, t, "ent")
        sure = margin > 1e-2
        assert np.array_equal(g["argmax"].reshape(-1)[sure], am[sure]), (name, t, "argmax")
        # the trajectory, while no decision hangs on the stack's rounding
        amb = _ambiguous(rec, w)
        if np.any(g["argmax"] != rec["argmax"]):
            assert np.all(amb[g["argmax"] != rec["argmax"]]), (name, t, "argmax against the trajectory")
            break
        q0 = rec["q0"]
        blk_diff = g["stable"][:, q0:q0 + blk] != rec["stable"][:, q0:q0 + blk]
        if np.any(blk_diff):
            assert np.all(amb[blk_diff]), (name, t, "stable outside the ambiguous band")
            break
        assert np.array_equal(g["tok"], rec["tok"]), (name, t, "tok")
        assert np.array_equal(g["stable"], rec["stable"]), (name, t, "stable")
        assert np.array_equal(g["rows"], rec["rows_next"]), (name, t, "rows")
        assert np.array_equal(g["version"], rec["version"]), (name, t, "version")
        compared += 1
    assert compared >= 1, (name, compared)
