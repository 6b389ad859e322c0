"""Per-kernel parity of the CUDA path against the CPU oracle (GPU).

Every entry point of the C ABI runs in isolation on seeded inputs at sizes
the oracle finishes in seconds, with ragged tails against the GPU tiles
(rows not a multiple of 128, vocab 1000 = 7 tiles + 104, 160 keys = 2.5
key tiles), plus empty and out-of-range cases."""
import numpy as np
import pytest
import torch

import oracle as O
from denoising_step_kv_gb300 import _lib as K
from denoising_step_kv_gb300.loop import to_device
from gpu_util import cache_fields, close, i32, max_err, read_field, read_kv, tol, write_field, write_kv
from workloads import configs as C
from workloads import generate as G

pytestmark = pytest.mark.gpu

CFGS = ["tiny_fp32", "mid_bf16", "mid_bf16_dh64"]


def _setup(name):
    w = C.get(name)
    m = G.model(w)
    W = O.weights_f64(w, m)
    return w, m, W, {k: to_device(v) for k, v in m.items()}


def _fresh(w):
    return K.dllm_cache_init(K.make_cfg(w))


@pytest.mark.parametrize("name", CFGS)
def test_kv_refresh_all_rows(name):
    w, m, W, D = _setup(name)
    B, L, H, dh, d = w.batch, w.seq_len, w.n_heads, w.head_dim, w.d_model
    tok = G.integers(1, 1, w.vocab, (B, L))
    c = _fresh(w)
    try:
        K.kv_refresh(c, 0, None, i32(tok), D["embed"], D["w_qkv"][0], None, None, 7)
        assert K.dllm_cache_check(c) == 0
        q, k, v = O.project_qkv(W["embed"][tok.reshape(-1)], W["w_qkv"][0], np.tile(np.arange(L), B), H, w.dtype)
        for f, want in ((K.FIELD_Q, q), (K.FIELD_K, k), (K.FIELD_V, v)):
            got = read_kv(c, f, 0, w).reshape(B * L, H, dh)
            assert close(got, want, w), (name, f, max_err(got, want))
        ver = read_field(c, K.FIELD_VERSION, 0, (B * L,), "i32")
        tw = read_field(c, K.FIELD_TOK_W, 0, (B * L,), "i32")
        assert np.all(ver == 7) and np.array_equal(tw, tok.reshape(-1))
    finally:
        K.dllm_cache_free(c)


@pytest.mark.parametrize("name", CFGS)
def test_kv_refresh_ragged_rows(name):
    w, m, W, D = _setup(name)
    B, L, H, dh = w.batch, w.seq_len, w.n_heads, w.head_dim
    tok = G.integers(2, 1, w.vocab, (B, L))
    n = min(157, B * L - 3)
    rows = G.choice(3, B * L, n)
    c = _fresh(w)
    try:
        rows_d = torch.zeros(B * L, dtype=torch.int32, device="cuda")
        rows_d[:n] = i32(rows)
        K.kv_refresh(c, 0, None, i32(tok), D["embed"], D["w_qkv"][0], rows_d, i32([n]), 11)
        assert K.dllm_cache_check(c) == 0
        q, k, v = O.project_qkv(W["embed"][tok.reshape(-1)[rows]], W["w_qkv"][0], rows % L, H, w.dtype)
        untouched = np.setdiff1d(np.arange(B * L), rows)
        for f, want in ((K.FIELD_Q, q), (K.FIELD_K, k), (K.FIELD_V, v)):
            got = read_kv(c, f, 0, w).reshape(B * L, H, dh)
            assert close(got[rows], want, w), (name, f, max_err(got[rows], want))
            assert np.all(got[untouched] == 0)
        ver = read_field(c, K.FIELD_VERSION, 0, (B * L,), "i32")
        assert np.all(ver[rows] == 11) and np.all(ver[untouched] == O.NEVER)
    finally:
        K.dllm_cache_free(c)


@pytest.mark.parametrize("name", ["big_rows", "big_rows_dh64"])
@pytest.mark.parametrize("n", [None, 700, 530, 513, 512, 300, 257, 200])
def test_kv_refresh_large_m(name, n):
    """Row counts around the weight-streaming range: the host count (every
    row) and device counts on both sides of the 256-row limit of the split-K
    weight-streaming kernel and of the 512-row one of the pair kernel."""
    w, m, W, D = _setup(name)
    B, L, H, dh = w.batch, w.seq_len, w.n_heads, w.head_dim
    tok = G.integers(5, 1, w.vocab, (B, L))
    if n is not None and n > B * L:
        pytest.skip("more rows than the cache holds")
    rows = np.arange(B * L) if n is None else G.choice(6 + (n or 0), B * L, n)
    c = _fresh(w)
    try:
        if n is None:
            K.kv_refresh(c, 0, None, i32(tok), D["embed"], D["w_qkv"][0], None, None, 4)
        else:
            rows_d = torch.zeros(B * L, dtype=torch.int32, device="cuda")
            rows_d[:n] = i32(rows)
            K.kv_refresh(c, 0, None, i32(tok), D["embed"], D["w_qkv"][0], rows_d, i32([n]), 4)
        assert K.dllm_cache_check(c) == 0
        q, k, v = O.project_qkv(W["embed"][tok.reshape(-1)[rows]], W["w_qkv"][0], rows % L, H, w.dtype)
        untouched = np.setdiff1d(np.arange(B * L), rows)
        for f, want in ((K.FIELD_Q, q), (K.FIELD_K, k), (K.FIELD_V, v)):
            got = read_kv(c, f, 0, w).reshape(B * L, H, dh)
            assert close(got[rows], want, w), (name, n, f, max_err(got[rows], want))
            assert np.all(got[untouched] == 0)
    finally:
        K.dllm_cache_free(c)


@pytest.mark.parametrize("n", [0, 1, 200, 256, 272, 300, 512])
def test_kv_refresh_wide_projection(n):
    """The 8B-shaped projection (d 4096, N = 3d = 12288: 96 weight tiles, the
    weight-streaming kernel without a split of K) at device row counts up to
    512; rows past 256 take its second MMA.  Sampled rows on both sides of
    256, and the last, against the oracle; rows outside the list untouched;
    a count of 0 writes nothing."""
    from dataclasses import replace
    w = replace(C.get("8b_shaped"), batch=1, seq_len=640, n_prompt=576, vocab=1000)
    B, L, H, dh = w.batch, w.seq_len, w.n_heads, w.head_dim
    embed, wqkv = G.embed(w), G.w_qkv(w, 0)
    tok = G.integers(8, 1, w.vocab, (B, L))
    rows = G.choice(9 + n, B * L, n)
    c = _fresh(w)
    try:
        rows_d = torch.zeros(B * L, dtype=torch.int32, device="cuda")
        rows_d[:n] = i32(rows)
        K.kv_refresh(c, 0, None, i32(tok), to_device(embed), to_device(wqkv), rows_d, i32([n]), 4)
        assert K.dllm_cache_check(c) == 0
        if n == 0:
            for f in (K.FIELD_Q, K.FIELD_K, K.FIELD_V):
                assert not np.any(read_kv(c, f, 0, w))
            return
        pick = np.unique(np.clip([0, 1, 127, 128, 255, 256, 257, 271, 272, 300, n - 1], 0, n - 1))
        sel = rows[pick]
        x = O.bf16_bits_to_f64(embed)[tok.reshape(-1)[sel]]
        q, k, v = O.project_qkv(x, O.bf16_bits_to_f64(wqkv), sel % L, H, w.dtype, w.rope_theta, w.rms_eps)
        untouched = np.setdiff1d(np.arange(B * L), rows)
        for f, want in ((K.FIELD_Q, q), (K.FIELD_K, k), (K.FIELD_V, v)):
            got = read_kv(c, f, 0, w).reshape(B * L, H, dh)
            assert close(got[sel], want, w), (n, f, max_err(got[sel], want))
            assert np.all(got[untouched] == 0)
    finally:
        K.dllm_cache_free(c)


def test_kv_refresh_empty_and_bad_rows():
    w, m, W, D = _setup("mid_bf16")
    B, L = w.batch, w.seq_len
    tok = G.integers(4, 1, w.vocab, (B, L))
    c = _fresh(w)
    try:
        rows_d = torch.zeros(B * L, dtype=torch.int32, device="cuda")
        K.kv_refresh(c, 0, None, i32(tok), D["embed"], D["w_qkv"][0], rows_d, i32([0]), 1)
        assert K.dllm_cache_check(c) == 0
        assert np.all(read_field(c, K.FIELD_VERSION, 0, (B * L,), "i32") == O.NEVER)
        rows_d[:3] = i32([5, B * L + 7, 9])            # one row out of range
        K.kv_refresh(c, 0, None, i32(tok), D["embed"], D["w_qkv"][0], rows_d, i32([3]), 2)
        word = K.dllm_cache_error_word(c)
        assert word & K.ERR_ROW
        ver = read_field(c, K.FIELD_VERSION, 0, (B * L,), "i32")
        assert ver[5] == 2 and ver[9] == 2
        bad = tok.copy()
        bad[0, 3] = w.vocab + 5                         # token out of range
        rows_d[:2] = i32([3, 4])
        K.kv_refresh(c, 0, None, i32(bad), D["embed"], D["w_qkv"][0], rows_d, i32([2]), 3)
        assert K.dllm_cache_error_word(c) & K.ERR_TOKEN
        ver = read_field(c, K.FIELD_VERSION, 0, (B * L,), "i32")
        assert ver[3] == O.NEVER and ver[4] == 3
        with pytest.raises(K.DllmError):
            K.kv_refresh(c, 5, None, i32(tok), D["embed"], D["w_qkv"][0], None, None, 0)
    finally:
        K.dllm_cache_free(c)


@pytest.mark.parametrize("name", CFGS)
@pytest.mark.parametrize("q_start,q_len", [(0, 8), (-1, 16), (37, 13), (3, 64)])
def test_block_attn(name, q_start, q_len):
    w, m, W, D = _setup(name)
    B, L, H, dh, d = w.batch, w.seq_len, w.n_heads, w.head_dim, w.d_model
    if q_start < 0:
        q_start = L - q_len
    if q_start + q_len > L:
        pytest.skip("query range longer than the sequence")
    st = cache_fields(w)
    rnd = lambda s: O.round_store(G.normal(s, (B, L, H, dh), 1.0, "f32").astype(np.float64), w.dtype)
    q, k, v = rnd(21), rnd(22), rnd(23)
    c = _fresh(w)
    try:
        for f, a in ((K.FIELD_Q, q), (K.FIELD_K, k), (K.FIELD_V, v)):
            write_kv(c, f, 0, w, a)
        dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
        out = torch.zeros(B * q_len, d, dtype=dt, device="cuda")
        K.block_attn(c, 0, q_start, q_len, out, None)
        assert K.dllm_cache_check(c) == 0
        got = out.float().cpu().numpy().astype(np.float64).reshape(B, q_len, H, dh)
        for b in range(B):
            want = O.round_store(O.attention(q[b, q_start:q_start + q_len], k[b], v[b]), w.dtype)
            assert close(got[b], want, w), (name, b, max_err(got[b], want))
    finally:
        K.dllm_cache_free(c)


@pytest.mark.parametrize("name,q_len", [("8b_shaped", 32), ("bf16_d2048", 32), ("bf16_d2048", 16)])
def test_block_attn_many_tiles(name, q_len):
    """Full-size key ranges: every CTA streams many K/V tiles through the
    3-stage ring (8B-shaped: one split, 64 tiles per CTA), so every stage
    barrier goes through many phases; sampled (sequence, head) pairs are
    checked against the oracle."""
    w = C.get(name)
    B, L, H, dh, d = w.batch, w.seq_len, w.n_heads, w.head_dim, w.d_model
    q0 = w.n_prompt
    c = _fresh(w)
    try:
        fields = {}
        for f, seed in ((K.FIELD_Q, 51), (K.FIELD_K, 52), (K.FIELD_V, 53)):
            a = G.normal(seed, (B * L, d), 0.5, "bf16")
            fields[f] = O.bf16_bits_to_f64(a).reshape(B, L, H, dh)
            write_kv(c, f, 0, w, fields[f])
        out = torch.zeros(B * q_len, d, dtype=torch.bfloat16, device="cuda")
        for _ in range(3):                       # repeated launches reuse the same code path
            K.block_attn(c, 0, q0, q_len, out, None)
        assert K.dllm_cache_check(c) == 0
        got = out.float().cpu().numpy().astype(np.float64).reshape(B, q_len, H, dh)
        for b, h in [(0, 0), (B - 1, H - 1), (B // 2, H // 3)]:
            want = O.round_store(O.attention(fields[K.FIELD_Q][b, q0:q0 + q_len, h:h + 1],
                                             fields[K.FIELD_K][b, :, h:h + 1], fields[K.FIELD_V][b, :, h:h + 1]),
                                 "bf16")
            assert close(got[b, :, h:h + 1], want, w), (name, b, h, max_err(got[b, :, h:h + 1], want))
    finally:
        K.dllm_cache_free(c)


@pytest.mark.parametrize("name", CFGS)
def test_attn_out(name):
    w, m, W, D = _setup(name)
    B, L, d, blk = w.batch, w.seq_len, w.d_model, w.block_len
    tok = G.integers(5, 1, w.vocab, (B, L))
    q0 = w.n_prompt
    o = G.normal(31, (B * blk, d), 1.0, w.dtype)
    c = _fresh(w)
    try:
        dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
        h = torch.zeros(B * blk, d, dtype=dt, device="cuda")
        K.attn_out(c, to_device(o), D["w_o"][0], None, i32(tok), D["embed"], q0, blk, None, h, None)
        assert K.dllm_cache_check(c) == 0
        of = O.bf16_bits_to_f64(o) if w.dtype == "bf16" else o.astype(np.float64)
        x = W["embed"][tok[:, q0:q0 + blk].reshape(-1)]
        want = O.out_proj(of, W["w_o"][0], x, w.dtype)
        got = h.float().cpu().numpy().astype(np.float64)
        assert close(got, want, w), (name, max_err(got, want))
    finally:
        K.dllm_cache_free(c)


@pytest.mark.parametrize("name", CFGS)
def test_lmhead_conf(name):
    w, m, W, D = _setup(name)
    M = w.batch * w.block_len
    h = G.normal(41, (M, w.d_model), 1.0, w.dtype)
    c = _fresh(w)
    try:
        am = torch.zeros(M, dtype=torch.int32, device="cuda")
        p1 = torch.zeros(M, dtype=torch.float32, device="cuda")
        ent = torch.zeros(M, dtype=torch.float32, device="cuda")
        for scale in (1.0, 40.0):
            wl = G.normal(42, (w.vocab, w.d_model), 0.02 * scale, w.dtype)
            K.lmhead_conf(c, to_device(h), to_device(wl), M, w.vocab, w.d_model, w.mask_id, am, p1, ent, None)
            assert K.dllm_cache_check(c) == 0
            hf = O.bf16_bits_to_f64(h) if w.dtype == "bf16" else h.astype(np.float64)
            wf = O.bf16_bits_to_f64(wl) if w.dtype == "bf16" else wl.astype(np.float64)
            a_o, p_o, e_o, margin = O.lm_head_conf(hf, wf, w.mask_id)
            ok = margin > 1e-2
            assert ok.sum() > M // 2
            assert np.array_equal(am.cpu().numpy()[ok], a_o[ok])
            assert np.all(am.cpu().numpy() != w.mask_id)
            rtol, atol = tol(w)
            assert np.allclose(p1.cpu().numpy(), p_o, rtol=rtol, atol=atol), max_err(p1.cpu().numpy(), p_o)
            assert np.allclose(ent.cpu().numpy(), e_o, rtol=rtol, atol=atol), max_err(ent.cpu().numpy(), e_o)
    finally:
        K.dllm_cache_free(c)


@pytest.mark.parametrize("V,M", [(1640, 32), (1640, 200), (4100, 256), (9, 5), (50000, 129), (50000, 200),
                                 (50000, 256), (126464, 256), (32000, 128), (50000, 100), (126464, 64)])
def test_lmhead_conf_vocab_groups(V, M):
    """Vocab sizes whose 128-column tiles do not fill the last cluster group
    (13 tiles in groups of 4), more than one 128-row tile, a vocab below one
    group (the plain persistent kernel), large vocabularies at 129..256
    rows (pairs of row tiles on 256-column weight tiles; V 50000 leaves a
    80-column tail), and one row tile over large vocabularies (the shared-A
    kernel's 256-column tiles in groups of four: V 32000 leaves three tiles
    of the last group past the vocab, V 50000 an 80-column tail)."""
    from dataclasses import replace
    w = replace(C.get("mid_bf16"), vocab=V, batch=1, block_len=min(64, M), seq_len=max(160, M))
    c = K.dllm_cache_init(K.make_cfg(w))
    try:
        h = G.normal(43, (M, w.d_model), 1.0, "bf16")
        wl = G.normal(44, (V, w.d_model), 0.8, "bf16")
        am = torch.zeros(M, dtype=torch.int32, device="cuda")
        p1 = torch.zeros(M, dtype=torch.float32, device="cuda")
        ent = torch.zeros(M, dtype=torch.float32, device="cuda")
        out = K.lmhead_conf_noalloc if M > w.batch * w.block_len else None
        if out is None:
            K.lmhead_conf(c, to_device(h), to_device(wl), M, V, w.d_model, 0, am, p1, ent, None)
        else:
            K.lmhead_conf_noalloc(to_device(h), to_device(wl), M, V, w.d_model, K.DLLM_BF16, 0, 1e-6, am, p1, ent)
        assert K.dllm_cache_check(c) == 0
        torch.cuda.synchronize()
        a_o, p_o, e_o, margin = O.lm_head_conf(O.bf16_bits_to_f64(h), O.bf16_bits_to_f64(wl), 0)
        ok = margin > 1e-2
        assert np.array_equal(am.cpu().numpy()[ok], a_o[ok])
        rtol, atol = tol(w)
        assert np.allclose(p1.cpu().numpy(), p_o, rtol=rtol, atol=atol), max_err(p1.cpu().numpy(), p_o)
        assert np.allclose(ent.cpu().numpy(), e_o, rtol=rtol, atol=atol), max_err(ent.cpu().numpy(), e_o)
    finally:
        K.dllm_cache_free(c)


def _ring_to_lists(ht, hp, hn, K_):
    """Device ring (slot n % K) -> oracle per-position lists, oldest first."""
    toks, ps = [], []
    n = int(hn)
    for k in range(min(n, K_)):
        slot = (n - min(n, K_) + k) % K_
        toks.append(int(ht[slot]))
        ps.append(np.float32(hp[slot]))
    return toks, ps


@pytest.mark.parametrize("name", ["mid_bf16", "mid_bf16_dh64", "tiny_fp32", "mid_multi"])
@pytest.mark.parametrize("last", [False, True])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_stab_update_random_state(name, last, seed):
    w = C.get(name)
    B, L, blk, Kk, nl = w.batch, w.seq_len, w.block_len, w.swd_K, w.n_layers
    q0 = w.n_prompt + (seed % w.n_blocks) * blk
    s0 = 100 * seed + (1 if last else 0)
    t = 20
    tok = G.integers(s0 + 1, 0, 6, (B, L))
    tok_w = tok.copy()
    flip = G.integers(s0 + 2, 0, 25, (B, L)) == 0
    tok_w[flip] = G.integers(s0 + 3, 0, 6, (B, L))[flip]
    version = G.integers(s0 + 4, t - 4, t + 1, (nl, B, L))
    stable = np.zeros((B, L), dtype=bool)
    stable[:, q0:q0 + blk] = G.integers(s0 + 5, 0, 4, (B, blk)) == 0
    hist_tok = G.integers(s0 + 6, 1, 3, (B, blk, Kk))
    hist_p = G.uniform(s0 + 7, 0.8, 1.0, (B, blk, Kk))
    hist_n = G.integers(s0 + 8, 0, Kk + 3, (B, blk))
    argmax = G.integers(s0 + 9, 1, 3, (B, blk))
    p1 = G.uniform(s0 + 10, 0.8, 1.0, (B, blk))
    # oracle
    st = O.SWDState(B, blk)
    for b in range(B):
        for j in range(blk):
            st.tok[b][j], st.p[b][j] = _ring_to_lists(hist_tok[b, j], hist_p[b, j], hist_n[b, j], Kk)
            st.n[b, j] = hist_n[b, j]
    tok_o, stable_o = tok.copy().astype(np.int64), stable.copy()
    O.swd_update(st, q0, argmax, p1, tok_o, stable_o, Kk, w.swd_tau, last)
    if last:
        rows_o = np.arange(B * L)
    else:
        rows_o = O.refresh_rows(stable_o, tok_o, tok_w, version, q0, blk, w.swd_R, t + 1, w.expiry)
        if w.active_queries:             # the row list also holds every active row
            ac = (np.arange(B)[:, None] * L + q0 + np.arange(blk)[None, :]).reshape(-1)
            rows_o = np.union1d(rows_o, ac).astype(np.int32)
    # GPU
    c = _fresh(w)
    try:
        write_field(c, K.FIELD_TOK_W, 0, tok_w, "i32")
        write_field(c, K.FIELD_VERSION, 0, version, "i32")
        write_field(c, K.FIELD_STABLE, 0, stable.reshape(-1), "u8")
        write_field(c, K.FIELD_HIST_TOK, 0, hist_tok, "i32")
        write_field(c, K.FIELD_HIST_P, 0, hist_p, "f32")
        write_field(c, K.FIELD_HIST_N, 0, hist_n, "i32")
        tok_d = i32(tok)
        rows = torch.full((B * L,), -1, dtype=torch.int32, device="cuda")
        n_rows = torch.zeros(1, dtype=torch.int32, device="cuda")
        K.stab_update(c, i32(argmax), torch.from_numpy(p1.reshape(-1)).cuda(), None, tok_d, q0, t, 1, last, rows,
                      n_rows)
        assert K.dllm_cache_check(c) == 0
        n = int(n_rows.item())
        assert n == len(rows_o)
        assert np.array_equal(rows.cpu().numpy()[:n], rows_o)
        assert np.array_equal(tok_d.cpu().numpy(), tok_o)
        assert np.array_equal(read_field(c, K.FIELD_STABLE, 0, (B, L), "u8").astype(bool), stable_o)
        hn = read_field(c, K.FIELD_HIST_N, 0, (B, blk), "i32")
        if last:
            assert np.all(hn == 0)
        else:
            ht = read_field(c, K.FIELD_HIST_TOK, 0, (B, blk, Kk), "i32")
            hp = read_field(c, K.FIELD_HIST_P, 0, (B, blk, Kk), "f32")
            for b in range(B):
                for j in range(blk):
                    if stable[b, q0 + j]:
                        continue
                    gt, gp = _ring_to_lists(ht[b, j], hp[b, j], hn[b, j], Kk)
                    assert gt == st.tok[b][j][-len(gt):] and len(gt) == len(st.tok[b][j])
    finally:
        K.dllm_cache_free(c)


def test_refresh_all_lists_every_row():
    w = C.get("mid_bf16")
    c = _fresh(w)
    try:
        rows = torch.full((w.batch * w.seq_len,), -1, dtype=torch.int32, device="cuda")
        n_rows = torch.zeros(1, dtype=torch.int32, device="cuda")
        K.refresh_all(c, w.n_prompt, rows, n_rows)
        torch.cuda.synchronize()
        assert int(n_rows.item()) == w.batch * w.seq_len
        assert np.array_equal(rows.cpu().numpy(), np.arange(w.batch * w.seq_len))
    finally:
        K.dllm_cache_free(c)
