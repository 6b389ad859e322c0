"""The multi-layer denoiser (GPU) layer by layer and step by step against the
oracle on the GPU's own inputs (teacher-forced).

Every step runs the library's calls one at a time (kv_refresh,
block_attn_rows, attn_out, ffn_gelu per layer; active_rows, lmhead_conf,
stab_update) and reads the results between them.  For the rows of the step's
row list P (all of them on the small shapes, a sample spread over the batch on
the 12-layer shapes) each layer is compared element by element with the
oracle applied to the GPU's inputs of that layer:
  * the cached Q, K, V rows the projection wrote (within one bf16 step; a
    query-only row's K/V untouched);
  * the attention output over the GPU's cache, W_o + residual and the FFN
    (2e-2 relative / 1e-3 absolute);
  * the LM head's argmax (where the top-2 margin exceeds 1e-2), top-1
    probability and entropy (2e-2 / 1e-3).
The integer state (tokens, stability, versions of every layer, token-at-write
and the next row list) must equal the oracle's bookkeeping applied to the
GPU's argmax and top-1 probabilities, bit for bit, at every step.  The
12-layer shape runs one whole block (64 steps: full refreshes at block-local
steps 0, 3, 6, ... from version expiry), and its sharp variant commits
positions inside the block."""
import numpy as np
import pytest
import torch

import oracle as O
from denoising_step_kv_gb300 import _lib as K
from denoising_step_kv_gb300 import loop
from gpu_util import close, read_field, read_kv_seqs, tol, worst
from test_gpu_fullsize import _qkv_close, _qkv_worst
from workloads import configs as C
from workloads import generate as G

pytestmark = pytest.mark.gpu


_kv_seqs = read_kv_seqs


def _rows_f64(t, idx):
    return t[torch.from_numpy(idx).to(t.device).long()].double().cpu().numpy()


def _sample(P, w, n_per_seq, seqs):
    """Positions i of the row list P to compare: every row on small shapes,
    else up to n_per_seq rows of each sampled sequence (its active rows first,
    then rows spread over the rest)."""
    if n_per_seq is None:
        return np.arange(len(P))
    L, q0s = w.seq_len, None
    out = []
    for b in seqs:
        mine = np.flatnonzero(P // L == b)
        if not len(mine):
            continue
        pos = P[mine] % L
        act = mine[(pos >= w.n_prompt)][:8]
        rest = np.setdiff1d(mine, act)
        pick = rest[np.linspace(0, len(rest) - 1, min(len(rest), n_per_seq - len(act))).astype(int)] if len(rest) else rest
        out.extend(np.concatenate([act, pick]).tolist())
    return np.unique(np.array(out, dtype=np.int64))


def _check_step_layers(gen, w, W64, D, t, q0, s, P, rf, seqs, n_per_seq, stats):
    """Run one denoising step call by call; compare every layer of the
    sampled rows.  Returns nothing; raises on a mismatch."""
    c = gen.cache
    B, L, H, dh, d, nl, blk = w.batch, w.seq_len, w.n_heads, w.head_dim, w.d_model, w.n_layers, w.block_len
    n = len(P)
    pick = _sample(P, w, n_per_seq, seqs)
    rows = P[pick]
    b_of, pos_of = rows // L, rows % L
    seq_list = sorted(set(int(b) for b in b_of))
    sidx = {b: i for i, b in enumerate(seq_list)}
    quiet = ~np.isin(rows, rf)                     # query-only rows (K/V must stay)
    tok_pre = gen.tok.cpu().numpy().reshape(-1)
    x = None
    x_in = W64["embed"][tok_pre[rows]]             # layer-0 input of the sampled rows
    for l in range(nl):
        if quiet.any():
            kv_pre = [_kv_seqs(c, f, l, w, seq_list) for f in (K.FIELD_K, K.FIELD_V)]
        K.kv_refresh(c, l, x, gen.tok, D["embed"], D["w_qkv"][l], gen.rows, gen.n_rows, t)
        q_all, k_all, v_all = (_kv_seqs(c, f, l, w, seq_list) for f in (K.FIELD_Q, K.FIELD_K, K.FIELD_V))
        si = np.array([sidx[int(b)] for b in b_of])
        qg, kg, vg = q_all[si, pos_of], k_all[si, pos_of], v_all[si, pos_of]
        qo, ko, vo = O.project_qkv(x_in, W64["w_qkv"][l], pos_of, H, w.dtype, w.rope_theta, w.rms_eps)
        assert _qkv_close(qg, qo), (w.name, t, l, "q", _qkv_worst(qg, qo))
        wr = ~quiet
        if wr.any():
            assert _qkv_close(kg[wr], ko[wr]), (w.name, t, l, "k", _qkv_worst(kg[wr], ko[wr]))
            assert _qkv_close(vg[wr], vo[wr]), (w.name, t, l, "v", _qkv_worst(vg[wr], vo[wr]))
        if quiet.any():
            qi = np.flatnonzero(quiet)
            assert np.array_equal(kg[qi], kv_pre[0][si[qi], pos_of[qi]]), (w.name, t, l, "k of a query-only row")
            assert np.array_equal(vg[qi], kv_pre[1][si[qi], pos_of[qi]]), (w.name, t, l, "v of a query-only row")
            stats["quiet"] += int(quiet.sum())
        # attention over the GPU's cache of the row's own sequence
        K.block_attn_rows(c, l, gen.rows, gen.n_rows, gen.O)
        og = _rows_f64(gen.O, pick)
        ow = np.zeros_like(og)
        for j in range(len(seq_list)):                    # the sampled queries of each sequence together
            sel = si == j
            if sel.any():
                ow[sel] = O.round_store(O.attention(qg[sel], k_all[j], v_all[j]).reshape(int(sel.sum()), -1),
                                        w.dtype)
        assert close(og, ow, w), (w.name, t, l, "o", worst(og, ow, w))
        # W_o + residual, then the FFN
        h = gen.H[l % 2]
        K.attn_out(c, gen.O, D["w_o"][l], x, None, None, 0, 1, gen.n_rows, h)
        h1 = _rows_f64(h, pick)
        hw = O.out_proj(og, W64["w_o"][l], x_in, w.dtype)
        assert close(h1, hw, w), (w.name, t, l, "h", worst(h1, hw, w))
        K.ffn_gelu(c, h, D["w1"][l], D["w2"][l], w.ffn, 0, gen.n_rows, h)
        h2 = _rows_f64(h, pick)
        fw = O.ffn(h1, W64["w1"][l], W64["w2"][l], w.dtype, w.rms_eps)
        assert close(h2, fw, w), (w.name, t, l, "ffn", worst(h2, fw, w))
        x, x_in = h, h2
        stats["rows"] += len(pick)
    # LM head of the active rows
    K.active_rows(c, x, gen.rows, gen.n_rows, q0, blk, gen.h)
    K.active_rows(c, gen.O, gen.rows, gen.n_rows, q0, blk, gen.o)
    K.lmhead_conf(c, gen.h, D["w_lm"], B * blk, w.vocab, d, w.mask_id, gen.argmax, gen.p1, gen.ent)
    ac_b = seqs if n_per_seq is not None else list(range(B))
    ia = np.concatenate([b * blk + np.arange(blk) for b in ac_b])
    hg = _rows_f64(gen.h, ia)
    am, p1, ent, margin = O.lm_head_conf(hg, W64["w_lm"], w.mask_id, w.rms_eps)
    rtol, atol = tol(w)
    g_am, g_p1, g_ent = gen.argmax.cpu().numpy(), gen.p1.cpu().numpy(), gen.ent.cpu().numpy()
    assert np.allclose(g_p1[ia], p1, rtol=rtol, atol=atol), (w.name, t, "p1", worst(g_p1[ia], p1, w))
    assert np.allclose(g_ent[ia], ent, rtol=rtol, atol=atol), (w.name, t, "ent", worst(g_ent[ia], ent, w))
    sure = margin > 1e-2
    assert np.array_equal(g_am[ia][sure], am[sure]), (w.name, t, "argmax")
    stats["sure"] += int(sure.sum())
    return g_am.reshape(B, blk), g_p1.reshape(B, blk), g_ent.reshape(B, blk)


def _teacher_forced(name, n_steps, seqs=None, n_per_seq=None):
    w = C.get(name)
    m = G.model(w)
    W64 = O.weights_f64(w, m)
    D = {k: loop.to_device(v) for k, v in m.items()}
    gen = loop.LayerStackGenerator(w, D)
    B, L, blk, nl = w.batch, w.seq_len, w.block_len, w.n_layers
    tok0 = G.prompt_tokens(w)
    # the oracle's bookkeeping, fed with the GPU's argmax / top-1 probabilities
    tok_o = tok0.astype(np.int64)
    stable_o = np.zeros((B, L), dtype=bool)
    version_o = np.full((nl, B, L), O.NEVER, dtype=np.int64)
    tok_w_o = np.full((B, L), -1, dtype=np.int64)
    swd = O.SWDState(B, blk)
    stats = {"rows": 0, "quiet": 0, "sure": 0, "commits": 0, "full": 0}
    try:
        gen.tok_in.copy_(torch.from_numpy(tok0))
        K.dllm_cache_reset(gen.cache)
        gen.tok.copy_(gen.tok_in)
        rf = None
        for t, q0, s in gen.schedule():
            if t >= n_steps:
                break
            if t == 0:
                K.refresh_all(gen.cache, q0, gen.rows, gen.n_rows)
                rf = np.arange(B * L)
            ac = (np.arange(B)[:, None] * L + q0 + np.arange(blk)[None, :]).reshape(-1)
            P = gen.rows[:int(gen.n_rows.item())].cpu().numpy().astype(np.int64)
            want_P = rf if len(rf) == B * L else np.union1d(rf, ac)
            assert np.array_equal(P, want_P), (name, t, "row list")
            stats["full"] += int(len(rf) == B * L)
            g_am, g_p1, g_ent = _check_step_layers(gen, w, W64, D, t, q0, s, P, rf, seqs, n_per_seq, stats)
            # bookkeeping of the refresh set, then SWD on the GPU's outputs
            version_o[:, rf // L, rf % L] = t
            tok_w_o.reshape(-1)[rf] = tok_o.reshape(-1)[rf]
            last = s == w.steps_per_block - 1
            newly = O.swd_update(swd, q0, g_am, g_p1, tok_o, stable_o, w.swd_K, w.swd_tau, last)
            stats["commits"] += int(newly.sum())
            K.stab_update(gen.cache, gen.argmax, gen.p1, gen.ent, gen.tok, q0, t, s, last, gen.rows, gen.n_rows)
            if last or O.full_refresh_at(s + 1, w.full_every):
                if last:
                    swd.reset()
                rf = np.arange(B * L)
            elif w.gate == "confidence":
                rf = O.confidence_rows(stable_o, tok_o, tok_w_o, version_o, q0, blk, g_ent, np.log(w.vocab - 1),
                                       t + 1, w.expiry, w.conf_alpha, w.conf_beta, 3.0 / w.steps_per_block,
                                       w.conf_theta)
            else:
                R = O.radius_at(s + 1, w.steps_per_block, w.swd_R, w.swd_R_min)
                rf = O.refresh_rows(stable_o, tok_o, tok_w_o, version_o, q0, blk, R, t + 1, w.expiry)
            assert np.array_equal(gen.tok.cpu().numpy(), tok_o), (name, t, "tok")
            assert np.array_equal(read_field(gen.cache, K.FIELD_STABLE, 0, (B, L), "u8").astype(bool), stable_o), \
                (name, t, "stable")
            assert np.array_equal(read_field(gen.cache, K.FIELD_VERSION, 0, (nl, B, L), "i32"), version_o), \
                (name, t, "version")
            assert np.array_equal(read_field(gen.cache, K.FIELD_TOK_W, 0, (B, L), "i32"), tok_w_o), \
                (name, t, "token-at-write")
        assert K.dllm_cache_check(gen.cache) == 0
    finally:
        gen.close()
    return stats


@pytest.mark.parametrize("name", ["mid_multi", "mid_multi_sharp", "mid_multi_conf"])
def test_layers_teacher_forced_small(name):
    w = C.get(name)
    stats = _teacher_forced(name, w.n_steps)
    assert stats["rows"] > 0 and stats["full"] >= w.n_blocks
    if name.endswith("sharp"):
        assert stats["commits"] > 0 and stats["quiet"] > 0      # query-only rows were checked
    if name.endswith("conf"):                                   # confident rows only query
        assert stats["quiet"] > 0


@pytest.mark.parametrize("name", ["twelve_layer", "twelve_layer_sharp"])
def test_layers_teacher_forced_twelve_layer_block(name):
    """One whole SAR block of the 12-layer denoiser at full batch, sampled
    sequences 0, 7 and 15."""
    w = C.get(name)
    stats = _teacher_forced(name, w.steps_per_block, seqs=[0, 7, 15], n_per_seq=24)
    if name.endswith("sharp"):
        assert stats["commits"] > 0
    else:           # version expiry: every row at block-local steps 0, 3, 6, ...
        assert stats["full"] >= w.steps_per_block // 3
