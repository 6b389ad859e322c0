"""Oracle step loops: the cached algorithm and the plain full recompute.

Sources, cited by page title and section:
  [LaCache] "Inference workflow": the first denoising step of a block runs a
            full forward and refills the caches; later steps reuse the states
            of unchanged tokens and recompute only what changed.
            "Limitations": reuse is exact only for the first layer; deeper
            layers reuse stale states (an approximation).
  [SWD]     3.3: per step, compute on the masked-in positions, then update the
            stability history and the stable set.
  [Sinks]   "Attention Sinks and Where to Cache Them" explainer
            (wmrh.cn/news/159578), 2.3 / 3.1 / 3.2 / 3.3: keep the first S
            tokens' K/V for ever plus a rolling window of the newest W; the new
            token's K/V joins the window before its query attends; positions
            never roll (each token keeps its own stream index).

Two dense modes:
  * ``cached``: explicit per-layer Q/K/V caches with versions; only the refresh
    set Rf is recomputed (single-layer: exactly the method; multi-layer: the
    rows P = Rf, plus the active block when the workload asks for active
    queries, pass through every layer as queries; only the rows of Rf rewrite
    their K/V and version, so the stability mask gates the per-layer refresh,
    and every other row's deeper-layer K/V stays as cached);
  * ``recompute``: the plain definition, a full forward of every row every step.
For one layer the two agree bit for bit (tested).
"""
from collections import deque

import numpy as np

from . import model as M
from .swd import SWDState, swd_update, refresh_rows, radius_at, full_refresh_at, confidence_rows, step_stats

NEVER = -(1 << 30)     # version of a cache entry that was never written


def weights_f64(w, m):
    """Generated weight arrays -> fp64 values."""
    conv = M.bf16_bits_to_f64 if w.dtype == "bf16" else (lambda a: np.asarray(a, np.float64))
    return {k: ([conv(x) for x in v] if isinstance(v, list) else conv(v)) for k, v in m.items()}


def _layer_stack(w, W, x, pos_rows, rows_flat, caches, write_kv=None):
    """Run rows through every layer of the cached algorithm.

    x: [n, d] layer-0 input of the rows; rows_flat: their flat ids b*L+pos.
    write_kv: bool [n], the rows that rewrite their K/V (the refresh set);
    None = every row.  Every row's Q is computed and stored; the queries are
    the rows themselves and attend over the layer's cache after this layer's
    K/V writes.  Returns (last O stored [n, d], final hidden [n, d]).
    """
    B, L, H = w.batch, w.seq_len, w.n_heads
    b_of = rows_flat // L
    o_last = None
    for l in range(w.n_layers):
        q, k, v = M.project_qkv(x, W["w_qkv"][l], pos_rows, H, w.dtype, w.rope_theta, w.rms_eps)
        Qc, Kc, Vc = caches
        wr = np.ones(len(rows_flat), dtype=bool) if write_kv is None else write_kv
        Qc[l].reshape(B * L, H, -1)[rows_flat] = q
        Kc[l].reshape(B * L, H, -1)[rows_flat[wr]] = k[wr]
        Vc[l].reshape(B * L, H, -1)[rows_flat[wr]] = v[wr]
        o = np.zeros_like(q)
        for b in range(B):
            sel = b_of == b
            if sel.any():
                o[sel] = M.attention(q[sel], Kc[l][b], Vc[l][b])
        o_st = M.round_store(o.reshape(len(x), -1), w.dtype)
        h = M.out_proj(o_st, W["w_o"][l], x, w.dtype)
        if w.ffn:
            h = M.ffn(h, W["w1"][l], W["w2"][l], w.dtype, w.rms_eps)
        x, o_last = h, o_st
    return o_last, x


def run_dense(w, W, tok0, n_steps=None, mode="cached", force_all=False, keep_pre=False, facache=False):
    """Run the SAR step loop.  Returns a list of per-step records.

    W: fp64 weights (``weights_f64``); tok0: [B, L] int32 initial tokens.
    mode: "cached" or "recompute"; force_all: refresh every row every step.
    keep_pre: record the pre-step state (including caches) of every step.
    n_steps caps the number of steps run.
    facache (single-layer cached mode): [LaCache] LSM, FACache - the
    online-softmax state of the active queries over the keys outside the
    block's window [q0 - R, q0 + blk + R) is kept per sequence with the
    block start and the queries' token-at-write, and reused (merged with the
    window's fresh state) while they are unchanged; the record's
    "fa_rebuilt" lists the sequences whose state was recomputed.
    With the workload's early_exit ([SWD] 3.2 and 4.2: when no position is
    unstable the step may "compute all or end"): a sequence whose active
    rows are all stable after a step that is not its block's last ends the
    block - the later steps of the block refresh none of its rows and
    compute no attention, LM head or update for it (the record's "done"
    lists those sequences; their argmax is -1 and p1 / entropy NaN).
    """
    B, L, H, dh, d = w.batch, w.seq_len, w.n_heads, w.head_dim, w.d_model
    nl, blk = w.n_layers, w.block_len
    tok = tok0.copy()
    stable = np.zeros((B, L), dtype=bool)
    version = np.full((nl, B, L), NEVER, dtype=np.int64)
    tok_w = np.full((B, L), -1, dtype=np.int64)
    swd = SWDState(B, blk)
    caches = tuple(np.zeros((nl, B, L, H, dh)) for _ in range(3))
    pos_all = np.tile(np.arange(L), B)
    flat_all = np.arange(B * L)
    trace = []
    t = 0
    rows_next = None
    fa_key, fa_state = {}, {}
    total = w.n_steps if n_steps is None else min(n_steps, w.n_steps)
    for bi in range(w.n_blocks):
        q0 = w.n_prompt + bi * blk
        ac_flat = (np.arange(B)[:, None] * L + q0 + np.arange(blk)[None, :]).reshape(-1)
        done = np.zeros(B, dtype=bool)            # sequences whose block has ended
        for s in range(w.steps_per_block):
            if t >= total:
                return trace
            rec = {"t": t, "block": bi, "s": s, "q0": q0}
            if keep_pre:
                rec["pre"] = {"tok": tok.copy(), "stable": stable.copy(), "version": version.copy(),
                              "tok_w": tok_w.copy(), "swd": swd.copy(),
                              "caches": tuple(c.copy() for c in caches)}
            full = s == 0 or force_all or mode == "recompute"
            rows = flat_all if full else rows_next          # the refresh set Rf
            rec["rows"] = rows.copy()
            rec["done"] = done.copy()
            live_ac = ac_flat[~done[ac_flat // L]]           # active rows of the sequences still running
            # layer-0 bookkeeping of the refreshed rows
            version[:, rows // L, rows % L] = t
            tok_w.reshape(-1)[rows] = tok.reshape(-1)[rows]
            x_emb = W["embed"][tok.reshape(-1)]                                   # [B*L, d]
            if mode == "recompute":
                o_ac, h_ac = _recompute_step(w, W, x_emb, pos_all, ac_flat)
            elif nl == 1 and not w.ffn:
                q, k, v = M.project_qkv(x_emb[rows], W["w_qkv"][0], rows % L, H, w.dtype,
                                        w.rope_theta, w.rms_eps)
                for c, val in zip(caches, (q, k, v)):
                    c[0].reshape(B * L, H, dh)[rows] = val
                o = np.zeros((B * blk, H, dh))
                rec["fa_rebuilt"] = []
                for b in range(B):
                    if done[b]:
                        continue
                    qa = caches[0][0][b, q0:q0 + blk]
                    kb, vb = caches[1][0][b], caches[2][0][b]
                    if not facache:
                        o[b * blk:(b + 1) * blk] = M.attention(qa, kb, vb)
                        continue
                    win = np.arange(max(0, q0 - w.swd_R), min(L, q0 + blk + w.swd_R))
                    unch = np.setdiff1d(np.arange(L), win)
                    key = (q0, tuple(int(x) for x in tok_w[b, q0:q0 + blk]))
                    if fa_key.get(b) != key:
                        fa_state[b] = M.attention_partial(qa, kb[unch], vb[unch])
                        fa_key[b] = key
                        rec["fa_rebuilt"].append(b)
                    o[b * blk:(b + 1) * blk] = M.merge_partials(
                        [fa_state[b], M.attention_partial(qa, kb[win], vb[win])])
                o_ac = M.round_store(o.reshape(B * blk, d), w.dtype)
                h_ac = M.out_proj(o_ac, W["w_o"][0], x_emb[ac_flat], w.dtype)
            else:
                P = _query_rows(w, rows, live_ac)
                rec["queries"] = P.copy()
                o_p, h_p = _layer_stack(w, W, x_emb[P], P % L, P, caches, np.isin(P, rows))
                o_ac, h_ac = np.zeros((B * blk, d)), np.zeros((B * blk, d))
                live = ~done[ac_flat // L]
                where = np.searchsorted(P, live_ac)
                assert np.array_equal(P[where], live_ac), "active rows must pass through the layers"
                o_ac[live], h_ac[live] = o_p[where], h_p[where]
            am, p1, ent, margin = M.lm_head_conf(h_ac, W["w_lm"], w.mask_id, w.rms_eps)
            gone = done[ac_flat // L]                        # no LM head for ended sequences
            am, p1, ent, margin = (np.where(gone, -1, am).astype(np.int32), np.where(gone, np.nan, p1),
                                   np.where(gone, np.nan, ent), np.where(gone, np.inf, margin))
            am, p1 = am.reshape(B, blk), p1.reshape(B, blk)
            rec.update(argmax=am, p1=p1, ent=ent.reshape(B, blk), margin=margin.reshape(B, blk),
                       o=o_ac.reshape(B, blk, d), h=h_ac.reshape(B, blk, d))
            last = s == w.steps_per_block - 1
            rec["newly"] = swd_update(swd, q0, am, p1, tok, stable, w.swd_K, w.swd_tau, last)
            if w.early_exit and not last:
                done |= stable[:, q0:q0 + blk].all(axis=1)
            if last:
                swd.reset()
                rows_next = flat_all
            elif full_refresh_at(s + 1, w.full_every):
                rows_next = flat_all
            elif w.gate == "confidence":
                rows_next = confidence_rows(stable, tok, tok_w, version, q0, blk, rec["ent"], np.log(w.vocab - 1),
                                            t + 1, w.expiry, w.conf_alpha, w.conf_beta, 3.0 / w.steps_per_block,
                                            w.conf_theta)
            else:
                R_next = radius_at(s + 1, w.steps_per_block, w.swd_R, w.swd_R_min)
                rows_next = refresh_rows(stable, tok, tok_w, version, q0, blk, R_next, t + 1, w.expiry)
            if not last and done.any():                 # ended sequences refresh nothing
                rows_next = rows_next[~done[rows_next // L]]
            partial_next = not last and not full_refresh_at(s + 1, w.full_every)
            rec["stats"] = step_stats(rows_next, stable, rec["newly"], version, q0, blk, L, t + 1, w.expiry, last,
                                      partial_next, done)
            # the row list the next step runs on: Rf, plus the active block of
            # the running sequences when every active row queries (the next
            # step is in this block unless this was its last step, and then
            # Rf is every row)
            nxt_ac = ac_flat if last else ac_flat[~done[ac_flat // L]]
            rec.update(tok=tok.copy(), stable=stable.copy(), version=version.copy(),
                       tok_w=tok_w.copy(), swd=swd.copy(), rf_next=rows_next.copy(),
                       rows_next=_query_rows(w, rows_next, nxt_ac), done_next=done.copy() if not last else
                       np.zeros(B, dtype=bool))
            trace.append(rec)
            t += 1
    return trace


def _query_rows(w, rf, ac_flat):
    """Rows that pass through the layers: the refresh set, plus the active
    rows (of the running sequences) when the workload runs every active row
    as a query."""
    if not w.active_queries or len(rf) == w.batch * w.seq_len:
        return rf.copy()
    return np.union1d(rf, ac_flat).astype(np.int64)


def _recompute_step(w, W, x_emb, pos_all, ac_flat):
    """Plain definition: full forward of every row, no cache."""
    B, L, H, dh, d = w.batch, w.seq_len, w.n_heads, w.head_dim, w.d_model
    x = x_emb
    o_st = None
    for l in range(w.n_layers):
        q, k, v = M.project_qkv(x, W["w_qkv"][l], pos_all, H, w.dtype, w.rope_theta, w.rms_eps)
        last = l == w.n_layers - 1
        qs = (ac_flat if last else np.arange(B * L))
        o = np.zeros((len(qs), H, dh))
        for b in range(B):
            sel = (qs // L) == b
            o[sel] = M.attention(q[qs[sel]], k[b * L:(b + 1) * L], v[b * L:(b + 1) * L])
        o_st = M.round_store(o.reshape(len(qs), d), w.dtype)
        h = M.out_proj(o_st, W["w_o"][l], x[qs], w.dtype)
        if w.ffn:
            h = M.ffn(h, W["w1"][l], W["w2"][l], w.dtype, w.rms_eps)
        x = h
    return o_st, x


class RingSim:
    """Sink + rolling cache bookkeeping of [Sinks] 3.2, one token at a time:
    the first S tokens fill the sinks; every later token is appended to the
    rolling part, which then drops its oldest entry while longer than W."""

    def __init__(self, S, W):
        self.S, self.W = S, W
        self.sinks, self.rolling = [], deque()

    def push(self, pos):
        if len(self.sinks) < self.S:
            self.sinks.append(pos)
            return
        self.rolling.append(pos)
        while len(self.rolling) > self.W:
            self.rolling.popleft()

    def held(self):
        return self.sinks + list(self.rolling)


def ring_positions(n, S, W):
    """Stream positions the sink + rolling cache holds after token n joined."""
    sim = RingSim(S, W)
    for i in range(n + 1):
        sim.push(i)
    return sim.held()


def run_stream(w, W, stream, n_tokens=None, sample=None):
    """Attention-sink stream: for token n, O_n = attention of its query over the
    K/V of the positions the sink + rolling cache holds after n joined.

    Q/K/V of every position are the pure token-level function of (token, pos)
    (one layer, [LaCache] LSM), so they are computed once per position.
    Returns ({n: O_n [H, dh] stored}, {n: held positions}).
    """
    S, Wn, H = w.sink, w.window, w.n_heads
    n_tokens = len(stream) if n_tokens is None else n_tokens
    todo = list(range(n_tokens)) if sample is None else sorted(set(sample))
    want = set(todo)
    held = {}
    sim = RingSim(S, Wn)
    for n in range(todo[-1] + 1):
        sim.push(n)
        if n in want:
            held[n] = sim.held()
    need = np.array(sorted(set().union(*[set(h) for h in held.values()])))
    x = W["embed"][stream[need]]
    q, k, v = M.project_qkv(x, W["w_qkv"][0], need, H, w.dtype, w.rope_theta, w.rms_eps)
    idx = {p: i for i, p in enumerate(need)}
    out = {}
    for n in todo:
        ids = np.array([idx[p] for p in held[n]])
        o = M.attention(q[idx[n]][None], k[ids], v[ids])
        out[n] = M.round_store(o[0], w.dtype)
    return out, held
