"""Pins of the CPU oracle against the pages, closed forms and independent
library routines (no GPU).  A plausible slip anywhere in the oracle (a dropped
term, a wrong sign or index, a transposed operand) fails one of these."""
import itertools
import math

import numpy as np
import pytest
from scipy import special, stats

import oracle as O
from conftest import parse_ranges, read_golden
from workloads import configs as C
from workloads import generate as G

RNG = np.random.default_rng(1234)


# --- storage rounding ---------------------------------------------------------
def test_bf16_round_ties_and_cases():
    one = 1.0
    cases = [
        (one + 2.0 ** -8, one),                          # tie -> even (down)
        (one + 3 * 2.0 ** -8, one + 2.0 ** -6),          # tie -> even (up)
        (one + 2.0 ** -8 + 2.0 ** -20, one + 2.0 ** -7),  # above the tie -> up
        (-(one + 2.0 ** -8 + 2.0 ** -20), -(one + 2.0 ** -7)),
        (3.0, 3.0), (0.0, 0.0),
    ]
    for x, want in cases:
        assert O.round_store(np.array([x]), "bf16")[0] == want


def test_bf16_round_matches_independent_fp32_encoder():
    # The input generator encodes fp32 -> bf16 from the fp32 bit pattern; the
    # oracle rounds fp64 at bit 45.  For fp32 inputs the two must agree.
    x = (RNG.standard_normal(20000) * np.exp(RNG.uniform(-20, 20, 20000))).astype(np.float32)
    a = O.round_store(x.astype(np.float64), "bf16")
    b = O.bf16_bits_to_f64(G.f32_to_bf16_bits(x))
    assert np.array_equal(a, b)


# --- normalisation, RoPE, GELU -----------------------------------------------------
def test_rms_scale_closed_form():
    x = RNG.standard_normal((7, 64)) * 3.0
    y = x * O.rms_scale(x, eps=0.0)
    assert np.allclose(np.sqrt(np.mean(y * y, axis=1)), 1.0, rtol=1e-13)
    assert np.allclose(O.rms_scale(5.0 * x, 0.0) * 5.0, O.rms_scale(x, 0.0), rtol=1e-13)


def test_rope_identity_at_zero_and_complex_form():
    H, dh = 3, 16
    x = RNG.standard_normal((5, H, dh))
    assert np.array_equal(O.rope(x, np.zeros(5, dtype=int)), x)
    pos = np.array([0, 1, 7, 100, 4095])
    y = O.rope(x, pos, theta=10000.0)
    # independent formulation: pair (x_i, x_{i+dh/2}) as a complex number
    # multiplied by exp(i * pos * theta^(-2i/dh))
    half = dh // 2
    z = x[..., :half] + 1j * x[..., half:]
    freq = 10000.0 ** (-np.arange(0, dh, 2) / dh)
    zr = z * np.exp(1j * pos[:, None, None] * freq[None, None, :])
    assert np.allclose(y[..., :half], zr.real, atol=1e-12)
    assert np.allclose(y[..., half:], zr.imag, atol=1e-12)


def test_rope_relative_position_property():
    # <rope(q, m), rope(k, n)> depends only on m - n
    q = RNG.standard_normal((1, 1, 32))
    k = RNG.standard_normal((1, 1, 32))
    d0 = np.sum(O.rope(q, [5]) * O.rope(k, [2]))
    d1 = np.sum(O.rope(q, [105]) * O.rope(k, [102]))
    d2 = np.sum(O.rope(q, [6]) * O.rope(k, [2]))
    assert abs(d0 - d1) < 1e-12
    assert abs(d0 - d2) > 1e-6
    assert np.allclose(np.linalg.norm(O.rope(q, [77])), np.linalg.norm(q))


def test_gelu_closed_form():
    xs = np.array([-3.0, -1.0, -0.5, 0.0, 0.25, 1.0, 2.0])
    want = np.array([x * 0.5 * (1 + math.erf(x / math.sqrt(2))) for x in xs])
    assert np.allclose(O.gelu(xs), want, atol=1e-15)
    assert np.allclose(O.gelu(xs) - O.gelu(-xs), xs, atol=1e-15)


# --- projection ---------------------------------------------------------------------
def test_project_qkv_with_permutation_weights():
    # W_qkv = [P; I; 2I] with P a non-symmetric permutation: q = rope(P xn),
    # k = rope(xn), v = 2 xn.  A transposed operand gives P^T instead of P.
    H, dh = 2, 8
    d = H * dh
    perm = RNG.permutation(d)
    P = np.eye(d)[perm]
    assert not np.array_equal(P, P.T)
    W = np.concatenate([P, np.eye(d), 2 * np.eye(d)])
    x = RNG.standard_normal((3, d))
    pos = np.array([0, 3, 9])
    q, k, v = O.project_qkv(x, W, pos, H, "f32", 10000.0, 1e-6)
    xn = x / np.sqrt(np.mean(x * x, axis=1, keepdims=True) + 1e-6)
    f32 = lambda a: a.astype(np.float32).astype(np.float64)
    assert np.allclose(q, f32(O.rope(xn[:, perm].reshape(3, H, dh), pos)), atol=1e-6)
    assert np.allclose(k, f32(O.rope(xn.reshape(3, H, dh), pos)), atol=1e-6)
    assert np.allclose(v, f32(2 * xn.reshape(3, H, dh)), atol=1e-6)


# --- attention ------------------------------------------------------------------------
def test_attention_single_key_and_identical_keys():
    q = RNG.standard_normal((4, 2, 8))
    k = RNG.standard_normal((1, 2, 8))
    v = RNG.standard_normal((1, 2, 8))
    assert np.allclose(O.attention(q, k, v), np.broadcast_to(v, (4, 2, 8)), atol=1e-15)
    kk = np.repeat(k, 6, axis=0)
    vv = RNG.standard_normal((6, 2, 8))
    assert np.allclose(O.attention(q, kk, vv), vv.mean(axis=0)[None], atol=1e-14)


def test_attention_vs_scipy_softmax_and_permutation():
    q = RNG.standard_normal((5, 3, 16))
    k = RNG.standard_normal((40, 3, 16))
    v = RNG.standard_normal((40, 3, 16))
    o = O.attention(q, k, v)
    for h in range(3):
        w = special.softmax(q[:, h] @ k[:, h].T / 4.0, axis=1)
        assert np.allclose(o[:, h], w @ v[:, h], atol=1e-13)
    p = RNG.permutation(40)
    assert np.allclose(O.attention(q, k[p], v[p]), o, atol=1e-13)
    # queries are independent (no causal mask, no mixing across queries)
    assert np.allclose(O.attention(q[2:3], k, v), o[2:3], atol=1e-14)


def test_out_proj_and_ffn_reduce():
    x = O.round_store(RNG.standard_normal((3, 8)), "bf16")
    o = RNG.standard_normal((3, 8))
    assert np.array_equal(O.out_proj(o, np.zeros((8, 8)), x, "bf16"), x)
    ws = np.diag(np.arange(1, 9, dtype=float))
    h = O.out_proj(o, ws, x, "f32")
    want = (x + O.round_store(o, "f32") * np.arange(1, 9)).astype(np.float32)
    assert np.allclose(h, want, atol=1e-6)
    assert np.array_equal(O.ffn(x, np.ones((4, 8)), np.zeros((8, 4)), "bf16"), x)


def _bf16_rne(x):
    """Round one float to bf16 (8 significant bits, ties to even), written
    from frexp and Python's round() (which rounds halves to even)."""
    if x == 0.0 or not math.isfinite(x):
        return x
    m, e = math.frexp(x)                 # x = m * 2^e, 0.5 <= |m| < 1
    return round(m * 256.0) / 256.0 * 2.0 ** e


def _gelu_erf(x):
    return 0.5 * x * (1.0 + math.erf(x / math.sqrt(2.0)))


def test_ffn_closed_form_with_selection_weights():
    """FFN = h + W2 . store(GELU(W1 . RMSNorm(h))) pinned by weights that
    select entries: W1 row j picks input a[j] (rows past d are zero), W2 row i
    adds 2 f[b[i]] - f[c[i]].  The expected rows come from scalar code; the
    alternatives that a slip would give (no norm, GELU after W2, no bf16 store
    of the GELU output, a transposed W1) differ from it."""
    d, F, n = 64, 96, 6
    rng = np.random.default_rng(77)
    h = O.round_store(rng.standard_normal((n, d)) * 3.0, "bf16")
    a = rng.permutation(d)
    b = rng.permutation(d)
    c = (b + 1 + rng.integers(0, d - 1, d)) % d          # c[i] != b[i]
    w1 = np.zeros((F, d))
    w1[np.arange(d), a] = 1.0
    w2 = np.zeros((d, F))
    w2[np.arange(d), b] = 2.0
    w2[np.arange(d), c] = -1.0
    got = O.ffn(h, w1, w2, "bf16", eps=1e-6)

    def expect(norm=True, store=True, gelu_after=False, w1_t=False):
        out = np.zeros((n, d))
        pick = np.argsort(a) if w1_t else a
        for r in range(n):
            row = [float(x) for x in h[r]]
            scale = 1.0 / math.sqrt(math.fsum(x * x for x in row) / d + 1e-6) if norm else 1.0
            x1 = [scale * row[pick[j]] for j in range(d)]     # W1 . (norm h), first d rows
            if gelu_after:
                f = [2.0 * x1[b[i]] - x1[c[i]] for i in range(d)]
                out[r] = [_bf16_rne(row[i] + _gelu_erf(f[i])) for i in range(d)]
                continue
            g = [_gelu_erf(v) for v in x1]
            g = [_bf16_rne(v) for v in g] if store else g
            out[r] = [_bf16_rne(row[i] + 2.0 * g[b[i]] - g[c[i]]) for i in range(d)]
        return out

    want = expect()
    assert np.array_equal(got, want)
    for slip in (dict(norm=False), dict(store=False), dict(gelu_after=True), dict(w1_t=True)):
        assert not np.array_equal(expect(**slip), want), slip


def test_bf16_scalar_rounding_agrees_with_the_oracle():
    x = RNG.standard_normal(2000) * np.exp(RNG.uniform(-10, 10, 2000))
    assert np.array_equal(O.round_store(x, "bf16"), np.array([_bf16_rne(float(v)) for v in x]))


# --- LM head confidence ----------------------------------------------------------------------
def test_lm_head_uniform_logits():
    V = 50
    h = RNG.standard_normal((4, 8))
    am, p1, ent, _ = O.lm_head_conf(h, np.zeros((V, 8)), mask_id=0)
    assert np.all(am == 1)                          # lowest id other than the mask
    assert np.allclose(p1, 1.0 / (V - 1))
    assert np.allclose(ent, np.log(V - 1))


def test_lm_head_vs_scipy_and_mask_exclusion():
    V, d = 300, 16
    h = RNG.standard_normal((6, d))
    W = RNG.standard_normal((V, d)) * 0.7
    W[0] = 10 * h.mean(axis=0)                      # make the mask id's logit large
    am, p1, ent, margin = O.lm_head_conf(h, W, mask_id=0)
    hn = h / np.sqrt(np.mean(h * h, axis=1, keepdims=True) + 1e-6)
    lg = hn @ W.T
    lg_ex = lg[:, 1:]
    p = special.softmax(lg_ex, axis=1)
    assert np.all(am != 0)
    assert np.array_equal(am, np.argmax(lg_ex, axis=1) + 1)
    assert np.allclose(p1, p.max(axis=1), rtol=1e-12)
    assert np.allclose(ent, stats.entropy(p, axis=1), rtol=1e-10)
    assert np.all(ent >= 0) and np.all(ent <= np.log(V - 1) + 1e-12)
    srt = np.sort(lg_ex, axis=1)
    assert np.allclose(margin, srt[:, -1] - srt[:, -2])


def test_lm_head_tie_goes_to_lowest_index():
    W = np.zeros((10, 4))
    W[3] = W[7] = [1, 0, 0, 0]
    am, _, _, margin = O.lm_head_conf(np.array([[1.0, 0.5, 0.5, 0.5]]), W, mask_id=0)
    assert am[0] == 3 and margin[0] == 0.0


# --- SWD stability rule: brute force over small histories --------------------------------------
def _drive(tokens, probs, K, tau):
    """Feed one position's per-step (token, prob) into the oracle; return the
    step at which it became stable (or None) and the committed token."""
    st = O.SWDState(1, 1)
    tok = np.zeros((1, 1), dtype=np.int64)
    stable = np.zeros((1, 1), dtype=bool)
    when = None
    for i, (a, p) in enumerate(zip(tokens, probs)):
        was = bool(stable[0, 0])
        O.swd_update(st, 0, np.array([[a]]), np.array([[p]]), tok, stable, K, tau, False)
        if was:
            assert stable[0, 0]                       # absorbing
        if stable[0, 0] and when is None:
            when = i
    return when, int(tok[0, 0])


def _first_run_end(tokens, K):
    """First index where a run of K equal tokens ends (itertools.groupby)."""
    i = 0
    for _, grp in itertools.groupby(tokens):
        n = len(list(grp))
        if n >= K:
            return i + K - 1
        i += n
    return None


@pytest.mark.parametrize("K", [1, 2, 3, 4])
def test_swd_brute_force_low_tau_is_run_length(K):
    # tau below every probability: stable exactly when the first run of K
    # equal top-1 tokens completes; the committed token is that run's token.
    for n in range(1, 7):
        for toks in itertools.product([1, 2, 3], repeat=n):
            when, tok = _drive(toks, [0.5] * n, K, tau=0.1)
            want = _first_run_end(toks, K)
            assert when == want, (toks, K)
            if want is not None:
                assert tok == toks[want]


def test_swd_brute_force_constant_prob_threshold():
    # constant probability c, constant token: stable at step K-1 iff c > tau
    grid = [0.85, 0.9, 0.9 + 1e-6, 0.95]
    for K in (1, 2, 3):
        for c in grid:
            when, _ = _drive([5] * 6, [c] * 6, K, tau=0.9)
            assert when == (K - 1 if np.float32(c) > np.float32(0.9) else None), (K, c)


def test_swd_brute_force_mean_over_last_K_only():
    # K = 3, tau = 0.9: probabilities enter the mean only while in the window
    rng = np.random.default_rng(7)
    for _ in range(3000):
        n = rng.integers(1, 8)
        toks = rng.integers(1, 3, size=n)
        ps = rng.choice([0.6, 0.85, 0.9, 0.95, 0.99], size=n)
        when, _ = _drive(list(toks), list(ps), 3, 0.9)
        # independent statement of the page's formula over full arrays
        first = None
        for t in range(2, n):
            same = toks[t - 2] == toks[t - 1] == toks[t]
            mean = np.float32(np.float32(np.float32(ps[t - 2]) + np.float32(ps[t - 1])) + np.float32(ps[t])) / np.float32(3)
            if same and mean > np.float32(0.9):
                first = t
                break
        assert when == first, (toks, ps)


def test_swd_forced_commit_at_last_step():
    st = O.SWDState(1, 4)
    tok = np.zeros((1, 10), dtype=np.int64)
    stable = np.zeros((1, 10), dtype=bool)
    stable[0, 5] = True
    tok[0, 5] = 99
    O.swd_update(st, 4, np.array([[11, 12, 13, 14]]), np.full((1, 4), 0.1), tok, stable, 3, 0.9, True)
    assert list(tok[0, 4:8]) == [11, 99, 13, 14]       # stable row keeps its commit
    assert list(tok[0, :4]) == [0, 0, 0, 0]


# --- dilation, expiry, refresh set --------------------------------------------------------
def test_dilation_page_example():
    g = read_golden("swd_dilation_L20.txt")
    L = int(g["L"])
    stable1 = set(parse_ranges(g["stable"]))
    unstable0 = [p - 1 for p in range(1, L + 1) if p not in stable1]
    assert [p + 1 for p in unstable0] == parse_ranges(g["unstable_windows"])
    for R in (0, 1, 2, 5):
        m = O.dilate(unstable0, R, L)
        assert [i + 1 for i in np.flatnonzero(m)] == parse_ranges(g[f"window_R{R}"]), R


def test_dilation_vs_convolution():
    rng = np.random.default_rng(3)
    for _ in range(500):
        L = int(rng.integers(1, 40))
        R = int(rng.integers(0, 4))
        u = rng.random(L) < 0.2
        m = O.dilate(np.flatnonzero(u), R, L)
        conv = np.convolve(u.astype(int), np.ones(2 * R + 1, dtype=int), mode="same")[:L] > 0
        if 2 * R + 1 > L:     # np.convolve 'same' centres on the longer input
            conv = np.array([u[max(0, i - R):i + R + 1].any() for i in range(L)])
        assert np.array_equal(m, conv)


def test_version_expiry_page_rule():
    g = read_golden("version_expiry.txt")
    thr = int(g["threshold"])
    for case in g["case"]:
        t, v, rej = (int(s) for s in case.split(","))
        ver = np.full((1, 1, 1), v)
        assert bool(O.expired_rows(ver, t, thr)[0, 0]) == bool(rej), case
    assert not O.expired_rows(np.zeros((1, 1, 1)), 100, -1).any()


def test_refresh_rows_composition():
    B, L = 2, 12
    tok = np.ones((B, L), dtype=np.int64)
    tok_w = tok.copy()
    stable = np.zeros((B, L), dtype=bool)
    stable[:, 4:8] = True
    stable[0, 5] = False                 # one unstable active row in sequence 0
    tok[1, 1] = 7                        # a changed row in sequence 1
    version = np.full((1, B, L), 10)
    version[0, 0, 11] = 7                # expired at t=10 with expiry 2
    rows = O.refresh_rows(stable, tok, tok_w, version, 4, 4, 1, 10, 2)
    assert list(rows) == [4, 5, 6, 11, 12 + 1]


def test_radius_schedule_and_full_refresh_steps():
    # fixed radius unless a starting radius is given
    assert [O.radius_at(s, 32, 2, -1) for s in (0, 15, 31)] == [2, 2, 2]
    # 0 -> 2 over 32 steps in three equal stages; monotone, ends at R
    rs = [O.radius_at(s, 32, 2, 0) for s in range(32)]
    assert rs[0] == 0 and rs[-1] == 2 and all(a <= b for a, b in zip(rs, rs[1:]))
    assert [rs.count(r) for r in (0, 1, 2)] == [11, 11, 10]
    assert [O.radius_at(s, 10, 3, 1) for s in range(10)] == [1, 1, 1, 1, 2, 2, 2, 3, 3, 3]
    assert [s for s in range(12) if O.full_refresh_at(s, 4)] == [0, 4, 8]
    assert not any(O.full_refresh_at(s, 0) for s in range(12))


def test_schedules_shape_the_refresh_sets():
    """mid_bf16_sched: every 4th step of a block refreshes every row; the
    other steps dilate the unstable rows by the scheduled radius."""
    w, W, tok0 = _load("mid_bf16_sched")
    tr = O.run_dense(w, W, tok0, mode="cached")
    full = w.batch * w.seq_len
    saw_partial = 0
    for prev, r in zip(tr[:-1], tr[1:]):
        s = r["s"]
        if s == 0 or s % w.full_every == 0:
            assert len(r["rows"]) == full, (r["t"], s)
            continue
        R = O.radius_at(s, w.steps_per_block, w.swd_R, w.swd_R_min)
        want = O.refresh_rows(prev["stable"], prev["tok"], prev["tok_w"], prev["version"], r["q0"], w.block_len, R,
                              r["t"], w.expiry)
        assert np.array_equal(r["rows"], want), (r["t"], s)
        saw_partial += len(r["rows"]) < full
    assert saw_partial > 0


def test_confidence_closed_form_and_rows():
    """[FlashdLLM] 3.1: alpha (1 - H / H_max) + beta exp(-lambda age), against
    scalar code; the rows are the unstable active positions below theta, plus
    changed and expired rows."""
    H_max = math.log(999.0)
    for ent, age in ((0.0, 0), (H_max, 0), (2.5, 3), (6.0, 10)):
        want = 0.7 * (1.0 - ent / H_max) + 0.3 * math.exp(-0.3 * age)
        assert abs(float(O.confidence(ent, H_max, age, 0.7, 0.3, 0.3)) - want) < 1e-6
    B, L, q0, blk = 1, 12, 4, 4
    stable = np.zeros((B, L), dtype=bool)
    stable[0, 5] = True
    tok = np.ones((B, L), dtype=np.int64)
    tok_w = tok.copy()
    tok_w[0, 10] = 3                                     # a changed row
    version = np.full((1, B, L), 9)
    version[0, 0, 7] = 2                                 # an old entry: low confidence
    ent = np.array([[6.5, 0.1, 0.2, 0.2]])               # position 4 is unsure, 5 stable, 6 and 7 sure
    rows = O.confidence_rows(stable, tok, tok_w, version, q0, blk, ent, H_max, 10, -1, 0.7, 0.3, 0.3, 0.5)
    # 4: 0.7 * 0.06 + 0.3 e^-0.3 < 0.5; 6: 0.68 + ...; 7: 0.68 + 0.3 e^-2.4 > 0.5; 10: changed
    assert list(rows) == [4, 10]
    ent2 = np.array([[6.5, 0.1, 0.2, 4.9]])             # 7: 0.7 * 0.29 + 0.3 e^-2.4 < 0.5
    assert list(O.confidence_rows(stable, tok, tok_w, version, q0, blk, ent2, H_max, 10, -1, 0.7, 0.3, 0.3,
                                  0.5)) == [4, 7, 10]


def test_confidence_gate_loop():
    """mid_bf16_conf: every partial step's refresh set is the confidence
    rule applied to the step's entropies and versions; some steps refresh a
    part of the block only, and some positions commit."""
    w, W, tok0 = _load("mid_bf16_conf")
    tr = O.run_dense(w, W, tok0, mode="cached")
    partial = 0
    for prev, r in zip(tr[:-1], tr[1:]):
        if r["s"] == 0:
            continue
        want = O.confidence_rows(prev["stable"], prev["tok"], prev["tok_w"], prev["version"], r["q0"], w.block_len,
                                 prev["ent"], np.log(w.vocab - 1), r["t"], w.expiry, w.conf_alpha, w.conf_beta,
                                 3.0 / w.steps_per_block, w.conf_theta)
        assert np.array_equal(r["rows"], want), r["t"]
        partial += 0 < len(r["rows"]) < w.batch * w.block_len
    assert partial > 0 and sum(int(r["newly"].sum()) for r in tr) > 0


@pytest.mark.parametrize("name", ["mid_bf16_exit", "mid_multi_exit"])
def test_early_exit_changes_no_token(name):
    """A sequence whose active rows are all stable ends its block: its later
    steps refresh nothing and compute nothing, and every token of every step
    equals the run without early exit (stable positions never change)."""
    from dataclasses import replace
    w, W, tok0 = _load(name)
    a = O.run_dense(w, W, tok0, mode="cached")
    b = O.run_dense(replace(w, early_exit=0), W, tok0, mode="cached")
    L, blk = w.seq_len, w.block_len
    ended = 0
    for ra, rb in zip(a, b):
        assert np.array_equal(ra["tok"], rb["tok"]), ra["t"]
        assert np.array_equal(ra["stable"], rb["stable"]), ra["t"]
        for s in np.flatnonzero(ra["done"]):
            ended += 1
            assert ra["stable"][s, ra["q0"]:ra["q0"] + blk].all()
            assert not np.any(ra["rows"] // L == s)                  # nothing of it refreshed
            assert np.all(ra["argmax"][s] == -1)
        assert len(ra["rows"]) <= len(rb["rows"])
    assert ended > 0


def test_multilayer_queries_and_kv_gate():
    """Multi-layer denoiser: the rows that pass through the layers are the
    refresh set plus the active block, and only refresh-set rows rewrite K/V
    and versions; an active row that is stable and outside the refresh set
    queries every layer but leaves its cached K/V and version untouched."""
    w, W, tok0 = _load("mid_multi_sharp")
    tr = O.run_dense(w, W, tok0, mode="cached", keep_pre=True)
    B, L, blk, H, dh = w.batch, w.seq_len, w.block_len, w.n_heads, w.head_dim
    gated = 0
    for r in tr:
        ac = (np.arange(B)[:, None] * L + r["q0"] + np.arange(blk)[None, :]).reshape(-1)
        assert np.array_equal(r["queries"], np.union1d(r["rows"], ac))
        quiet = np.setdiff1d(ac, r["rows"])             # query-only rows of this step
        if r["s"] == 0 or not len(quiet):
            continue
        nxt = next((x for x in tr if x["t"] == r["t"] + 1), None)
        if nxt is None:
            continue
        pre, post = r["pre"], nxt["pre"]
        for f in (1, 2):                                 # K and V
            a = pre["caches"][f].reshape(w.n_layers, B * L, H, dh)[:, quiet]
            bq = post["caches"][f].reshape(w.n_layers, B * L, H, dh)[:, quiet]
            assert np.array_equal(a, bq)
        assert np.array_equal(pre["version"].reshape(w.n_layers, -1)[:, quiet],
                              r["version"].reshape(w.n_layers, -1)[:, quiet])
        gated += len(quiet)
    assert gated > 0


def test_split_kv_merge_equals_single_pass():
    """The online-softmax states over disjoint key sets merge into the plain
    attention over their union (the split-KV identity FACache rests on); an
    empty part contributes nothing; one key gives m = s, l = 1, O~ = v."""
    q = RNG.standard_normal((5, 3, 16))
    k = RNG.standard_normal((40, 3, 16)) * 2.0
    v = RNG.standard_normal((40, 3, 16))
    want = O.attention(q, k, v)
    for cut in ([0, 40], [0, 1, 40], [0, 13, 13, 29, 40], [0, 39, 40]):
        parts = [O.attention_partial(q, k[a:b], v[a:b]) for a, b in zip(cut[:-1], cut[1:])]
        assert np.allclose(O.merge_partials(parts), want, rtol=1e-13, atol=1e-14), cut
    idx = RNG.permutation(40)                                   # not contiguous
    parts = [O.attention_partial(q, k[idx[:17]], v[idx[:17]]), O.attention_partial(q, k[idx[17:]], v[idx[17:]])]
    assert np.allclose(O.merge_partials(parts), want, rtol=1e-13, atol=1e-14)
    m, l, o = O.attention_partial(q[:1], k[:1], v[:1])
    assert np.allclose(m[:, 0], np.einsum("hd,hd->h", q[0], k[0]) / 4.0)
    assert np.array_equal(l, np.ones_like(l)) and np.allclose(o[0], v[0])


@pytest.mark.parametrize("name", ["mid_bf16", "mid_bf16_sharp", "mid_bf16_dh64"])
def test_facache_loop_equals_the_plain_loop(name):
    """Reusing the kept softmax state changes nothing but rounding order:
    the same tokens, argmaxes and stability at every step, outputs to 1e-6;
    the state is rebuilt for every sequence at each block start and
    otherwise only after one of its block's tokens changed."""
    w, W, tok0 = _load(name)
    a = O.run_dense(w, W, tok0, mode="cached")
    b = O.run_dense(w, W, tok0, mode="cached", facache=True)
    for ra, rb in zip(a, b):
        for key in ("argmax", "tok", "stable"):
            assert np.array_equal(ra[key], rb[key]), (name, ra["t"], key)
        assert np.allclose(ra["o"], rb["o"], rtol=1e-6, atol=1e-9)
        assert np.allclose(ra["p1"], rb["p1"], rtol=1e-9)
    for prev, rb in zip(b[:-1], b[1:]):
        q0, blk = rb["q0"], w.block_len
        if rb["s"] == 0:
            assert rb["fa_rebuilt"] == list(range(w.batch))
        else:      # the key: the active rows' token-at-write when the attention ran
            changed = [bb for bb in range(w.batch)
                       if not np.array_equal(rb["tok_w"][bb, q0:q0 + blk], prev["tok_w"][bb, q0:q0 + blk])]
            assert rb["fa_rebuilt"] == changed, (name, rb["t"])
    assert b[0]["fa_rebuilt"] == list(range(w.batch))
    if name == "mid_bf16":                          # nothing commits inside a block
        assert all(rb["fa_rebuilt"] == [] for rb in b if rb["s"] > 0)
    if name == "mid_bf16_sharp":
        assert any(rb["fa_rebuilt"] for rb in b if rb["s"] > 0)


# --- whole-loop pins (refresh-all == recompute; unchanged => identical K/V) ---------------
def _load(name):
    w = C.get(name)
    return w, O.weights_f64(w, G.model(w)), G.prompt_tokens(w)


@pytest.mark.parametrize("name", ["tiny_fp32", "mid_multi"])
def test_refresh_all_equals_recompute(name):
    w, W, tok0 = _load(name)
    a = O.run_dense(w, W, tok0, n_steps=8, mode="cached", force_all=True)
    b = O.run_dense(w, W, tok0, n_steps=8, mode="recompute")
    for ra, rb in zip(a, b):
        for key in ("argmax", "p1", "ent", "o", "h", "tok", "stable"):
            assert np.array_equal(ra[key], rb[key]), (name, ra["t"], key)


@pytest.mark.parametrize("name", ["tiny_fp32_sharp", "mid_bf16_sharp"])
def test_single_layer_cached_equals_recompute(name):
    w, W, tok0 = _load(name)
    a = O.run_dense(w, W, tok0, mode="cached")
    b = O.run_dense(w, W, tok0, mode="recompute")
    assert sum(int(r["newly"].sum()) for r in a) > 0          # commits happened
    assert any(len(r["rows"]) < w.batch * w.seq_len for r in a)
    for ra, rb in zip(a, b):
        for key in ("argmax", "p1", "ent", "o", "h", "tok"):
            assert np.array_equal(ra[key], rb[key]), (name, ra["t"], key)


def test_unchanged_tokens_have_identical_cached_kv():
    w, W, tok0 = _load("mid_bf16_sharp")
    tr = O.run_dense(w, W, tok0, mode="cached", keep_pre=True)
    L, H, dh = w.seq_len, w.n_heads, w.head_dim
    checked = 0
    for r in tr[1:]:
        pre = r["pre"]
        same = (pre["tok"] == pre["tok_w"]).reshape(-1)
        rows = np.flatnonzero(same)
        x = W["embed"][pre["tok"].reshape(-1)[rows]]
        q, k, v = O.project_qkv(x, W["w_qkv"][0], rows % L, H, w.dtype)
        for c, val in zip(pre["caches"], (q, k, v)):
            assert np.array_equal(c[0].reshape(-1, H, dh)[rows], val)
        checked += len(rows)
    assert checked > 0


def test_block_start_and_expiry_refresh_pattern():
    # with nothing stable and expiry 2, block-local steps 0, 3, 6, ... refresh
    # every row; the others refresh the dilated active block only
    w, W, tok0 = _load("mid_bf16")
    tr = O.run_dense(w, W, tok0, mode="cached")
    full = w.batch * w.seq_len
    for r in tr:
        if r["s"] % 3 == 0:
            assert len(r["rows"]) == full
        else:
            lo = max(0, r["q0"] - w.swd_R)
            hi = min(w.seq_len - 1, r["q0"] + w.block_len - 1 + w.swd_R)
            assert len(r["rows"]) == w.batch * (hi - lo + 1)


# --- sink + rolling cache --------------------------------------------------------------------
def test_sink_ring_page_example():
    g = read_golden("sink_s3_c7.txt")
    S, Cmax, W = int(g["attention_sinks"]), int(g["max_cache_length"]), int(g["rolling_window"])
    assert W == Cmax - S
    shape = [int(s) for s in g["k_cache_shape"].split(",")]
    assert shape[2] == Cmax
    sim = O.RingSim(S, W)
    for n in range(60):
        sim.push(n)
        held = sim.held()
        assert len(held) == min(n + 1, S + W)              # constant S+W after warm-up
        assert held[:min(S, n + 1)] == list(range(min(S, n + 1)))   # sinks never move
        assert held == list(range(S)) + list(range(max(S, n - W + 1), n + 1)) or n < S


def test_sink_stream_outputs_bit_stable_sinks():
    w = C.get("mid_sink")
    W = O.weights_f64(w, G.model(w))
    stream = G.stream_tokens(w)
    out, held = O.run_stream(w, W, stream, n_tokens=w.stream_len)
    S = w.sink
    for n, h in held.items():
        assert len(h) == min(n + 1, w.sink + w.window)
    # the first query attends to itself only: O_0 = v_0
    x = W["embed"][stream[:1]]
    _, _, v0 = O.project_qkv(x, W["w_qkv"][0], np.array([0]), w.n_heads, w.dtype)
    assert np.array_equal(out[0], O.round_store(v0[0], w.dtype))
    assert all(h[:S] == list(range(S)) for n, h in held.items() if n >= S)


@pytest.mark.parametrize("name", ["mid_bf16", "mid_bf16_sharp", "mid_bf16_exit", "mid_bf16_sched"])
def test_step_stats_stability_curve(name):
    """The per-step counters against what they count, independently: each
    block commits every position of every sequence exactly once (by
    stability or at its last step); the stable count never falls inside a
    block and grows by exactly the positions committed by stability; the
    refresh count is the next step's refresh set per sequence; expired rows
    are a subset of it and vanish when expiry is off."""
    w, W, tok0 = _load(name)
    tr = O.run_dense(w, W, tok0, mode="cached")
    B, L, blk = w.batch, w.seq_len, w.block_len
    prev_stable = np.zeros(B, dtype=np.int64)
    committed = np.zeros(B, dtype=np.int64)
    for i, r in enumerate(tr):
        st = r["stats"]
        if r["s"] == 0:
            prev_stable[:] = 0
            committed[:] = 0
        last = r["s"] == w.steps_per_block - 1
        for b in range(B):
            assert st[b, 0] == np.sum(r["rf_next"] // L == b), (r["t"], b)
            assert st[b, 2] <= st[b, 0]
            if w.expiry < 0:
                assert st[b, 2] == 0
            assert st[b, 1] >= prev_stable[b]                       # stable is absorbing
            assert st[b, 1] == int(r["stable"][b, r["q0"]:r["q0"] + blk].sum())
            by_stability = st[b, 1] - prev_stable[b]
            assert st[b, 3] == by_stability + (blk - st[b, 1] if last else 0)
        prev_stable[:] = st[:, 1]
        committed += st[:, 3]
        if last:
            assert np.all(committed == blk), (r["t"], committed)
            assert np.all(st[:, 0] == L)                             # the next block starts with a full refresh
    if name != "mid_bf16":
        assert sum(int(r["stats"][:, 1].sum()) for r in tr) > 0      # something stabilises
    if w.expiry >= 0 and name == "mid_bf16":
        assert sum(int(r["stats"][:, 2].sum()) for r in tr) > 0      # expired rows occur


def test_sharp_variants_exercise_swd():
    for name in ("tiny_fp32_sharp", "mid_bf16_sharp"):
        w, W, tok0 = _load(name)
        tr = O.run_dense(w, W, tok0, mode="cached")
        assert sum(int(r["newly"].sum()) for r in tr) >= 8, name


# --- the multi-layer quality figure (cached loop against full recompute) -----
def test_drift_is_zero_where_the_cache_is_exact():
    """Reuse is exact in the first layer, so a one-layer model drifts nowhere;
    with several layers nothing drifts while no token changes inside a block
    (the stale deeper-layer K/V then equal the recomputed ones), and every
    block's first step is a full refresh in both loops."""
    from oracle.drift import drift
    for name in ("mid_bf16_sharp", "mid_multi"):
        w = C.get(name)
        steps, tok_agree, first = drift(w, G.model(w), G.prompt_tokens(w))
        assert all(r["max_dp1"] == 0.0 and r["argmax_agree"] == 1.0 for r in steps), name
        assert tok_agree == 1.0 and first is None, name
    w = C.get("mid_multi_sharp")
    steps, _, _ = drift(w, G.model(w), G.prompt_tokens(w))
    assert all(r["max_dp1"] == 0.0 for r in steps if r["s"] == 0)
    assert any(r["max_dp1"] > 0.0 for r in steps)          # commits inside a block: stale K/V
