"""Oracle of the Stable-Window-Decoding bookkeeping and the refresh set.

Sources, cited by page title and section:
  [SWD]  "Stable Window Decoding" page (wmrh.cn/news/51151):
         3.1  the stability criterion: position i is stable at step t when its
              top-1 token was the same over the last K steps and the mean of
              those K top-1 probabilities exceeds tau;
         3.2  the computation window: every unstable position u contributes
              [u-R, u+R], clipped to the sequence; worked example L = 20;
         3.3  the algorithm: a position already in the stable set is skipped;
         4.2  the scheduler: a per-position history trimmed to its last K
              (token, prob) records; the test runs once K records exist.
  [TA]   "Diffusion latent cache with time anchors" page (mhpq.cn/news/1098081),
         2.3 and 3.1: every cache entry carries the step it was written at; a
         lookup at step t rejects it when t - version > 2.
  [FlashdLLM] "I/O-aware KV cache and self-verifying parallel decoding"
         (bjdmk.com.cn/news/5926815), 3.1: the cache confidence of position i
         at step t, alpha (1 - H_i / H_max) + beta exp(-lambda (t - t_write));
         alpha ~ 0.7, beta ~ 0.3, lambda ~ 3 / T.
  [LaCache] "Problem statement" / "Inference workflow": the prompt and the
         masked suffix keep their token ids inside a block; the block's first
         step runs a full forward and refills the caches.

Readings (also listed in the design notes):
  * "exceeds" is strict: mean > tau; the mean is (sum oldest->newest)/K in fp32;
  * a position that becomes stable commits its top-1 token (masked diffusion
    freezes a stable position by unmasking it); at the block's last step every
    position still unstable commits its top-1 token;
  * unstable = active-block positions not yet stable (prompt, committed and
    future masked positions keep fixed ids inside a block);
  * the all-stable case adds no window (the page's "compute all" is one of two
    options it offers; the other, ending, is what a fixed Tb gives);
  * t is the global step counter; refresh set for step t+1 =
      dilate_R(unstable) U {p : tok[p] != token the entry was computed from}
      U {p : (t+1) - version[p] > expiry}.
  * schedules ([SWD] 4.4: R may grow along the sampling steps, small or 0
    early and larger late; [FlashdLLM] 5.1: a full refresh every few steps,
    incremental updates between): radius_at gives R at block-local step s
    rising in equal stages from R_min to R; full_refresh_at marks the steps
    s % every == 0 whose refresh set is every row.
"""
import numpy as np


class SWDState:
    """Per-sequence history of (top-1 token, top-1 prob) for active positions."""

    def __init__(self, batch, block_len):
        self.batch = batch
        self.block_len = block_len
        self.reset()

    def reset(self):
        self.tok = [[[] for _ in range(self.block_len)] for _ in range(self.batch)]
        self.p = [[[] for _ in range(self.block_len)] for _ in range(self.batch)]
        self.n = np.zeros((self.batch, self.block_len), dtype=np.int64)

    def copy(self):
        c = SWDState.__new__(SWDState)
        c.batch, c.block_len = self.batch, self.block_len
        c.tok = [[list(x) for x in row] for row in self.tok]
        c.p = [[list(x) for x in row] for row in self.p]
        c.n = self.n.copy()
        return c


def _mean_f32(ps, K):
    s = np.float32(0.0)
    for p in ps:                      # oldest -> newest
        s = np.float32(s + np.float32(p))
    return np.float32(s / np.float32(K))


def swd_update(state, q0, argmax, p1, tok, stable, K, tau, last_step):
    """One SWD update for the active block [q0, q0 + blk) of every sequence.

    argmax, p1: [B, blk] (p1 is kept in fp32, as the GPU keeps it).
    tok, stable: [B, L], updated in place.  Returns the [B, blk] bool array of
    positions that became stable at this step.
    """
    B, blk = argmax.shape
    newly = np.zeros((B, blk), dtype=bool)
    tau32 = np.float32(tau)
    for b in range(B):
        for j in range(blk):
            r = q0 + j
            if stable[b, r]:
                continue                         # [SWD] 3.3 d: stable is absorbing
            hist_t, hist_p = state.tok[b][j], state.p[b][j]
            hist_t.append(int(argmax[b, j]))
            hist_p.append(np.float32(p1[b, j]))
            state.n[b, j] += 1
            if len(hist_t) > K:                  # [SWD] 4.2: keep the last K
                del hist_t[0]
                del hist_p[0]
            if len(hist_t) == K and len(set(hist_t)) == 1 and _mean_f32(hist_p, K) > tau32:
                stable[b, r] = True
                tok[b, r] = hist_t[-1]
                newly[b, j] = True
        if last_step:
            for j in range(blk):
                r = q0 + j
                if not stable[b, r]:
                    tok[b, r] = int(argmax[b, j])
    return newly


def dilate(unstable, R, L):
    """[SWD] 3.2: union of [u-R, u+R] over unstable positions u, clipped to
    [0, L-1].  Returns a bool mask of length L."""
    m = np.zeros(L, dtype=bool)
    for u in unstable:
        m[max(0, u - R):min(L - 1, u + R) + 1] = True
    return m


def expired_rows(version, t, expiry):
    """[TA] 2.3 / 3.1: entries whose version is more than ``expiry`` steps old.

    version: [n_layers, B, L]; returns a [B, L] bool mask (a row is stale when
    any layer's entry is stale)."""
    if expiry < 0:
        return np.zeros(version.shape[1:], dtype=bool)
    return np.any(t - version > expiry, axis=0)


def radius_at(s, steps, R, R_min):
    """Dilation radius at block-local step s of a block of `steps` steps:
    R when R_min < 0, else R_min + floor((R - R_min + 1) * s / steps)
    (R_min at s = 0, R over the last stage)."""
    if R_min < 0:
        return R
    return R_min + ((R - R_min + 1) * s) // steps


def full_refresh_at(s, every):
    """Is block-local step s a scheduled refresh of every row?"""
    return every > 0 and s % every == 0


def confidence(ent, H_max, age, alpha, beta, lam):
    """[FlashdLLM] 3.1 cache confidence, in fp32 in this order:
    alpha * (1 - ent / H_max) + beta * exp(-lam * age)."""
    f = np.float32
    a = f(alpha) * (f(1.0) - f(ent) / f(H_max))
    b = f(beta) * np.exp(-(f(lam) * f(age)), dtype=np.float32)
    return f(a + b)


def confidence_rows(stable, tok, tok_w, version, q0, blk, ent, H_max, t_next, expiry, alpha, beta, lam, theta):
    """Refresh set for step t_next with the confidence criterion in place of
    the window: an active position still unstable is refreshed when its cache
    confidence (its entropy at this step, the age t_next - version of its
    layer-0 entry) is below theta; plus changed and expired rows as always.
    ent: [B, blk] entropies of the active block."""
    B, L = tok.shape
    rf = np.zeros((B, L), dtype=bool)
    for b in range(B):
        for j in range(blk):
            p = q0 + j
            if stable[b, p]:
                continue
            age = t_next - int(version[0, b, p])
            if confidence(ent[b, j], H_max, age, alpha, beta, lam) < np.float32(theta):
                rf[b, p] = True
    rf |= tok != tok_w
    rf |= expired_rows(version, t_next, expiry)
    return np.flatnonzero(rf.reshape(-1)).astype(np.int32)


def step_stats(rf_next, stable, newly, version, q0, blk, L, t_next, expiry, last, partial_next, done):
    """Per-sequence counters of one SWD update ([SWD] 4.4 plots the stability
    curve: how many positions are stable, and how much is recomputed, as the
    steps go on).  Returns int [B, 4]:
      rows of the next step's refresh set (rf_next, flat ids);
      stable rows of the active block after the update;
      rows in that refresh set because their version expired ([TA] 2.3),
        counted when the next step builds the set by the rules
        (partial_next) and the sequence is still running;
      rows committed by this update: newly stable ones, plus at the block's
        last step every row still unstable (its argmax is committed)."""
    B = stable.shape[0]
    out = np.zeros((B, 4), dtype=np.int64)
    exp = expired_rows(version, t_next, expiry)
    for b in range(B):
        out[b, 0] = int(np.sum(rf_next // L == b))
        act = stable[b, q0:q0 + blk]
        out[b, 1] = int(act.sum())
        out[b, 2] = int(exp[b].sum()) if partial_next and not done[b] else 0
        out[b, 3] = int(newly[b].sum()) + (int((~act).sum()) if last else 0)
    return out


def refresh_rows(stable, tok, tok_w, version, q0, blk, R, t_next, expiry):
    """Refresh set for step t_next as sorted flat row indices b*L + pos."""
    B, L = tok.shape
    rf = np.zeros((B, L), dtype=bool)
    for b in range(B):
        unstable = [q0 + j for j in range(blk) if not stable[b, q0 + j]]
        rf[b] |= dilate(unstable, R, L)
    rf |= tok != tok_w
    rf |= expired_rows(version, t_next, expiry)
    return np.flatnonzero(rf.reshape(-1)).astype(np.int32)
