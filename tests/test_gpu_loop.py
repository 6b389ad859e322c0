"""Step-by-step parity of whole generations (GPU): free-running until an
ambiguous position (top-2 logit margin <= 1e-2, or mean top-1 probability
within 1e-3 of tau) could send the two trajectories apart."""
import numpy as np
import pytest
import torch

import oracle as O
from denoising_step_kv_gb300 import _lib as K
from denoising_step_kv_gb300 import loop
from gpu_util import cache_fields, close, i32, max_err, read_field, tol, write_field, write_kv
from workloads import configs as C
from workloads import generate as G

pytestmark = pytest.mark.gpu


def _ambiguous(rec, w):
    amb = rec["margin"] <= 1e-2
    # a position whose SWD mean lands within 1e-3 of tau
    for b in range(w.batch):
        for j in range(w.block_len):
            ps = rec["swd"].p[b][j]
            if len(ps) == w.swd_K and abs(float(np.mean(ps)) - w.swd_tau) < 1e-3:
                amb[b, j] = True
    return amb


CONF_BAND = 1e-2     # confidences this close to theta may fall either way (entropy within its tolerance)


def _conf_ambiguous(rec, w):
    """Flat rows b * L + q0 + j whose cache confidence for the next step (the
    oracle's entropy and versions) lies within CONF_BAND of theta."""
    if w.gate != "confidence" or rec["s"] == w.steps_per_block - 1:
        return np.zeros(0, dtype=np.int64)
    out = []
    for b in range(w.batch):
        for j in range(w.block_len):
            p = rec["q0"] + j
            if rec["stable"][b, p]:
                continue
            c = O.confidence(rec["ent"][b, j], np.log(w.vocab - 1), rec["t"] + 1 - int(rec["version"][0, b, p]),
                             w.conf_alpha, w.conf_beta, 3.0 / w.steps_per_block)
            if abs(float(c) - w.conf_theta) < CONF_BAND:
                out.append(b * w.seq_len + p)
    return np.array(out, dtype=np.int64)


@pytest.mark.parametrize("name", ["tiny_fp32", "tiny_fp32_sharp", "mid_bf16", "mid_bf16_dh64", "mid_bf16_sharp",
                                  "big_rows", "mid_bf16_sched", "mid_bf16_conf"])
def test_free_running_generation(name):
    w = C.get(name)
    m = G.model(w)
    tok0 = G.prompt_tokens(w)
    trace = O.run_dense(w, O.weights_f64(w, m), tok0)
    gen = loop.DenseGenerator(w, {k: loop.to_device(v) for k, v in m.items()})
    B, L, blk, d = w.batch, w.seq_len, w.block_len, w.d_model
    got = []

    def grab(t, q0, s):
        got.append(dict(argmax=gen.argmax.cpu().numpy().reshape(B, blk), p1=gen.p1.cpu().numpy().reshape(B, blk),
                        ent=gen.ent.cpu().numpy().reshape(B, blk), tok=gen.tok.cpu().numpy().copy(),
                        o=gen.o.float().cpu().numpy().reshape(B, blk, d), h=gen.h.float().cpu().numpy().reshape(B, blk, d),
                        rows=gen.rows.cpu().numpy()[:int(gen.n_rows.item())].copy(),
                        version=read_field(gen.cache, K.FIELD_VERSION, 0, (1, B, L), "i32"),
                        stable=read_field(gen.cache, K.FIELD_STABLE, 0, (B, L), "u8").astype(bool)))

    gen.tok_in.copy_(torch.from_numpy(tok0))
    try:
        gen.run(on_step=grab)
        assert K.dllm_cache_check(gen.cache) == 0
        stats = read_field(gen.cache, K.FIELD_STEP_STATS, 0, (K.STATS_STEPS, B, 4), "i32")
    finally:
        gen.close()
    assert not np.any(stats[len(trace):])          # steps not run record nothing
    rtol, atol = tol(w)
    compared = 0
    for rec, g in zip(trace, got):
        t = rec["t"]
        assert close(g["o"], rec["o"], w), (name, t, "o", max_err(g["o"], rec["o"]))
        assert close(g["h"], rec["h"], w), (name, t, "h", max_err(g["h"], rec["h"]))
        assert np.allclose(g["p1"], rec["p1"], rtol=rtol, atol=atol), (name, t, "p1")
        assert np.allclose(g["ent"], rec["ent"], rtol=rtol, atol=atol), (name, t, "ent")
        amb = _ambiguous(rec, w)
        ok = ~amb
        assert np.array_equal(g["argmax"][ok], rec["argmax"][ok]), (name, t, "argmax")
        if np.any(g["argmax"][amb] != rec["argmax"][amb]):
            break        # trajectories may part here: stop free-running comparison
        assert np.array_equal(g["tok"], rec["tok"]), (name, t, "tok")
        assert np.array_equal(g["stable"], rec["stable"]), (name, t, "stable")
        assert np.array_equal(g["version"], rec["version"]), (name, t, "version")
        camb = _conf_ambiguous(rec, w)
        if len(camb):       # a confidence decision within the band: rows may part from here on
            assert np.array_equal(np.setdiff1d(g["rows"], camb), np.setdiff1d(rec["rows_next"], camb)), (name, t)
            compared += 1
            break
        assert np.array_equal(g["rows"], rec["rows_next"]), (name, t, "rows")
        # the stability curve: refresh, stable, expired and committed rows per sequence
        assert np.array_equal(stats[t], rec["stats"]), (name, t, "stats", stats[t], rec["stats"])
        compared += 1
    assert compared >= 1 or np.any(trace[0]["margin"] <= 1e-2), (name, compared)


def _load_pre(gen, w, rec):
    """Put the oracle's pre-step state into the GPU handle and buffers."""
    pre = rec["pre"]
    B, L, blk, Kk = w.batch, w.seq_len, w.block_len, w.swd_K
    c = gen.cache
    gen.tok.copy_(torch.from_numpy(pre["tok"].astype(np.int32)))
    write_field(c, K.FIELD_VERSION, 0, pre["version"], "i32")
    write_field(c, K.FIELD_TOK_W, 0, pre["tok_w"], "i32")
    write_field(c, K.FIELD_STABLE, 0, pre["stable"].reshape(-1), "u8")
    ht = np.zeros((B, blk, Kk), np.int32)
    hp = np.zeros((B, blk, Kk), np.float32)
    hn = pre["swd"].n.astype(np.int32)
    for b in range(B):
        for j in range(blk):
            toks, ps = pre["swd"].tok[b][j], pre["swd"].p[b][j]
            n = int(hn[b, j])
            for k, (a, p) in enumerate(zip(toks, ps)):
                slot = (n - len(toks) + k) % Kk
                ht[b, j, slot], hp[b, j, slot] = a, p
    write_field(c, K.FIELD_HIST_TOK, 0, ht, "i32")
    write_field(c, K.FIELD_HIST_P, 0, hp, "f32")
    write_field(c, K.FIELD_HIST_N, 0, hn, "i32")
    for f, arr in zip((K.FIELD_Q, K.FIELD_K, K.FIELD_V), pre["caches"]):
        write_kv(c, f, 0, w, arr[0])
    rows = rec["rows"]
    gen.rows.zero_()
    gen.rows[:len(rows)] = i32(rows)
    gen.n_rows.fill_(len(rows))


@pytest.mark.parametrize("name", ["tiny_fp32_sharp", "mid_bf16", "mid_bf16_dh64", "mid_bf16_sharp", "mid_bf16_sched",
                                  "mid_bf16_conf"])
def test_teacher_forced_steps(name):
    """Every step starts from the oracle's pre-step state (caches included);
    exactness is required away from ambiguous positions."""
    w = C.get(name)
    m = G.model(w)
    tok0 = G.prompt_tokens(w)
    trace = O.run_dense(w, O.weights_f64(w, m), tok0, keep_pre=True)
    gen = loop.DenseGenerator(w, {k: loop.to_device(v) for k, v in m.items()})
    B, L, blk, d, R = w.batch, w.seq_len, w.block_len, w.d_model, w.swd_R
    rtol, atol = tol(w)
    try:
        K.dllm_cache_reset(gen.cache)
        for rec in trace:
            t, q0, s = rec["t"], rec["q0"], rec["s"]
            _load_pre(gen, w, rec)
            gen.step(t, q0, s)
            assert K.dllm_cache_check(gen.cache) == 0
            o = gen.o.float().cpu().numpy().reshape(B, blk, d)
            h = gen.h.float().cpu().numpy().reshape(B, blk, d)
            assert close(o, rec["o"], w), (name, t, "o", max_err(o, rec["o"]))
            assert close(h, rec["h"], w), (name, t, "h", max_err(h, rec["h"]))
            assert np.allclose(gen.p1.cpu().numpy().reshape(B, blk), rec["p1"], rtol=rtol, atol=atol), (name, t)
            assert np.allclose(gen.ent.cpu().numpy().reshape(B, blk), rec["ent"], rtol=rtol, atol=atol), (name, t)
            amb = _ambiguous(rec, w)
            am = gen.argmax.cpu().numpy().reshape(B, blk)
            assert np.array_equal(am[~amb], rec["argmax"][~amb]), (name, t, "argmax")
            # positions whose fate hangs on an ambiguous decision
            skip = np.zeros((B, L), dtype=bool)
            for b, j in zip(*np.nonzero(amb)):
                skip[b, max(0, q0 + j - R):q0 + j + R + 1] = True
            tok = gen.tok.cpu().numpy()
            stable = read_field(gen.cache, K.FIELD_STABLE, 0, (B, L), "u8").astype(bool)
            assert np.array_equal(tok[~skip], rec["tok"][~skip]), (name, t, "tok")
            assert np.array_equal(stable[~skip], rec["stable"][~skip]), (name, t, "stable")
            rows = gen.rows.cpu().numpy()[:int(gen.n_rows.item())]
            skip.reshape(-1)[_conf_ambiguous(rec, w)] = True
            keep = lambda r: r[~skip.reshape(-1)[r]]
            assert np.array_equal(keep(rows), keep(rec["rows_next"])), (name, t, "rows")
            ver = read_field(gen.cache, K.FIELD_VERSION, 0, (1, B, L), "i32")
            assert np.array_equal(ver, rec["version"]), (name, t, "version")
    finally:
        gen.close()
