"""Step-by-step parity of whole generations (GPU): free-running until an
ambiguous position (top-2 logit margin <= 1e-2, or mean top-1 probability
within 1e-3 of tau) could send the two trajectories apart."""
import numpy as np
import pytest
import torch

import oracle as O
from denoising_step_kv_gb300 import _lib as K
from denoising_step_kv_gb300 import loop
from gpu_util import close, max_err, read_field, tol
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


@pytest.mark.parametrize("name", ["tiny_fp32", "tiny_fp32_sharp", "mid_bf16", "mid_bf16_dh64", "mid_bf16_sharp"])
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
    finally:
        gen.close()
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
        assert np.array_equal(g["rows"], rec["rows_next"]), (name, t, "rows")
        assert np.array_equal(g["version"], rec["version"]), (name, t, "version")
        compared += 1
    assert compared >= min(len(trace), 6), (name, compared)
