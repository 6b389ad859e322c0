"""lmhead_conf_noalloc (GPU): the LM-head confidence entry point for callers
that cannot allocate device memory (a host whose memory planner owns every
device byte, code that must avoid cudaMalloc's implicit synchronisation, a
caller without a handle).  Its scratch is a static device array, so two calls
in a row reuse the same bytes; both must agree with lmhead_conf, the entry
point that uses the handle's scratch.  This file runs last in the suite."""
import numpy as np
import pytest
import torch

from denoising_step_kv_gb300 import _lib as K
from denoising_step_kv_gb300.loop import to_device
from gpu_util import tol
from workloads import configs as C
from workloads import generate as G

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["mid_bf16", "bf16_d2048", "tiny_fp32"])
def test_noalloc_matches_handle_entry_on_two_calls(name):
    w = C.get(name)
    M, V, d = w.batch * w.block_len, w.vocab, w.d_model
    dt = K.DLLM_BF16 if w.dtype == "bf16" else K.DLLM_F32
    cache = K.dllm_cache_init(K.make_cfg(w))
    try:
        out = {}
        for call, seed in enumerate((71, 72)):          # two calls in a row, different inputs
            h = to_device(G.normal(seed, (M, d), 1.0, w.dtype))
            wl = to_device(G.normal(seed + 10, (V, d), 0.02 * (1 + 20 * call), w.dtype))
            res = []
            for fn in ("handle", "noalloc"):
                am = torch.full((M,), -1, dtype=torch.int32, device="cuda")
                p1 = torch.zeros(M, dtype=torch.float32, device="cuda")
                ent = torch.zeros(M, dtype=torch.float32, device="cuda")
                if fn == "handle":
                    K.lmhead_conf(cache, h, wl, M, V, d, w.mask_id, am, p1, ent)
                else:
                    K.lmhead_conf_noalloc(h, wl, M, V, d, dt, w.mask_id, w.rms_eps, am, p1, ent)
                torch.cuda.synchronize()
                res.append((am.cpu().numpy(), p1.cpu().numpy(), ent.cpu().numpy()))
            (a0, p0, e0), (a1, p1_, e1) = res
            rtol, atol = tol(w)
            assert np.array_equal(a0, a1), (name, call)
            assert np.allclose(p0, p1_, rtol=rtol, atol=atol), (name, call)
            assert np.allclose(e0, e1, rtol=rtol, atol=atol), (name, call)
            assert np.all(a1 >= 0) and np.all(a1 != w.mask_id)
            out[call] = a1
        assert not np.array_equal(out[0], out[1])        # the second call did not reuse stale results
        assert K.dllm_cache_check(cache) == 0
    finally:
        K.dllm_cache_free(cache)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_noalloc_at_the_scratch_capacity_against_the_oracle(dtype):
    """M in (128, 256] (bf16: the pair-tile path) and V = 131072, the
    largest the static scratch takes, against the oracle; the device's free
    memory is the same before and after two calls."""
    import oracle as O
    M, V, d = 200, 131072, 128 if dtype == "bf16" else 64
    h_np = G.normal(81, (M, d), 1.0, dtype)
    w_np = G.normal(82, (V, d), 0.5, dtype)
    h, wl = to_device(h_np), to_device(w_np)
    dt = K.DLLM_BF16 if dtype == "bf16" else K.DLLM_F32
    outs = [(torch.zeros(M, dtype=torch.int32, device="cuda"), torch.zeros(M, device="cuda"),
             torch.zeros(M, device="cuda")) for _ in range(2)]
    K.lmhead_conf_noalloc(h, wl, M, V, d, dt, 0, 1e-6, *outs[0])      # first call on the device: set-up
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for o in outs:
        K.lmhead_conf_noalloc(h, wl, M, V, d, dt, 0, 1e-6, *o)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    to64 = O.bf16_bits_to_f64 if dtype == "bf16" else (lambda a: a.astype(np.float64))
    am, p1, ent, margin = O.lm_head_conf(to64(h_np), to64(w_np), 0, 1e-6)
    rtol, atol = (2e-2, 1e-3) if dtype == "bf16" else (1e-5, 1e-5)
    for a, p, e in outs:
        a, p, e = a.cpu().numpy(), p.cpu().numpy(), e.cpu().numpy()
        sure = margin > 1e-2
        assert np.array_equal(a[sure], am[sure])
        assert np.allclose(p, p1, rtol=rtol, atol=atol)
        assert np.allclose(e, ent, rtol=rtol, atol=atol)


def test_noalloc_rejects_sizes_beyond_the_static_scratch():
    h = torch.zeros(300, 64, dtype=torch.bfloat16, device="cuda")
    wl = torch.zeros(1000, 64, dtype=torch.bfloat16, device="cuda")
    out_i = torch.zeros(300, dtype=torch.int32, device="cuda")
    out_f = torch.zeros(300, dtype=torch.float32, device="cuda")
    with pytest.raises(K.DllmError):
        K.lmhead_conf_noalloc(h, wl, 300, 1000, 64, K.DLLM_BF16, 0, 1e-6, out_i, out_f, out_f)
    big_v = torch.zeros(1, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(K.DllmError):
        K.lmhead_conf_noalloc(big_v, big_v, 1, 200000, 64, K.DLLM_BF16, 0, 1e-6, out_i, out_f, out_f)
    with pytest.raises(K.DllmError):                  # d must be a multiple of 64
        K.lmhead_conf_noalloc(big_v, big_v, 1, 1000, 40, K.DLLM_BF16, 0, 1e-6, out_i, out_f, out_f)
