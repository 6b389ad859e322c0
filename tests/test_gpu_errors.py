"""Failure paths on the GPU that fault nothing: a bounded barrier wait that
runs out (a barrier that nothing arrives on) sets the timeout bit and returns,
leaving the context usable; device-side range checks set their bits and skip
the item."""
import time

import numpy as np
import pytest
import torch

from denoising_step_kv_gb300 import _lib as K
from gpu_util import i32
from workloads import configs as C
from workloads import generate as G
from denoising_step_kv_gb300.loop import to_device

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_the_context_stays_usable():
    w = C.get("mid_bf16")
    c = K.dllm_cache_init(K.make_cfg(w))
    try:
        assert K.dllm_cache_error_word(c) == 0
        t0 = time.perf_counter()
        K.dllm_wait_selftest(c, 50_000_000)            # 50 ms
        err = K.dllm_cache_error_word(c)              # synchronises
        dt = time.perf_counter() - t0
        assert err & K.ERR_TIMEOUT
        assert 0.05 <= dt < 5.0
        with pytest.raises(K.DllmError):
            K.dllm_wait_selftest(c, 10)               # below the accepted range: nothing launched
        # the same handle and context still run the step's kernels
        m = G.model(w)
        tok = i32(G.integers(3, 1, w.vocab, (w.batch, w.seq_len)))
        K.kv_refresh(c, 0, None, tok, to_device(m["embed"]), to_device(m["w_qkv"][0]), None, None, 1)
        out = torch.zeros(w.batch * w.block_len, w.d_model, dtype=torch.bfloat16, device="cuda")
        K.block_attn(c, 0, w.n_prompt, w.block_len, out)
        assert K.dllm_cache_check(c) == 0
        assert torch.isfinite(out.float()).all() and out.float().abs().sum() > 0
    finally:
        K.dllm_cache_free(c)


def test_state_copy_refuses_unknown_fields_and_wrong_sizes():
    """A field outside the enumeration (negative or past the last) and a byte
    count other than the field's size are refused before anything is copied;
    the handle keeps working."""
    w = C.get("mid_bf16")
    c = K.dllm_cache_init(K.make_cfg(w))
    try:
        for f in (-1, -7, K.FIELD_STEP_STATS + 1):
            with pytest.raises(K.DllmError) as e:
                K.state_size(c, f)
            assert e.value.status == 1 and "unknown field" in K.last_error()
        n = K.state_size(c, K.FIELD_TOK_W)
        assert n == w.batch * w.seq_len * 4
        with pytest.raises(K.DllmError) as e:
            K.dllm_state_copy(c, K.FIELD_TOK_W, 0, torch.zeros(n // 4 - 1, dtype=torch.int32), False)
        assert e.value.status == 1
        host = torch.full((n // 4,), -5, dtype=torch.int32)
        K.dllm_state_copy(c, K.FIELD_TOK_W, 0, host, False)
        assert K.dllm_cache_check(c) == 0
    finally:
        K.dllm_cache_free(c)


def test_out_of_range_rows_and_tokens_set_bits_and_are_skipped():
    w = C.get("mid_bf16")
    m = G.model(w)
    c = K.dllm_cache_init(K.make_cfg(w))
    try:
        tok = G.integers(4, 1, w.vocab, (w.batch, w.seq_len))
        tok[0, 5] = w.vocab + 3                        # a token past the vocabulary
        rows = i32([5, 7, w.batch * w.seq_len + 11])    # the last row is past the cache
        K.kv_refresh(c, 0, None, i32(tok), to_device(m["embed"]), to_device(m["w_qkv"][0]), rows, i32([3]), 2)
        err = K.dllm_cache_error_word(c)
        assert err & K.ERR_TOKEN and err & K.ERR_ROW
        from gpu_util import read_field
        ver = read_field(c, K.FIELD_VERSION, 0, (w.batch * w.seq_len,), "i32")
        assert ver[7] == 2 and ver[5] != 2             # the valid row was written, the bad one skipped
    finally:
        K.dllm_cache_free(c)
