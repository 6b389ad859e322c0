"""Step-loop driver of the cached denoising step on one GPU.

A generation runs every SAR block for Tb denoising steps on one CUDA stream.
One step of a single-layer denoiser is:

    kv_refresh   rows of the refresh set -> versioned Q/K/V cache
    block_attn   active block's queries over the whole cached sequence
    attn_out     h = x + O W_o^T
    lmhead_conf  argmax, top-1 probability, entropy of the active rows
    stab_update  SWD update, commits, next step's refresh set

A multi-layer step runs the refresh rows through every layer (kv_refresh,
block_attn_rows, attn_out, ffn_gelu per layer) before the LM head.  An
attention-sink stream appends one token per step and attends over the sink
and rolling entries.

The refresh-set size stays on the device, so no step synchronises with the
host and a whole generation can be captured as one CUDA graph.
"""
import numpy as np
import torch

from . import _lib as K


def to_device(a, device="cuda"):
    """Generated array -> device tensor (uint16 bf16 bit patterns -> bfloat16)."""
    if isinstance(a, list):
        return [to_device(x, device) for x in a]
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)


class DenseGenerator:
    """Single-layer cached denoiser (dense positional cache).  facache: the
    attention keeps the softmax state of the key tiles outside the block's
    window (bf16 only; see block_attn)."""

    def __init__(self, w, weights, device="cuda", facache=False):
        assert not w.streaming and w.n_layers == 1 and not w.ffn
        self.w = w
        self.W = weights
        B, L, d, blk = w.batch, w.seq_len, w.d_model, w.block_len
        dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
        self.cache = K.dllm_cache_init(K.make_cfg(w, facache=facache))
        i32 = dict(dtype=torch.int32, device=device)
        self.tok = torch.zeros(B, L, **i32)
        self.rows = torch.zeros(B * L, **i32)
        self.n_rows = torch.zeros(1, **i32)
        self.o = torch.zeros(B * blk, d, dtype=dt, device=device)
        self.h = torch.zeros(B * blk, d, dtype=dt, device=device)
        self.argmax = torch.zeros(B * blk, **i32)
        self.p1 = torch.zeros(B * blk, dtype=torch.float32, device=device)
        self.ent = torch.zeros(B * blk, dtype=torch.float32, device=device)
        self.tok_in = torch.zeros(B, L, **i32)
        self.graph = None
        self.prof = {}          # kernel id -> [(begin, end) per step] of the last run

    def close(self):
        if self.cache is not None:
            K.dllm_cache_free(self.cache)
            self.cache = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- one step -------------------------------------------------------------
    def step(self, t, q0, s, stream=None):
        w, c, W = self.w, self.cache, self.W
        blk = w.block_len
        if t == 0:
            K.refresh_all(c, q0, self.rows, self.n_rows, stream)
        K.kv_refresh(c, 0, None, self.tok, W["embed"], W["w_qkv"][0], self.rows, self.n_rows, t, stream)
        K.block_attn(c, 0, q0, blk, self.o, stream)
        K.attn_out(c, self.o, W["w_o"][0], None, self.tok, W["embed"], q0, blk, None, self.h, stream)
        K.lmhead_conf(c, self.h, W["w_lm"], w.batch * blk, w.vocab, w.d_model, w.mask_id, self.argmax,
                      self.p1, self.ent, stream)
        K.stab_update(c, self.argmax, self.p1, self.ent, self.tok, q0, t, s, s == w.steps_per_block - 1, self.rows,
                      self.n_rows, stream)

    def schedule(self):
        """(t, q0, s) of every step of a generation."""
        w = self.w
        t = 0
        for bi in range(w.n_blocks):
            q0 = w.n_prompt + bi * w.block_len
            for s in range(w.steps_per_block):
                yield t, q0, s
                t += 1

    def make_prof_events(self, kernels):
        """One (begin, end) CUDA event pair per step for each kernel id
        (_lib.PROF_*), created now (a torch event exists once recorded)."""
        ev = {k: [] for k in kernels}
        for k in kernels:
            for _ in range(self.w.n_steps):
                pair = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                pair[0].record()
                pair[1].record()
                ev[k].append(pair)
        return ev

    def run(self, stream=None, on_step=None, n_steps=None, prof=None):
        """Reset the cache, copy tok_in -> tok and run the step loop.

        prof: {kernel id: [(begin, end) per step]} from make_prof_events; the
        library records the pair around that kernel's launch in every step.
        """
        K.dllm_cache_reset(self.cache, stream)
        self.tok.copy_(self.tok_in)
        prof = prof or {}
        self.prof = prof
        for t, q0, s in self.schedule():
            if n_steps is not None and t >= n_steps:
                break
            for k, pairs in prof.items():
                K.dllm_profile_events(self.cache, k, *pairs[t])
            self.step(t, q0, s, stream)
            if on_step is not None:
                on_step(t, q0, s)
        for k in prof:
            K.dllm_profile_events(self.cache, k, None, None)
        return self.tok

    def generate(self, tok0):
        self.tok_in.copy_(tok0)
        return self.run()

    # -- CUDA graph of a whole generation -------------------------------------------
    def capture(self, prof=None):
        """Capture run() as one CUDA graph (after one eager warm-up run)."""
        self.run()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.run(prof=prof)
        self.graph = g
        return g

    def replay(self):
        self.graph.replay()
        return self.tok

    def kernel_times_ms(self, kernel):
        """Per-step durations of `kernel` recorded by the last run/replay."""
        return [a.elapsed_time(b) for a, b in self.prof.get(kernel, [])]


class LayerStackGenerator:
    """Multi-layer cached denoiser (dense positional cache).

    The rows P of the refresh set (sorted flat ids; the active block is part
    of it) pass through every layer: their Q/K/V are re-projected into that
    layer's cache, their queries attend over the layer's whole cache, then
    W_o + residual and the FFN.  Every other row's deeper-layer K/V stays as
    cached.  The LM head and the SWD update then run on the active rows.
    Buffers are compact over P (row i = rows[i]); its size stays on the device.
    """

    def __init__(self, w, weights, device="cuda"):
        assert not w.streaming and w.ffn
        self.w = w
        self.W = weights
        B, L, d, blk = w.batch, w.seq_len, w.d_model, w.block_len
        dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
        self.cache = K.dllm_cache_init(K.make_cfg(w))
        i32 = dict(dtype=torch.int32, device=device)
        self.tok = torch.zeros(B, L, **i32)
        self.rows = torch.zeros(B * L, **i32)
        self.n_rows = torch.zeros(1, **i32)
        self.O = torch.zeros(B * L, d, dtype=dt, device=device)          # attention output of the rows
        self.H = [torch.zeros(B * L, d, dtype=dt, device=device) for _ in range(2)]
        self.o = torch.zeros(B * blk, d, dtype=dt, device=device)        # last layer, active rows
        self.h = torch.zeros(B * blk, d, dtype=dt, device=device)
        self.argmax = torch.zeros(B * blk, **i32)
        self.p1 = torch.zeros(B * blk, dtype=torch.float32, device=device)
        self.ent = torch.zeros(B * blk, dtype=torch.float32, device=device)
        self.tok_in = torch.zeros(B, L, **i32)
        self.graph = None

    close = DenseGenerator.close
    __del__ = DenseGenerator.__del__
    schedule = DenseGenerator.schedule

    def step(self, t, q0, s, stream=None, prof=None):
        """One denoising step.  prof: {kernel id: [(begin, end) per layer]}
        events recorded around that kernel's launch in each layer (the LM
        head's list has one pair)."""
        w, c, W = self.w, self.cache, self.W
        blk = w.block_len
        if t == 0:
            K.refresh_all(c, q0, self.rows, self.n_rows, stream)
        x = None                       # layer 0: embeddings of the rows, gathered by kv_refresh
        for l in range(w.n_layers):
            if prof:
                for k, pairs in prof.items():
                    K.dllm_profile_events(c, k, *pairs[min(l, len(pairs) - 1)])
            K.kv_refresh(c, l, x, self.tok, W["embed"], W["w_qkv"][l], self.rows, self.n_rows, t, stream)
            K.block_attn_rows(c, l, self.rows, self.n_rows, self.O, stream)
            h = self.H[l % 2]
            K.attn_out(c, self.O, W["w_o"][l], x, None, None, 0, 1, self.n_rows, h, stream)
            K.ffn_gelu(c, h, W["w1"][l], W["w2"][l], w.ffn, 0, self.n_rows, h, stream)
            x = h
        K.active_rows(c, x, self.rows, self.n_rows, q0, blk, self.h, stream)
        K.active_rows(c, self.O, self.rows, self.n_rows, q0, blk, self.o, stream)
        K.lmhead_conf(c, self.h, W["w_lm"], w.batch * blk, w.vocab, w.d_model, w.mask_id, self.argmax,
                      self.p1, self.ent, stream)
        K.stab_update(c, self.argmax, self.p1, self.ent, self.tok, q0, t, s, s == w.steps_per_block - 1, self.rows,
                      self.n_rows, stream)

    def make_prof_events(self, kernels, n_steps):
        """{kernel id: [[(begin, end) per layer] per step]} CUDA event pairs
        for the first n_steps steps (the LM head: one pair per step)."""
        ev = {}
        for k in kernels:
            per_step = []
            for _ in range(n_steps):
                layers = []
                for _ in range(1 if k == K.PROF_LM_GEMM else self.w.n_layers):
                    pair = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                    pair[0].record()
                    pair[1].record()
                    layers.append(pair)
                per_step.append(layers)
            ev[k] = per_step
        return ev

    def run(self, stream=None, on_step=None, n_steps=None, prof=None):
        K.dllm_cache_reset(self.cache, stream)
        self.tok.copy_(self.tok_in)
        for t, q0, s in self.schedule():
            if n_steps is not None and t >= n_steps:
                break
            step_prof = {k: v[t] for k, v in prof.items()} if prof and t < len(next(iter(prof.values()))) else None
            self.step(t, q0, s, stream, step_prof)
            if prof:
                for k in prof:
                    K.dllm_profile_events(self.cache, k, None, None)
            if on_step is not None:
                on_step(t, q0, s)
        return self.tok

    def capture(self, n_steps=None, prof=None):
        self.run(n_steps=n_steps)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.run(n_steps=n_steps, prof=prof)
        self.graph = g
        return g

    def replay(self):
        self.graph.replay()
        return self.tok


class StreamGenerator:
    """Attention-sink stream through one layer (batch 1).

    Token n's step: its Q/K/V row joins the sink + rolling cache at ring slot
    n (sinks keep slots 0..S-1, later tokens cycle through the W rolling
    slots, RoPE at the absolute stream index), then its query attends over
    the min(n + 1, S + W) entries the cache holds.  O_n lands in out[n].
    preproject: every token's row is projected up front in one pass
    (kv_project) and each step only copies it into its slot (ring_append);
    otherwise each step projects its own row (kv_refresh of one row, which
    streams the whole projection weight).
    """

    def __init__(self, w, weights, device="cuda", preproject=True):
        assert w.streaming and w.n_layers == 1
        self.w = w
        self.W = weights
        self.preproject = preproject
        dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
        self.cache = K.dllm_cache_init(K.make_cfg(w))
        self.staged = torch.empty(w.stream_len if preproject else 0, 3 * w.d_model, dtype=dt, device=device)
        i32 = dict(dtype=torch.int32, device=device)
        self.pos = torch.arange(w.stream_len, **i32)      # row list: token n is row n
        self.one = torch.ones(1, **i32)
        self.tok = torch.zeros(w.stream_len, **i32)
        self.out = torch.zeros(w.stream_len, w.d_model, dtype=dt, device=device)
        self.graph = None

    def close(self):
        if self.cache is not None:
            K.dllm_cache_free(self.cache)
            self.cache = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def step(self, n, stream=None):
        c, W = self.cache, self.W
        if self.preproject:
            K.ring_append(c, 0, self.staged, n, 1, stream)
        else:
            K.kv_refresh(c, 0, None, self.tok, W["embed"], W["w_qkv"][0], self.pos[n:n + 1], self.one, n, stream)
        K.block_attn(c, 0, n, 1, self.out[n:n + 1], stream)

    def make_prof_events(self, kernels, n0, n1):
        """{kernel id: [(begin, end) per token n0 .. n1-1]} CUDA event pairs."""
        ev = {}
        for k in kernels:
            ev[k] = []
            for _ in range(n0, n1):
                pair = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                pair[0].record()
                pair[1].record()
                ev[k].append(pair)
        return ev

    def run(self, n_tokens=None, stream=None, prof=None, prof_from=0):
        """Run the stream; prof (from make_prof_events(kernels, prof_from, ..))
        brackets both kernels of tokens prof_from onwards."""
        K.dllm_cache_reset(self.cache, stream)
        n_tok = self.w.stream_len if n_tokens is None else n_tokens
        if self.preproject:
            K.kv_project(self.cache, 0, self.tok, self.W["embed"], self.W["w_qkv"][0], n_tok, self.staged, stream)
        n_prof = len(next(iter(prof.values()))) if prof else 0
        for n in range(n_tok):
            on = prof_from <= n < prof_from + n_prof
            if on:
                for k, pairs in prof.items():
                    K.dllm_profile_events(self.cache, k, *pairs[n - prof_from])
            self.step(n, stream)
            if on:
                for k in prof:
                    K.dllm_profile_events(self.cache, k, None, None)
        return self.out

    def capture(self, n_tokens=None, prof=None, prof_from=0):
        self.run(n_tokens)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.run(n_tokens, prof=prof, prof_from=prof_from)
        self.graph = g
        return g

    def replay(self):
        self.graph.replay()
        return self.out
