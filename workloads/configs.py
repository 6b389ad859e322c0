"""Workload shapes for one cached denoising step of a masked diffusion LM.

Five named workloads restate the shapes the pages run their methods on (a tiny
fp32 layer, a 2048-wide bf16 layer, an 8B-shaped layer, an attention-sink
stream and a 12-layer denoiser), plus small shapes that the CPU oracle finishes
in seconds and that still span several GPU tiles with ragged tails.

This module holds shapes and hyper-parameters only: no arithmetic of the method.
"""
from dataclasses import dataclass, field, replace


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: str            # "f32" or "bf16": storage/compute type of the path
    n_layers: int
    batch: int
    seq_len: int          # L (dense cache); unused by the sink stream
    n_prompt: int
    block_len: int        # SAR block length (active block Ac)
    steps_per_block: int  # Tb
    d_model: int
    n_heads: int
    head_dim: int
    vocab: int
    ffn: int = 0          # FFN hidden width (0 = single attention layer, no FFN)
    swd_K: int = 3
    swd_tau: float = 0.9
    swd_R: int = 2
    swd_R_min: int = -1   # dilation radius at a block's first step (growing to swd_R); -1 = fixed swd_R
    full_every: int = 0   # refresh every row at block-local steps s with s % full_every == 0 (0 = never)
    # refresh criterion of the active block: "window" (unstable rows dilated by
    # R) or "confidence" (unstable rows whose cache confidence is below theta)
    gate: str = "window"
    conf_alpha: float = 0.7
    conf_beta: float = 0.3
    conf_theta: float = 0.5
    early_exit: int = 0   # 1: a sequence whose active rows are all stable ends its block
    expiry: int = -1      # reject t - version > expiry; -1 = no expiry
    mask_id: int = 0
    rope_theta: float = 10000.0
    rms_eps: float = 1e-6
    seed: int = 0
    tokens: str = "zipf"  # "uniform255" or "zipf" (Zipf(1.1) over ids 1..V-1)
    zipf_a: float = 1.1
    lm_scale: float = 1.0  # multiplies W_lm ("sharp" variants make SWD fire)
    active_queries: int = 0  # 1: every active-block row passes through the layers as a query
    #                          (only the refresh set rewrites K/V; multi-layer denoiser)
    # attention-sink stream (sink > 0 selects streaming mode)
    sink: int = 0
    window: int = 0
    stream_len: int = 0

    @property
    def n_gen(self):
        return self.seq_len - self.n_prompt

    @property
    def n_blocks(self):
        return self.n_gen // self.block_len

    @property
    def n_steps(self):
        return self.n_blocks * self.steps_per_block

    @property
    def streaming(self):
        return self.sink > 0

    @property
    def cache_len(self):
        return self.sink + self.window if self.streaming else self.seq_len


# --- the five workloads (shapes as the pages' settings give them) -----------
TINY_FP32 = Workload(
    name="tiny_fp32", dtype="f32", n_layers=1, batch=1, seq_len=64, n_prompt=32,
    block_len=8, steps_per_block=16, d_model=64, n_heads=2, head_dim=32, vocab=256,
    swd_K=3, swd_tau=0.95, swd_R=2, expiry=-1, seed=0, tokens="uniform255")

BF16_D2048 = Workload(
    name="bf16_d2048", dtype="bf16", n_layers=1, batch=4, seq_len=1024, n_prompt=896,
    block_len=32, steps_per_block=32, d_model=2048, n_heads=16, head_dim=128,
    vocab=32000, swd_K=3, swd_tau=0.9, swd_R=2, expiry=2, seed=1)

LAYER_8B = Workload(
    name="8b_shaped", dtype="bf16", n_layers=1, batch=8, seq_len=4096, n_prompt=3584,
    block_len=32, steps_per_block=32, d_model=4096, n_heads=32, head_dim=128,
    vocab=126464, swd_K=3, swd_tau=0.95, swd_R=1, expiry=-1, seed=2)

SINK_RING = Workload(
    name="sink_ring", dtype="bf16", n_layers=1, batch=1, seq_len=0, n_prompt=0,
    block_len=1, steps_per_block=1, d_model=4096, n_heads=32, head_dim=128,
    vocab=32000, seed=3, sink=4, window=4092, stream_len=32768)

TWELVE_LAYER = Workload(
    name="twelve_layer", dtype="bf16", n_layers=12, batch=16, seq_len=2048,
    n_prompt=1536, block_len=64, steps_per_block=64, d_model=1024, n_heads=16,
    head_dim=64, vocab=32000, ffn=4096, swd_K=3, swd_tau=0.9, swd_R=2, expiry=2,
    seed=4, active_queries=1)

NAMED = {w.name: w for w in (TINY_FP32, BF16_D2048, LAYER_8B, SINK_RING, TWELVE_LAYER)}

# The 12-layer shape with W_lm scaled so that positions stabilise and commit
# inside a block (the stability mask then gates the per-layer refresh).
TWELVE_LAYER_SHARP = replace(TWELVE_LAYER, name="twelve_layer_sharp", lm_scale=40.0)

# --- small shapes for element-by-element parity ------------------------------
# Ragged on purpose: 320 rows (2.5 row tiles of 128), vocab 1000 (7 column
# tiles of 128 and a 104-wide tail), L = 160 keys (2.5 key tiles of 64).
MID_BF16 = Workload(
    name="mid_bf16", dtype="bf16", n_layers=1, batch=2, seq_len=160, n_prompt=128,
    block_len=16, steps_per_block=6, d_model=256, n_heads=2, head_dim=128,
    vocab=1000, swd_K=3, swd_tau=0.9, swd_R=2, expiry=2, seed=11)

MID_BF16_DH64 = replace(MID_BF16, name="mid_bf16_dh64", n_heads=4, head_dim=64,
                        seed=12, swd_R=1, expiry=-1)

# "Sharp" variants: W_lm scaled so that top-1 probabilities clear tau and the
# stable / commit / dilation paths run (with N(0, 0.02) weights p1 ~ 1/V).
TINY_FP32_SHARP = replace(TINY_FP32, name="tiny_fp32_sharp", lm_scale=60.0)
MID_BF16_SHARP = replace(MID_BF16, name="mid_bf16_sharp", lm_scale=40.0,
                         steps_per_block=10)

# The schedules of the refresh set: a dilation radius that grows from 0 at a
# block's first step to R = 3 at its last, and a full refresh every 4th step
# of a block (no version expiry, so only the schedule refreshes the prompt).
MID_BF16_SCHED = replace(MID_BF16_SHARP, name="mid_bf16_sched", swd_R=3, swd_R_min=0, full_every=4, expiry=-1,
                         seed=19)

MID_SINK = Workload(
    name="mid_sink", dtype="bf16", n_layers=1, batch=1, seq_len=0, n_prompt=0,
    block_len=1, steps_per_block=1, d_model=256, n_heads=2, head_dim=128,
    vocab=1000, seed=13, sink=4, window=92, stream_len=300)

# fp32 stream through a ring of 2 sinks + 13 rolling slots (wraps 3 times)
TINY_SINK_F32 = Workload(
    name="tiny_sink_f32", dtype="f32", n_layers=1, batch=1, seq_len=0, n_prompt=0,
    block_len=1, steps_per_block=1, d_model=64, n_heads=2, head_dim=32,
    vocab=256, seed=15, sink=2, window=13, stream_len=50)

MID_MULTI = Workload(
    name="mid_multi", dtype="bf16", n_layers=3, batch=2, seq_len=160, n_prompt=128,
    block_len=16, steps_per_block=6, d_model=256, n_heads=4, head_dim=64,
    vocab=1000, ffn=512, swd_K=3, swd_tau=0.9, swd_R=2, expiry=2, seed=14,
    active_queries=1)

MID_MULTI_SHARP = replace(MID_MULTI, name="mid_multi_sharp", lm_scale=40.0, steps_per_block=10, seed=18)

# The confidence criterion in place of the window, without version expiry:
# with W_lm x 12 the entropies sit around the threshold's reach, so a
# position is refreshed once its entry has aged enough for its entropy, and
# tau = 0.4 lets some positions commit.
MID_MULTI_CONF = replace(MID_MULTI, name="mid_multi_conf", lm_scale=12.0, steps_per_block=10, seed=21,
                         gate="confidence", expiry=-1, swd_tau=0.4)
MID_BF16_CONF = replace(MID_BF16, name="mid_bf16_conf", lm_scale=12.0, steps_per_block=10, seed=22,
                        gate="confidence", expiry=-1, swd_tau=0.4)

# Early block exit on sharp heads: sequences end their blocks at different
# steps (batch 3, 12 steps per block).
MID_BF16_EXIT = replace(MID_BF16_SHARP, name="mid_bf16_exit", batch=3, steps_per_block=12, early_exit=1, seed=23)
MID_MULTI_EXIT = replace(MID_MULTI_SHARP, name="mid_multi_exit", batch=3, steps_per_block=12, early_exit=1, seed=24)

# More rows than the weight-streaming path takes (256): the projection runs
# on the large-M kernels.  600 rows = 5 row tiles (an odd count: the last
# cluster pair has a half past the end), 900 rows = 7 tiles + 4 rows.
BIG_ROWS = replace(MID_BF16, name="big_rows", batch=2, seq_len=300, n_prompt=268, seed=16)
BIG_ROWS_DH64 = replace(MID_BF16_DH64, name="big_rows_dh64", batch=3, seq_len=300, n_prompt=268, seed=17)

ALL = dict(NAMED)
for _w in (MID_BF16, MID_BF16_DH64, TINY_FP32_SHARP, MID_BF16_SHARP, MID_SINK, TINY_SINK_F32, MID_MULTI,
           MID_MULTI_SHARP, BIG_ROWS, BIG_ROWS_DH64, TWELVE_LAYER_SHARP, MID_BF16_SCHED, MID_MULTI_CONF,
           MID_BF16_CONF, MID_BF16_EXIT, MID_MULTI_EXIT):
    ALL[_w.name] = _w


def get(name):
    return ALL[name]
