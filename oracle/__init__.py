"""CPU oracle for one cached denoising step of a masked diffusion LM.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the package's
``__graft_entry__.smoke()`` check and ``bench.py``'s CPU-baseline / reference
arm may import anything from here.  The GPU path never calls it, and shares no
code with it: the only common module is ``workloads`` (seeded inputs, no
arithmetic of the method).

Plain NumPy, fp64 arithmetic; values are rounded to the storage type (bf16 or
fp32) exactly where the GPU path stores them (Q/K/V cache rows, attention
output O, residual stream h, FFN intermediate).
"""
from .model import (bf16_bits_to_f64, round_store, rms_scale, rope, project_qkv,
                    attention, attention_partial, merge_partials, out_proj, ffn, lm_head_conf, gelu)
from .swd import (SWDState, swd_update, dilate, refresh_rows, expired_rows, radius_at, full_refresh_at,
                  confidence, confidence_rows, step_stats)
from .run import run_dense, run_stream, weights_f64, ring_positions, RingSim, NEVER

__all__ = [
    "bf16_bits_to_f64", "round_store", "rms_scale", "rope", "project_qkv",
    "attention", "attention_partial", "merge_partials", "out_proj", "ffn", "lm_head_conf", "gelu", "SWDState",
    "swd_update", "dilate", "refresh_rows", "expired_rows", "radius_at", "full_refresh_at", "confidence",
    "confidence_rows", "step_stats", "run_dense",
    "run_stream", "weights_f64", "ring_positions", "RingSim", "NEVER",
]
