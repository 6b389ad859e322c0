"""ctypes binding of libdllmkv.so: the C ABI's entry points under the same
names, taking torch tensors (device pointers) and a torch stream.  Argument
marshalling only: every step runs in the library's CUDA kernels.  There is no
fallback: importing a function raises if the library is missing."""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdllmkv.so")

DLLM_F32, DLLM_BF16 = 0, 1
(FIELD_Q, FIELD_K, FIELD_V, FIELD_VERSION, FIELD_TOK_W, FIELD_STABLE, FIELD_HIST_TOK, FIELD_HIST_P, FIELD_HIST_N,
 FIELD_FA_REBUILT, FIELD_SEQ_DONE, FIELD_STEP_STATS) = range(12)
STATS_STEPS = 4096   # global steps FIELD_STEP_STATS records: int32 [4096][batch][4]
ERR_ROW, ERR_TOKEN, ERR_TIMEOUT, ERR_POS, ERR_GUARD = 1, 2, 4, 8, 16
STATUS = {0: "OK", 1: "EINVAL", 2: "ENOMEM", 3: "ECUDA", 4: "EDEVICE", 5: "EUNSUPPORTED"}


class CacheCfg(ctypes.Structure):
    _fields_ = [
        ("n_layers", ctypes.c_int), ("batch", ctypes.c_int), ("seq_len", ctypes.c_int),
        ("n_heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("dtype", ctypes.c_int),
        ("sink", ctypes.c_int), ("window", ctypes.c_int), ("expiry", ctypes.c_int),
        ("rope_theta", ctypes.c_float), ("rms_eps", ctypes.c_float), ("swd_K", ctypes.c_int),
        ("swd_tau", ctypes.c_float), ("swd_R", ctypes.c_int), ("block_len", ctypes.c_int),
        ("mask_id", ctypes.c_int), ("active_queries", ctypes.c_int), ("vocab", ctypes.c_int),
        ("max_pos", ctypes.c_int), ("ffn", ctypes.c_int), ("swd_R_min", ctypes.c_int),
        ("steps_per_block", ctypes.c_int), ("full_every", ctypes.c_int), ("gate", ctypes.c_int),
        ("conf_alpha", ctypes.c_float), ("conf_beta", ctypes.c_float), ("conf_lambda", ctypes.c_float),
        ("conf_theta", ctypes.c_float), ("early_exit", ctypes.c_int), ("facache", ctypes.c_int),
    ]


class DllmError(RuntimeError):
    def __init__(self, name, status, msg):
        super().__init__(f"{name}: {STATUS.get(status, status)}: {msg}")
        self.status = status


_VP, _I, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
_SIGS = {
    "dllm_cache_init": [ctypes.POINTER(CacheCfg), _VP, ctypes.POINTER(_VP)],
    "dllm_cache_free": [_VP],
    "dllm_cache_reset": [_VP, _VP],
    "dllm_cache_check": [_VP, _VP, ctypes.POINTER(ctypes.c_uint32)],
    "dllm_state_copy": [_VP, _I, _I, _VP, _SZ, _I, ctypes.POINTER(_SZ)],
    "refresh_all": [_VP, _I, _VP, _VP, _VP],
    "kv_refresh": [_VP, _I, _VP, _VP, _VP, _VP, _VP, _VP, _I, _VP],
    "block_attn": [_VP, _I, _I, _I, _VP, _VP],
    "block_attn_rows": [_VP, _I, _VP, _VP, _VP, _VP],
    "active_rows": [_VP, _VP, _VP, _VP, _I, _I, _VP, _VP],
    "attn_out": [_VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _VP, _VP, _VP],
    "ffn_gelu": [_VP, _VP, _VP, _VP, _I, _I, _VP, _VP, _VP],
    "lmhead_conf": [_VP, _VP, _VP, _I, _I, _I, _I, _VP, _VP, _VP, _VP],
    "stab_update": [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _VP, _VP, _VP],
    "dllm_profile_events": [_VP, _I, _VP, _VP],
    "lmhead_conf_noalloc": [_VP, _VP, _I, _I, _I, _I, _I, ctypes.c_float, _VP, _VP, _VP, _VP],
    "dllm_wait_selftest": [_VP, ctypes.c_uint64, _VP],
    "kv_project": [_VP, _I, _VP, _VP, _VP, _I, _VP, _VP],
    "ring_append": [_VP, _I, _VP, _I, _I, _VP],
}
PROF_QKV_GEMM, PROF_ATTN, PROF_LM_GEMM, PROF_OUT_GEMM, PROF_FFN = 1, 2, 3, 4, 5
EXPORTS = list(_SIGS) + ["dllm_last_error"]

_lib = None


def lib():
    """Load libdllmkv.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, args in _SIGS.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        L.dllm_last_error.argtypes = []
        L.dllm_last_error.restype = ctypes.c_char_p
        _lib = L
    return _lib


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _s(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(name, status):
    if status != 0:
        raise DllmError(name, status, lib().dllm_last_error().decode())


def make_cfg(w, vocab=None, facache=False):
    """CacheCfg of a workload (see workloads.configs.Workload)."""
    c = CacheCfg()
    c.facache = 1 if facache else 0
    c.n_layers, c.batch, c.seq_len = w.n_layers, w.batch, w.seq_len
    c.n_heads, c.head_dim = w.n_heads, w.head_dim
    c.dtype = DLLM_BF16 if w.dtype == "bf16" else DLLM_F32
    c.sink, c.window, c.expiry = w.sink, w.window, w.expiry
    c.rope_theta, c.rms_eps = w.rope_theta, w.rms_eps
    c.swd_K, c.swd_tau, c.swd_R = w.swd_K, w.swd_tau, w.swd_R
    c.block_len, c.mask_id, c.active_queries = w.block_len, w.mask_id, w.active_queries
    c.vocab = w.vocab if vocab is None else vocab
    c.max_pos = w.stream_len if w.streaming else 0
    c.ffn = w.ffn
    c.swd_R_min, c.steps_per_block, c.full_every = w.swd_R_min, w.steps_per_block, w.full_every
    c.gate = 1 if w.gate == "confidence" else 0
    c.conf_alpha, c.conf_beta, c.conf_theta = w.conf_alpha, w.conf_beta, w.conf_theta
    c.conf_lambda = 3.0 / w.steps_per_block if w.steps_per_block else 0.0
    c.early_exit = w.early_exit
    return c


# --- entry points (same names as the C ABI) ---------------------------------------
def dllm_cache_init(cfg, stream=None):
    h = ctypes.c_void_p()
    _check("dllm_cache_init", lib().dllm_cache_init(ctypes.byref(cfg), _s(stream), ctypes.byref(h)))
    return h


def dllm_cache_free(c):
    _check("dllm_cache_free", lib().dllm_cache_free(c))


def dllm_cache_reset(c, stream=None):
    _check("dllm_cache_reset", lib().dllm_cache_reset(c, _s(stream)))


def dllm_cache_check(c, stream=None):
    """Synchronise and return the device error word (raises DllmError if set)."""
    w = ctypes.c_uint32(0)
    st = lib().dllm_cache_check(c, _s(stream), ctypes.byref(w))
    if st != 0:
        raise DllmError("dllm_cache_check", st, lib().dllm_last_error().decode())
    return w.value


def dllm_cache_error_word(c, stream=None):
    """Like dllm_cache_check but returns the word instead of raising."""
    w = ctypes.c_uint32(0)
    st = lib().dllm_cache_check(c, _s(stream), ctypes.byref(w))
    if st not in (0, 4):
        _check("dllm_cache_check", st)
    return w.value


def dllm_state_copy(c, field, layer, host_tensor, to_device):
    """Blocking copy of a state field from/to a contiguous CPU tensor."""
    assert host_tensor.device.type == "cpu" and host_tensor.is_contiguous()
    nbytes = host_tensor.numel() * host_tensor.element_size()
    _check("dllm_state_copy", lib().dllm_state_copy(c, field, layer, _p(host_tensor), nbytes,
                                                     1 if to_device else 0, None))


def state_size(c, field, layer=0):
    n = _SZ(0)
    _check("dllm_state_copy", lib().dllm_state_copy(c, field, layer, None, 0, 0, ctypes.byref(n)))
    return n.value


def last_error():
    return lib().dllm_last_error().decode()


def refresh_all(c, q_start, rows, n_rows, stream=None):
    _check("refresh_all", lib().refresh_all(c, q_start, _p(rows), _p(n_rows), _s(stream)))


def kv_refresh(c, layer, x, tok, embed, w_qkv, rows, n_rows, t, stream=None):
    _check("kv_refresh", lib().kv_refresh(c, layer, _p(x), _p(tok), _p(embed), _p(w_qkv), _p(rows),
                                          _p(n_rows), t, _s(stream)))


def block_attn(c, layer, q_start, q_len, out, stream=None):
    _check("block_attn", lib().block_attn(c, layer, q_start, q_len, _p(out), _s(stream)))


def block_attn_rows(c, layer, q_rows, n_q, out, stream=None):
    _check("block_attn_rows", lib().block_attn_rows(c, layer, _p(q_rows), _p(n_q), _p(out), _s(stream)))


def active_rows(c, src, rows, n_rows, q_start, q_len, dst, stream=None):
    _check("active_rows", lib().active_rows(c, _p(src), _p(rows), _p(n_rows), q_start, q_len, _p(dst), _s(stream)))


def attn_out(c, o, w_o, x_res, tok, embed, q_start, q_len, m_dev, h, stream=None):
    _check("attn_out", lib().attn_out(c, _p(o), _p(w_o), _p(x_res), _p(tok), _p(embed), q_start, q_len,
                                      _p(m_dev), _p(h), _s(stream)))


def ffn_gelu(c, h, w1, w2, F, M, m_dev, out, stream=None):
    _check("ffn_gelu", lib().ffn_gelu(c, _p(h), _p(w1), _p(w2), F, M, _p(m_dev), _p(out), _s(stream)))


def lmhead_conf(c, h, w_lm, M, V, d, mask_id, argmax, p_top1, entropy, stream=None):
    _check("lmhead_conf", lib().lmhead_conf(c, _p(h), _p(w_lm), M, V, d, mask_id, _p(argmax), _p(p_top1),
                                            _p(entropy), _s(stream)))


def stab_update(c, argmax, p_top1, entropy, tok, q_start, t, step_in_block, last_step, rows, n_rows, stream=None):
    _check("stab_update", lib().stab_update(c, _p(argmax), _p(p_top1), _p(entropy), _p(tok), q_start, t,
                                            step_in_block, 1 if last_step else 0, _p(rows), _p(n_rows), _s(stream)))


def dllm_profile_events(c, kernel, ev_begin, ev_end):
    """Bracket the next launches of `kernel` with torch.cuda.Event pairs
    (None, None clears the hook)."""
    b = None if ev_begin is None else ctypes.c_void_p(ev_begin.cuda_event)
    e = None if ev_end is None else ctypes.c_void_p(ev_end.cuda_event)
    _check("dllm_profile_events", lib().dllm_profile_events(c, kernel, b, e))


def lmhead_conf_noalloc(h, w_lm, M, V, d, dtype, mask_id, rms_eps, argmax, p_top1, entropy, stream=None):
    """lmhead_conf without a handle or any device allocation (scratch in a
    static device array; M <= 256, V <= 131072; overlapping calls race)."""
    _check("lmhead_conf_noalloc", lib().lmhead_conf_noalloc(_p(h), _p(w_lm), M, V, d, dtype, mask_id,
                                                            ctypes.c_float(rms_eps), _p(argmax), _p(p_top1),
                                                            _p(entropy), _s(stream)))


def dllm_wait_selftest(c, limit_ns, stream=None):
    """One bounded wait on a barrier nothing arrives on (sets ERR_TIMEOUT)."""
    _check("dllm_wait_selftest", lib().dllm_wait_selftest(c, ctypes.c_uint64(limit_ns), _s(stream)))


def kv_project(c, layer, tok, embed, w_qkv, n, staged, stream=None):
    _check("kv_project", lib().kv_project(c, layer, _p(tok), _p(embed), _p(w_qkv), n, _p(staged), _s(stream)))


def ring_append(c, layer, staged, n0, count, stream=None):
    _check("ring_append", lib().ring_append(c, layer, _p(staged), n0, count, _s(stream)))
