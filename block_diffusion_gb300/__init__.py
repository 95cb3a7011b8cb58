"""Python binding of libbdlm: one block-diffusion denoising round on GB300 (sm_103a).

Argument marshalling only.  Every step of the round runs in the CUDA kernels of
``libbdlm.so``; torch tensors supply device memory and the current stream.  There is no
fallback: if the library is missing or the device is not sm_103 the calls raise.

Entry points mirror ``include/bdlm.h``:
    bdlm_block_attention, bdlm_lm_head, bdlm_confidence_commit, bdlm_confidence_commit_rule,
    bdlm_apply_commit, bdlm_status_string, bdlm_device_error, bdlm_release
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libbdlm.so")

BDLM_OK = 0
BDLM_ERR_INVALID = -1
BDLM_ERR_CUDA = -2
BDLM_ERR_UNSUPPORTED = -3
BDLM_ERR_NOMEM = -4

BDLM_DEVERR_PAGE = 1
BDLM_DEVERR_LENGTH = 2
BDLM_DEVERR_TIMEOUT = 4
BDLM_DEVERR_ROW = 8

BDLM_COMMIT_THRESHOLD = 0
BDLM_COMMIT_TOPK = 1
BDLM_COMMIT_SEQUENTIAL = 2
BDLM_COMMIT_ANTI_SEQUENTIAL = 3
BDLM_COMMIT_ENTROPY_BOUNDED = 4

EXPORTS = ("bdlm_block_attention", "bdlm_block_attention_kv", "bdlm_prefill_attention", "bdlm_lm_head", "bdlm_lm_head_device_count",
           "bdlm_lm_head_commit", "bdlm_active_rows", "bdlm_write_block_kv", "bdlm_confidence_commit",
           "bdlm_confidence_commit_rule", "bdlm_apply_commit", "bdlm_round_loop_create",
           "bdlm_round_loop_launch", "bdlm_round_loop_destroy", "bdlm_status_string",
           "bdlm_device_error", "bdlm_selftest_wait_timeout", "bdlm_release")


class AttnDesc(ctypes.Structure):
    """bdlm_attn_desc."""
    _fields_ = [("B", ctypes.c_int), ("L", ctypes.c_int), ("Hq", ctypes.c_int),
                ("Hkv", ctypes.c_int), ("D", ctypes.c_int), ("page_size", ctypes.c_int),
                ("max_pages_per_seq", ctypes.c_int), ("num_pages", ctypes.c_int),
                ("sm_scale", ctypes.c_float)]


class RoundLoopDesc(ctypes.Structure):
    """bdlm_round_loop_desc (device pointers as integers)."""
    _P = ctypes.c_void_p
    _fields_ = [("attn", AttnDesc), ("steps", ctypes.c_int), ("H", ctypes.c_int),
                ("V", ctypes.c_int), ("rule", ctypes.c_int), ("k", ctypes.c_int),
                ("threshold", ctypes.c_float), ("temperature", ctypes.c_float),
                ("q_steps", _P), ("k_new_steps", _P), ("v_new_steps", _P), ("hidden_steps", _P),
                ("k_pages", _P), ("v_pages", _P), ("page_table", _P), ("prefix_lens", _P),
                ("w", _P), ("mask", _P), ("denoising", _P), ("tok_steps", _P),
                ("conf_steps", _P), ("commit_steps", _P), ("steps_done", _P),
                ("attn_out_steps", _P)]


class BdlmError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {status} ({status_string(status)})")
        self.status = status


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libbdlm.so (built by ``block_diffusion_gb300.build``); raises if missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with block_diffusion_gb300.build.build()")
    lib = ctypes.CDLL(path)
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.bdlm_block_attention.argtypes = [ctypes.POINTER(AttnDesc), P, P, P, P, P, I, P, P]
    lib.bdlm_block_attention.restype = I
    lib.bdlm_block_attention_kv.argtypes = [ctypes.POINTER(AttnDesc), P, P, P, P, P, P, P, I, P,
                                            P]
    lib.bdlm_block_attention_kv.restype = I
    lib.bdlm_lm_head.argtypes = [P, P, P, I, I, I, I, P, P]
    lib.bdlm_lm_head.restype = I
    lib.bdlm_confidence_commit.argtypes = [P, P, I, I, I, F, F, P, P, P, P]
    lib.bdlm_confidence_commit.restype = I
    lib.bdlm_confidence_commit_rule.argtypes = [P, P, I, I, I, I, I, F, F, P, P, P, P, P]
    lib.bdlm_confidence_commit_rule.restype = I
    lib.bdlm_lm_head_device_count.argtypes = [P, P, P, P, I, I, I, I, P, P]
    lib.bdlm_lm_head_device_count.restype = I
    lib.bdlm_lm_head_commit.argtypes = [P, P, P, P, I, I, I, I, I, I, F, F, P, P, P, P, P, P]
    lib.bdlm_lm_head_commit.restype = I
    lib.bdlm_active_rows.argtypes = [P, P, I, I, P, P, P]
    lib.bdlm_active_rows.restype = I
    lib.bdlm_write_block_kv.argtypes = [ctypes.POINTER(AttnDesc), P, P, P, P, P, P, P]
    lib.bdlm_write_block_kv.restype = I
    lib.bdlm_prefill_attention.argtypes = [ctypes.POINTER(AttnDesc), I, P, P, P, P, P, P, P, P,
                                           P]
    lib.bdlm_prefill_attention.restype = I
    lib.bdlm_round_loop_create.argtypes = [ctypes.POINTER(RoundLoopDesc),
                                           ctypes.POINTER(ctypes.c_void_p)]
    lib.bdlm_round_loop_create.restype = I
    lib.bdlm_round_loop_launch.argtypes = [P, P]
    lib.bdlm_round_loop_launch.restype = I
    lib.bdlm_round_loop_destroy.argtypes = [P]
    lib.bdlm_round_loop_destroy.restype = I
    lib.bdlm_apply_commit.argtypes = [P, P, I, P]
    lib.bdlm_apply_commit.restype = I
    lib.bdlm_status_string.argtypes = [I]
    lib.bdlm_status_string.restype = ctypes.c_char_p
    lib.bdlm_device_error.argtypes = [ctypes.POINTER(ctypes.c_int)]
    lib.bdlm_device_error.restype = I
    lib.bdlm_selftest_wait_timeout.argtypes = [I, P]
    lib.bdlm_selftest_wait_timeout.restype = I
    lib.bdlm_release.argtypes = []
    lib.bdlm_release.restype = I
    _lib = lib
    return lib


def _ptr(x) -> int | None:
    """Device address of a torch tensor (or an int address, or None)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, rc: int) -> None:
    if rc != BDLM_OK:
        raise BdlmError(fn, rc)


def status_string(status: int) -> str:
    return load_library().bdlm_status_string(int(status)).decode()


bdlm_status_string = status_string


def bdlm_block_attention(desc: AttnDesc, q, k_pages, v_pages, page_table, prefix_lens, L: int,
                         out, stream=None) -> None:
    lib = load_library()
    rc = lib.bdlm_block_attention(ctypes.byref(desc), _ptr(q), _ptr(k_pages), _ptr(v_pages),
                                  _ptr(page_table), _ptr(prefix_lens), int(L), _ptr(out),
                                  _stream(stream))
    _check("bdlm_block_attention", rc)


def bdlm_block_attention_kv(desc: AttnDesc, q, k_new, v_new, k_pages, v_pages, page_table,
                            prefix_lens, L: int, out, stream=None) -> None:
    lib = load_library()
    rc = lib.bdlm_block_attention_kv(ctypes.byref(desc), _ptr(q), _ptr(k_new), _ptr(v_new),
                                     _ptr(k_pages), _ptr(v_pages), _ptr(page_table),
                                     _ptr(prefix_lens), int(L), _ptr(out), _stream(stream))
    _check("bdlm_block_attention_kv", rc)


def bdlm_prefill_attention(desc: AttnDesc, prompt_len: int, q, k_new, v_new, k_pages, v_pages,
                           page_table, prefix_lens, out, stream=None) -> None:
    lib = load_library()
    rc = lib.bdlm_prefill_attention(ctypes.byref(desc), int(prompt_len), _ptr(q), _ptr(k_new),
                                    _ptr(v_new), _ptr(k_pages), _ptr(v_pages), _ptr(page_table),
                                    _ptr(prefix_lens), _ptr(out), _stream(stream))
    _check("bdlm_prefill_attention", rc)


def bdlm_lm_head(hidden, w, active_idx, n_active: int, n_rows: int, H: int, V: int, logits,
                 stream=None) -> None:
    lib = load_library()
    rc = lib.bdlm_lm_head(_ptr(hidden), _ptr(w), _ptr(active_idx), int(n_active), int(n_rows),
                          int(H), int(V), _ptr(logits), _stream(stream))
    _check("bdlm_lm_head", rc)


def bdlm_confidence_commit(logits, mask, B: int, L: int, V: int, threshold: float,
                           temperature: float, tok_out, conf_out, commit_out, stream=None) -> None:
    lib = load_library()
    rc = lib.bdlm_confidence_commit(_ptr(logits), _ptr(mask), int(B), int(L), int(V),
                                    float(threshold), float(temperature), _ptr(tok_out),
                                    _ptr(conf_out), _ptr(commit_out), _stream(stream))
    _check("bdlm_confidence_commit", rc)


def bdlm_confidence_commit_rule(logits, mask, B: int, L: int, V: int, rule: int, k: int,
                                threshold: float, temperature: float, tok_out, conf_out,
                                commit_out, stream=None, entropy_out=None) -> None:
    """entropy_out (keyword; the C call takes it between conf_out and commit_out) may be None."""
    lib = load_library()
    rc = lib.bdlm_confidence_commit_rule(_ptr(logits), _ptr(mask), int(B), int(L), int(V),
                                         int(rule), int(k), float(threshold), float(temperature),
                                         _ptr(tok_out), _ptr(conf_out), _ptr(entropy_out),
                                         _ptr(commit_out), _stream(stream))
    _check("bdlm_confidence_commit_rule", rc)


def bdlm_lm_head_device_count(hidden, w, active_idx, n_active_dev, max_active: int, n_rows: int,
                              H: int, V: int, logits, stream=None) -> None:
    lib = load_library()
    rc = lib.bdlm_lm_head_device_count(_ptr(hidden), _ptr(w), _ptr(active_idx),
                                       _ptr(n_active_dev), int(max_active), int(n_rows), int(H),
                                       int(V), _ptr(logits), _stream(stream))
    _check("bdlm_lm_head_device_count", rc)


def bdlm_lm_head_commit(hidden, w, mask, denoising, B: int, L: int, H: int, V: int, rule: int,
                        k: int, threshold: float, temperature: float, tok_out, conf_out,
                        commit_out, logits=None, stream=None, entropy_out=None) -> None:
    """entropy_out (keyword; the C call takes it between conf_out and commit_out) may be None."""
    lib = load_library()
    rc = lib.bdlm_lm_head_commit(_ptr(hidden), _ptr(w), _ptr(mask), _ptr(denoising), int(B),
                                 int(L), int(H), int(V), int(rule), int(k), float(threshold),
                                 float(temperature), _ptr(tok_out), _ptr(conf_out),
                                 _ptr(entropy_out), _ptr(commit_out), _ptr(logits),
                                 _stream(stream))
    _check("bdlm_lm_head_commit", rc)


def bdlm_active_rows(mask, denoising, B: int, L: int, active_idx, n_active_dev,
                     stream=None) -> None:
    lib = load_library()
    rc = lib.bdlm_active_rows(_ptr(mask), _ptr(denoising), int(B), int(L), _ptr(active_idx),
                              _ptr(n_active_dev), _stream(stream))
    _check("bdlm_active_rows", rc)


def bdlm_write_block_kv(desc: AttnDesc, k_new, v_new, k_pages, v_pages, page_table, prefix_lens,
                        stream=None) -> None:
    lib = load_library()
    rc = lib.bdlm_write_block_kv(ctypes.byref(desc), _ptr(k_new), _ptr(v_new), _ptr(k_pages),
                                 _ptr(v_pages), _ptr(page_table), _ptr(prefix_lens),
                                 _stream(stream))
    _check("bdlm_write_block_kv", rc)


def round_loop_desc(attn: AttnDesc, steps: int, H: int, V: int, rule: int, k: int,
                    threshold: float, temperature: float, **ptrs) -> RoundLoopDesc:
    """A bdlm_round_loop_desc; ptrs are tensors (or None) for the pointer fields."""
    d = RoundLoopDesc()
    d.attn = attn
    d.steps, d.H, d.V, d.rule, d.k = int(steps), int(H), int(V), int(rule), int(k)
    d.threshold, d.temperature = float(threshold), float(temperature)
    for name, t in ptrs.items():
        setattr(d, name, _ptr(t))
    return d


def bdlm_round_loop_create(desc: RoundLoopDesc) -> int:
    lib = load_library()
    out = ctypes.c_void_p()
    rc = lib.bdlm_round_loop_create(ctypes.byref(desc), ctypes.byref(out))
    _check("bdlm_round_loop_create", rc)
    return out.value


def bdlm_round_loop_launch(loop: int, stream=None) -> None:
    _check("bdlm_round_loop_launch", load_library().bdlm_round_loop_launch(loop, _stream(stream)))


def bdlm_round_loop_destroy(loop: int) -> None:
    _check("bdlm_round_loop_destroy", load_library().bdlm_round_loop_destroy(loop))


def bdlm_apply_commit(mask, commit, n: int, stream=None) -> None:
    lib = load_library()
    _check("bdlm_apply_commit", lib.bdlm_apply_commit(_ptr(mask), _ptr(commit), int(n),
                                                      _stream(stream)))


def bdlm_device_error() -> int:
    lib = load_library()
    v = ctypes.c_int(0)
    _check("bdlm_device_error", lib.bdlm_device_error(ctypes.byref(v)))
    return int(v.value)


def bdlm_selftest_wait_timeout(limit_us: int, stream=None) -> None:
    _check("bdlm_selftest_wait_timeout",
           load_library().bdlm_selftest_wait_timeout(int(limit_us), _stream(stream)))


def bdlm_release() -> None:
    _check("bdlm_release", load_library().bdlm_release())


def attn_desc(B, L, Hq, Hkv, D, max_pages_per_seq, num_pages, page_size=16, sm_scale=0.0):
    return AttnDesc(int(B), int(L), int(Hq), int(Hkv), int(D), int(page_size),
                    int(max_pages_per_seq), int(num_pages), float(sm_scale))
