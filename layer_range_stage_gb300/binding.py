"""ctypes binding of libstage.so: the C ABI of include/stage.h with the same names.

Argument marshalling only.  Every step of the stage forward runs in the library's CUDA
kernels; nothing here computes.  Device buffers are PyTorch tensors (PyTorch provides
device memory and the stream); host arrays are numpy arrays.  If the library has not
been built this module raises on load: there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional, Sequence

import numpy as np

from . import build as _build

STAGE_OK = 0
STAGE_E_INVALID = -1
STAGE_E_DOES_NOT_FIT = -2
STAGE_E_HANDOFF = -3
STAGE_E_POSITION = -4
STAGE_E_BUSY = -5
STAGE_E_NOT_LAST = -6
STAGE_E_CUDA = -7
STAGE_E_STATE = -8
STAGE_E_INJECTED = -9
STAGE_E_HOST = -10
ERROR_NAMES = {0: "STAGE_OK", -1: "STAGE_E_INVALID", -2: "STAGE_E_DOES_NOT_FIT", -3: "STAGE_E_HANDOFF",
               -4: "STAGE_E_POSITION", -5: "STAGE_E_BUSY", -6: "STAGE_E_NOT_LAST", -7: "STAGE_E_CUDA",
               -8: "STAGE_E_STATE", -9: "STAGE_E_INJECTED", -10: "STAGE_E_HOST"}


class StageError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERROR_NAMES.get(code, code)}: {msg}")
        self.code = code


class stage_model_cfg(C.Structure):
    _fields_ = [(n, C.c_int) for n in ("n_layers", "hidden", "n_q_heads", "n_kv_heads", "head_dim", "ffn", "vocab",
                                       "n_experts", "top_k", "expert_ffn")] + \
               [("rms_eps", C.c_float), ("rope_theta", C.c_float)] + \
               [(n, C.c_int) for n in ("max_seqs", "max_seq_len", "max_tokens", "gemm_bf16_min_tokens", "shared_ffn")]


class stage_layer_range(C.Structure):
    _fields_ = [("begin", C.c_int), ("end", C.c_int)]


class stage_q8(C.Structure):
    _fields_ = [("q", C.c_void_p), ("scale", C.c_void_p), ("rows", C.c_int64), ("cols", C.c_int64)]


class stage_layer_w(C.Structure):
    _fields_ = [("attn_norm", C.c_void_p), ("ffn_norm", C.c_void_p)] + \
               [(n, stage_q8) for n in ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down", "router")] + \
               [("e_gate", C.c_void_p), ("e_up", C.c_void_p), ("e_down", C.c_void_p)] + \
               [(n, stage_q8) for n in ("shared_score", "shared_gate", "shared_up", "shared_down")]


class stage_weights(C.Structure):
    _fields_ = [("embed", stage_q8), ("final_norm", C.c_void_p), ("lm_head", stage_q8), ("layers", C.c_void_p)]


class stage_act(C.Structure):
    _fields_ = [("data", C.c_void_p), ("rows", C.c_int), ("cols", C.c_int)]


_lib = None

_SIGS = {
    "stage_required_bytes": (C.c_size_t, [C.POINTER(stage_model_cfg), stage_layer_range]),
    "stage_plan_placement": (C.c_int, [C.POINTER(stage_model_cfg), C.c_int, C.POINTER(C.c_size_t),
                                       C.POINTER(C.c_int32), C.POINTER(C.c_size_t)]),
    "stage_create": (C.c_int, [C.POINTER(stage_model_cfg), stage_layer_range, C.c_void_p, C.c_size_t, C.c_void_p,
                               C.POINTER(C.c_void_p)]),
    "stage_load_layer": (C.c_int, [C.c_void_p, C.c_int, C.c_void_p]),
    "stage_load_endpoints": (C.c_int, [C.c_void_p, C.c_void_p]),
    "stage_prefill": (C.c_int, [C.c_void_p, C.c_int, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p]),
    "stage_decode": (C.c_int, [C.c_void_p, C.c_int, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p]),
    "stage_logits": (C.c_int, [C.c_void_p, C.c_int, C.c_void_p, C.c_void_p, C.c_void_p]),
    "stage_commit": (C.c_int, [C.c_void_p, C.c_int, C.c_void_p, C.c_void_p]),
    "stage_truncate": (C.c_int, [C.c_void_p, C.c_int, C.c_int]),
    "stage_reset": (C.c_int, [C.c_void_p]),
    "stage_committed_len": (C.c_int, [C.c_void_p, C.c_int, C.POINTER(C.c_int)]),
    "stage_gemm_mode": (C.c_int, [C.c_void_p, C.c_int, C.POINTER(C.c_int)]),
    "stage_read_kv": (C.c_int, [C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_void_p, C.c_void_p]),
    "stage_write_kv": (C.c_int, [C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_int, C.c_void_p, C.c_void_p]),
    "stage_last_error": (C.c_char_p, [C.c_void_p]),
    "stage_create_error": (C.c_char_p, []),
    "stage_destroy": (None, [C.c_void_p]),
    "stage_debug_inject": (C.c_int, [C.c_void_p, C.c_int, C.c_int]),
    "stage_pipeline_create": (C.c_int, [C.c_void_p, C.c_int, C.POINTER(C.c_void_p)]),
    "stage_pipeline_step": (C.c_int, [C.c_void_p, C.c_int, C.c_int, C.c_void_p, C.c_void_p, C.c_void_p, C.c_int,
                                      C.c_void_p, C.c_void_p, C.c_void_p]),
    "stage_pipeline_generate": (C.c_int, [C.c_void_p, C.c_int, C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_void_p]),
    "stage_pipeline_handoff_stats": (C.c_int, [C.c_void_p, C.c_int, C.POINTER(C.c_int64), C.POINTER(C.c_int64)]),
    "stage_pipeline_kernel_timing": (C.c_int, [C.c_void_p, C.c_int]),
    "stage_pipeline_kernel_time": (C.c_int, [C.c_void_p, C.POINTER(C.c_float), C.POINTER(C.c_int)]),
    "stage_pipeline_last_error": (C.c_char_p, [C.c_void_p]),
    "stage_pipeline_destroy": (None, [C.c_void_p]),
    "stage_op_q8_device_bytes": (C.c_int, [C.c_int64, C.c_int64, C.POINTER(C.c_size_t), C.POINTER(C.c_size_t)]),
    "stage_op_q8_pack": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p]),
    "stage_op_embed": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int64, C.c_int64, C.c_void_p, C.c_int, C.c_void_p,
                                 C.c_void_p]),
    "stage_op_gemv": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int64, C.c_int64, C.c_void_p, C.c_int, C.c_void_p,
                                C.c_float, C.c_void_p, C.c_void_p]),
    "stage_op_attention_workspace_bytes": (C.c_size_t, [C.c_int] * 5),
    "stage_op_gemm_bf16": (C.c_int, [C.c_void_p, C.c_int, C.c_int, C.c_void_p, C.c_void_p, C.c_int64, C.c_int64,
                                     C.c_void_p, C.c_void_p]),
    "stage_op_attention_decode": (C.c_int, [C.c_void_p] * 5 + [C.c_int] * 6 + [C.c_void_p, C.c_void_p, C.c_size_t,
                                                                              C.c_void_p]),
    "stage_op_attention_decode_static": (C.c_int, [C.c_void_p] * 5 + [C.c_int] * 6 + [C.c_void_p, C.c_void_p]),
    "stage_op_last_error": (C.c_char_p, []),
}


def declared_symbols() -> list:
    """Every function the headers in include/ declare (parsed from the headers)."""
    import re
    names = []
    inc = os.path.join(_build.ROOT, "include")
    for h in sorted(os.listdir(inc)):
        if h.endswith(".h"):
            names += re.findall(r"^STAGE_API [^(]*?\b(stage_\w+)\(", open(os.path.join(inc, h)).read(), flags=re.M)
    return names


def lib():
    """Load libstage.so (built by __graft_entry__.build()).  Raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(_build.LIB):
            raise ImportError(f"{_build.LIB} is not built: run __graft_entry__.build() (nvcc, sm_103a)")
        # make libcudart resolvable even when PyTorch has not loaded it yet
        try:
            C.CDLL(os.path.join(_build.cuda_lib_dir(), "libcudart.so"), mode=C.RTLD_GLOBAL)
        except OSError:
            pass
        L = C.CDLL(_build.LIB)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


# ----------------------------------------------------------------------------- marshalling

def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


def make_cfg(model, max_seqs: int, max_seq_len: int, max_tokens: int, gemm_bf16_min_tokens: int = 0) -> stage_model_cfg:
    """stage_model_cfg from any object with the model's shape fields (e.g. synth.ModelCfg)."""
    return stage_model_cfg(model.n_layers, model.hidden, model.n_q_heads, model.n_kv_heads, model.head_dim,
                           model.ffn, model.vocab, model.n_experts, model.top_k, model.expert_ffn,
                           model.rms_eps, model.rope_theta, max_seqs, max_seq_len, max_tokens, gemm_bf16_min_tokens,
                           getattr(model, "shared_ffn", 0))


class _Keep:
    """Holds the numpy arrays behind a stage_weights so their memory outlives the call."""

    def __init__(self):
        self.refs = []

    def q8(self, m) -> stage_q8:
        if m is None:
            return stage_q8(None, None, 0, 0)
        q = np.ascontiguousarray(m.q, dtype=np.int8)
        s = np.ascontiguousarray(m.s, dtype=np.uint16)
        self.refs += [q, s]
        return stage_q8(q.ctypes.data, s.ctypes.data, q.shape[0], q.shape[1])

    def f32(self, a):
        if a is None:
            return None
        a = np.ascontiguousarray(a, dtype=np.float32)
        self.refs.append(a)
        return a.ctypes.data

    def layer(self, lw) -> stage_layer_w:
        w = stage_layer_w()
        w.attn_norm, w.ffn_norm = self.f32(lw.attn_norm), self.f32(lw.ffn_norm)
        for n in ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down", "router", "shared_score", "shared_gate",
                  "shared_up", "shared_down"):
            setattr(w, n, self.q8(getattr(lw, n, None)))
        for n in ("e_gate", "e_up", "e_down"):
            mats = getattr(lw, n, None) or []
            if mats:
                arr = (stage_q8 * len(mats))(*[self.q8(m) for m in mats])
                self.refs.append(arr)
                setattr(w, n, C.cast(arr, C.c_void_p))
            else:
                setattr(w, n, None)
        return w

    def weights(self, sw) -> stage_weights:
        w = stage_weights()
        w.embed = self.q8(sw.embed)
        w.final_norm = self.f32(sw.final_norm)
        w.lm_head = self.q8(sw.lm_head)
        if sw.layers:
            arr = (stage_layer_w * len(sw.layers))(*[self.layer(l) for l in sw.layers])
            self.refs.append(arr)
            w.layers = C.cast(arr, C.c_void_p)
        return w


def _act(t) -> Optional[stage_act]:
    if t is None:
        return None
    if t.dtype.__str__() != "torch.float32" or not t.is_cuda or not t.is_contiguous() or t.dim() != 2:
        raise StageError(STAGE_E_HANDOFF, "hidden activations are contiguous float32 CUDA tensors [n, hidden]")
    return stage_act(t.data_ptr(), t.shape[0], t.shape[1])


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return int(stream) if not hasattr(stream, "cuda_stream") else stream.cuda_stream


# ----------------------------------------------------------------------------- functions (same names as the C ABI)

def stage_required_bytes(cfg: stage_model_cfg, begin: int, end: int) -> int:
    return int(lib().stage_required_bytes(C.byref(cfg), stage_layer_range(begin, end)))


def stage_plan_placement(cfg: stage_model_cfg, budgets) -> tuple:
    """Block bounds [n_devices + 1] and each stage's required bytes for the given per-device
    budgets (see include/stage.h); raises StageError (DoesNotFit when no placement is legal)."""
    n = len(budgets)
    bud = (C.c_size_t * max(n, 1))(*[int(b) for b in budgets])
    bounds = (C.c_int32 * (n + 1))()
    req = (C.c_size_t * max(n, 1))()
    rc = lib().stage_plan_placement(C.byref(cfg), n, bud, bounds, req)
    if rc != STAGE_OK:
        raise StageError(rc, "no legal placement" if rc == STAGE_E_DOES_NOT_FIT else "invalid placement request")
    return [int(b) for b in bounds], [int(r) for r in req[:n]]


def stage_create(cfg: stage_model_cfg, begin: int, end: int, weights=None, budget: Optional[int] = None, stream=None):
    """Returns a stage handle (int).  ``weights``: an object shaped like synth.StageWeights or None."""
    keep = _Keep()
    wp = C.byref(keep.weights(weights)) if weights is not None else None
    h = C.c_void_p()
    budget = (1 << 62) if budget is None else int(budget)
    rc = lib().stage_create(C.byref(cfg), stage_layer_range(begin, end), wp, budget, _stream(stream), C.byref(h))
    if rc != STAGE_OK:
        raise StageError(rc, lib().stage_create_error().decode())
    return h.value


def _check(st, rc):
    if rc != STAGE_OK:
        raise StageError(rc, lib().stage_last_error(st).decode())


def stage_load_layer(st, global_layer: int, layer_weights) -> None:
    keep = _Keep()
    lw = keep.layer(layer_weights)
    _check(st, lib().stage_load_layer(st, global_layer, C.byref(lw)))


def stage_load_endpoints(st, weights) -> None:
    keep = _Keep()
    w = keep.weights(weights)
    _check(st, lib().stage_load_endpoints(st, C.byref(w)))


def _fwd(fn, st, seq_ids, positions, tokens, hidden_in, hidden_out):
    seq, pos = _i32(seq_ids), _i32(positions)
    tok = None if tokens is None else _i32(tokens)
    hin, hout = _act(hidden_in), _act(hidden_out)
    rc = fn(st, len(pos), _ptr(seq), _ptr(pos), _ptr(tok), C.byref(hin) if hin else None,
            C.byref(hout) if hout else None)
    _check(st, rc)


def stage_prefill(st, seq_ids, positions, tokens=None, hidden_in=None, hidden_out=None) -> None:
    _fwd(lib().stage_prefill, st, seq_ids, positions, tokens, hidden_in, hidden_out)


def stage_decode(st, seq_ids, positions, tokens=None, hidden_in=None, hidden_out=None) -> None:
    _fwd(lib().stage_decode, st, seq_ids, positions, tokens, hidden_in, hidden_out)


def stage_logits(st, row_index: Sequence[int], logits_out=None, argmax_out=None) -> None:
    rows = _i32(row_index)
    lp = None if logits_out is None else logits_out.data_ptr()
    ap = None if argmax_out is None else argmax_out.data_ptr()
    _check(st, lib().stage_logits(st, len(rows), _ptr(rows), lp, ap))


def stage_commit(st, seq_ids, new_len) -> None:
    s, n = _i32(seq_ids), _i32(new_len)
    _check(st, lib().stage_commit(st, len(s), _ptr(s), _ptr(n)))


def stage_truncate(st, seq_id: int, length: int) -> None:
    _check(st, lib().stage_truncate(st, seq_id, length))


def stage_reset(st) -> None:
    _check(st, lib().stage_reset(st))


def stage_committed_len(st, seq_id: int) -> int:
    v = C.c_int()
    _check(st, lib().stage_committed_len(st, seq_id, C.byref(v)))
    return v.value


def stage_read_kv(st, global_layer: int, seq_id: int, n_pos: int, n_kv_heads: int, head_dim: int):
    """(K, V) of one owned block and sequence as float16 [n_kv_heads, n_pos, head_dim]."""
    k = np.zeros((n_kv_heads, n_pos, head_dim), dtype=np.uint16)
    v = np.zeros_like(k)
    _check(st, lib().stage_read_kv(st, global_layer, seq_id, n_pos, _ptr(k), _ptr(v)))
    return k.view(np.float16), v.view(np.float16)


def stage_write_kv(st, global_layer: int, seq_id: int, pos0: int, k, v) -> None:
    """Write (K, V) float16 [n_kv_heads, n_pos, head_dim] at positions pos0.. of one owned
    block and sequence."""
    k = np.ascontiguousarray(np.asarray(k, dtype=np.float16)).view(np.uint16)
    v = np.ascontiguousarray(np.asarray(v, dtype=np.float16)).view(np.uint16)
    if k.shape != v.shape or k.ndim != 3:
        raise ValueError("k and v must both be [n_kv_heads, n_pos, head_dim]")
    _check(st, lib().stage_write_kv(st, global_layer, seq_id, pos0, k.shape[1], _ptr(k), _ptr(v)))


def stage_gemm_mode(st, n_tokens: int) -> int:
    v = C.c_int()
    _check(st, lib().stage_gemm_mode(st, n_tokens, C.byref(v)))
    return v.value


def stage_last_error(st) -> str:
    return lib().stage_last_error(st).decode()


def stage_create_error() -> str:
    return lib().stage_create_error().decode()


def stage_destroy(st) -> None:
    lib().stage_destroy(st)


def stage_debug_inject(st, what: int, value: int) -> None:
    _check(st, lib().stage_debug_inject(st, what, value))


def _pcheck(p, rc):
    if rc != STAGE_OK:
        raise StageError(rc, lib().stage_pipeline_last_error(p).decode())


def stage_pipeline_create(stages: Sequence[int]):
    arr = (C.c_void_p * len(stages))(*stages)
    h = C.c_void_p()
    rc = lib().stage_pipeline_create(arr, len(stages), C.byref(h))
    if rc != STAGE_OK:
        raise StageError(rc, "stages must tile [0, n_layers) in order with one model, device and stream")
    return h.value


def stage_pipeline_step(p, is_prefill: bool, seq_ids, positions, tokens, row_index=(), logits_out=None,
                        want_tokens: bool = True):
    seq, pos, tok = _i32(seq_ids), _i32(positions), _i32(tokens)
    rows = _i32(row_index)
    nxt = np.zeros(len(rows), dtype=np.int32) if (want_tokens and len(rows)) else None
    lp = None if logits_out is None else logits_out.data_ptr()
    rc = lib().stage_pipeline_step(p, int(bool(is_prefill)), len(pos), _ptr(seq), _ptr(pos), _ptr(tok), len(rows),
                                   _ptr(rows) if len(rows) else None, lp, _ptr(nxt))
    _pcheck(p, rc)
    return nxt


def stage_pipeline_generate(p, seq_ids, first_tokens, n_steps: int, use_graph: bool = True) -> np.ndarray:
    seq, tok = _i32(seq_ids), _i32(first_tokens)
    out = np.zeros((n_steps, len(seq)), dtype=np.int32)
    _pcheck(p, lib().stage_pipeline_generate(p, len(seq), _ptr(seq), _ptr(tok), n_steps, int(bool(use_graph)), _ptr(out)))
    return out


def stage_pipeline_handoff_stats(p, boundary: int):
    c, b = C.c_int64(), C.c_int64()
    _pcheck(p, lib().stage_pipeline_handoff_stats(p, boundary, C.byref(c), C.byref(b)))
    return c.value, b.value


def stage_pipeline_kernel_timing(p, enable: bool) -> None:
    _pcheck(p, lib().stage_pipeline_kernel_timing(p, int(bool(enable))))


def stage_pipeline_kernel_time(p):
    """(mean microseconds, count) of the FFN up-projection launches of the last timed step."""
    m, n = C.c_float(), C.c_int()
    _pcheck(p, lib().stage_pipeline_kernel_time(p, C.byref(m), C.byref(n)))
    return m.value, n.value


def stage_pipeline_last_error(p) -> str:
    return lib().stage_pipeline_last_error(p).decode()


def stage_pipeline_destroy(p) -> None:
    lib().stage_pipeline_destroy(p)


# ----------------------------------------------------------------------------- kernel-level entry points

def stage_op_last_error() -> str:
    return lib().stage_op_last_error().decode()


def _opcheck(rc):
    if rc != STAGE_OK:
        raise StageError(rc, lib().stage_op_last_error().decode())


def stage_op_q8_device_bytes(rows: int, cols: int):
    qb, sb = C.c_size_t(), C.c_size_t()
    _opcheck(lib().stage_op_q8_device_bytes(rows, cols, C.byref(qb), C.byref(sb)))
    return qb.value, sb.value


def stage_op_q8_pack(m, q_dev, s_dev) -> None:
    keep = _Keep()
    h = keep.q8(m)
    _opcheck(lib().stage_op_q8_pack(C.byref(h), q_dev.data_ptr(), s_dev.data_ptr()))


def stage_op_embed(q_dev, s_dev, rows: int, cols: int, tok, out, stream=None) -> None:
    """tok: int32 device tensor [n_tok]; out: f32 device tensor [n_tok, cols]."""
    _opcheck(lib().stage_op_embed(q_dev.data_ptr(), s_dev.data_ptr(), rows, cols, tok.data_ptr(), tok.shape[0],
                                  out.data_ptr(), _stream(stream)))


def stage_op_gemv(q_dev, s_dev, rows: int, cols: int, x, y, gamma=None, eps: float = 1e-5, stream=None) -> None:
    _opcheck(lib().stage_op_gemv(q_dev.data_ptr(), s_dev.data_ptr(), rows, cols, x.data_ptr(), x.shape[0],
                                 None if gamma is None else gamma.data_ptr(), eps, y.data_ptr(), _stream(stream)))


def stage_op_gemm_bf16(a_bits, q_dev, s_dev, rows: int, cols: int, y, stream=None) -> None:
    """a_bits: int16/uint16 device tensor [M, lda] of bf16 bit patterns; y: f32 [M, rows]."""
    M, lda = a_bits.shape
    _opcheck(lib().stage_op_gemm_bf16(a_bits.data_ptr(), lda, M, q_dev.data_ptr(), s_dev.data_ptr(), rows, cols,
                                      y.data_ptr(), _stream(stream)))


def stage_op_attention_workspace_bytes(n_tok, n_q_heads, n_kv_heads, head_dim, n_chunks) -> int:
    return int(lib().stage_op_attention_workspace_bytes(n_tok, n_q_heads, n_kv_heads, head_dim, n_chunks))


def stage_op_attention_decode(q, k_cache, v_cache, seq, pos, out, n_chunks: int, workspace, stream=None) -> None:
    """q [n_tok, Hq, D] f32; k/v_cache [seqs, Hkv, max_len, D] f16; seq/pos int32 [n_tok] (device tensors)."""
    n_tok, hq, d = q.shape
    hkv, max_len = k_cache.shape[1], k_cache.shape[2]
    _opcheck(lib().stage_op_attention_decode(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), seq.data_ptr(),
                                             pos.data_ptr(), n_tok, hq, hkv, d, max_len, n_chunks, out.data_ptr(),
                                             workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                             _stream(stream)))


def stage_op_attention_decode_static(q, k_cache, v_cache, seq, pos, out, n_chunks: int, stream=None) -> None:
    """stage_op_attention_decode without a workspace: scratch is the library's fixed array
    (no device allocation; calls must not overlap on the GPU)."""
    n_tok, hq, d = q.shape
    hkv, max_len = k_cache.shape[1], k_cache.shape[2]
    _opcheck(lib().stage_op_attention_decode_static(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                                    seq.data_ptr(), pos.data_ptr(), n_tok, hq, hkv, d, max_len,
                                                    n_chunks, out.data_ptr(), _stream(stream)))
