"""Seeded synthetic inputs for the layer-range stage: model shapes, weights, gains, prompts.

This module is input generation only.  Both the CPU oracle and the CUDA path
consume the arrays it returns; it holds none of the stage's arithmetic.  The
generator itself (SplitMix64 used counter-style, Box-Muller normals, the int8
block-32 quantiser) is in ``gen.c`` and is compiled here on first use.

Every tensor is addressed by ``(seed, config id, layer, tensor id, expert)`` so a
stage can generate exactly the tensors it owns and nothing else -- the pages'
rule that each stage imports only its own weights ("RFC: pipeline placement
across multiple GPUs for models larger than one device", section "Larger-than-
single-card proof"; "Multi-node layer splitting and tensor parallelism",
section "Supported stage executors").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field, replace
from typing import Dict, List, Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_DIR = os.path.join(_HERE, "_lib")
_LIB_PATH = os.path.join(_LIB_DIR, "libsynth.so")
_lib = None
_lib_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile gen.c into synth/_lib/libsynth.so (plain gcc, no GPU)."""
    src = os.path.join(_HERE, "gen.c")
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(src):
        return _LIB_PATH
    os.makedirs(_LIB_DIR, exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-shared", "-fPIC", "-pthread", "-o", tmp, src, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lib_lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, u64, dbl = ctypes.c_int64, ctypes.c_uint64, ctypes.c_double
            vp = ctypes.c_void_p
            lib.synth_key.restype = u64
            lib.synth_key.argtypes = [vp, ctypes.c_int]
            lib.synth_normal_f32.restype = None
            lib.synth_normal_f32.argtypes = [u64, i64, i64, dbl, dbl, vp]
            lib.synth_q8.restype = ctypes.c_int
            lib.synth_q8.argtypes = [u64, i64, i64, i64, dbl, vp, vp, ctypes.c_int]
            lib.synth_quantize.restype = None
            lib.synth_quantize.argtypes = [vp, i64, i64, vp, vp]
            lib.synth_uniform_int.restype = None
            lib.synth_uniform_int.argtypes = [u64, i64, i64, i64, vp]
            lib.synth_f32_to_f16.restype = None
            lib.synth_f32_to_f16.argtypes = [vp, i64, vp]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


# ----------------------------------------------------------------------------- model shapes

@dataclass(frozen=True)
class ModelCfg:
    """Shape of a decoder (all sizes in elements)."""
    name: str
    cfg_id: int
    n_layers: int
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    n_experts: int = 0
    top_k: int = 0
    expert_ffn: int = 0
    rms_eps: float = 1e-5
    rope_theta: float = 10000.0
    shared_ffn: int = 0  # MoE only: width of the shared expert (0 = none)

    @property
    def is_moe(self) -> bool:
        return self.n_experts > 0

    @property
    def q_dim(self) -> int:
        return self.n_q_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim


# The five workloads of the stage forward.  ``splits`` are the block boundaries of
# the stages; the pages' own 40-block split is 0..20 / 21..39 ("RFC: pipeline
# placement ...", section "Larger-than-single-card proof").
CONFIGS: Dict[int, ModelCfg] = {
    0: ModelCfg("tiny-dense-4L", 0, 4, 256, 4, 2, 64, 688, 1024),
    1: ModelCfg("dense-8B-shape", 1, 32, 4096, 32, 8, 128, 14336, 32000),
    2: ModelCfg("moe-40L-A3B-like", 2, 40, 2048, 32, 4, 128, 0, 151936, n_experts=128, top_k=8, expert_ffn=768),
    3: ModelCfg("dense-8B-shape-prefill", 3, 32, 4096, 32, 8, 128, 14336, 32000),
    4: ModelCfg("dense-70B-shape", 4, 80, 8192, 64, 8, 128, 28672, 128256),
}
SPLITS: Dict[int, List[int]] = {0: [0, 2, 4], 1: [0, 16, 32], 2: [0, 21, 40], 3: [0, 16, 32], 4: [0, 20, 40, 60, 80]}

# The book chapter's CPU pipeline run: 4 layers, hidden 512, 8 query / 4 KV heads,
# vocabulary 1024 ("41. Many GPUs ...", section "Measured").  Its FFN width is not
# printed; 1376 is used where a width is needed.
BOOK_CPU = ModelCfg("book-cpu-4L", 9, 4, 512, 8, 4, 64, 1376, 1024)

# tensor ids of the stream keys
T_EMBED, T_HEAD, T_FINAL_NORM = 0, 1, 2
T_ATTN_NORM, T_FFN_NORM, T_WQ, T_WK, T_WV, T_WO = 10, 11, 12, 13, 14, 15
T_GATE, T_UP, T_DOWN, T_ROUTER, T_EGATE, T_EUP, T_EDOWN = 16, 17, 18, 19, 20, 21, 22
T_SSCORE, T_SGATE, T_SUP, T_SDOWN = 23, 24, 25, 26
T_PROMPT, T_KVFILL = 100, 101

WEIGHT_SIGMA = 0.02
GAMMA_SIGMA = 0.1
DEFAULT_SEED = 1234


def key(*fields: int) -> int:
    arr = np.asarray(fields, dtype=np.int64)
    return int(_load().synth_key(_ptr(arr), len(arr)))


def tensor_key(seed: int, cfg_id: int, layer: int, tensor: int, expert: int = 0) -> int:
    return key(seed, cfg_id, layer, tensor, expert)


def n_threads_default() -> int:
    return max(1, os.cpu_count() or 1)


def q8(k: int, rows: int, cols: int, row0: int = 0, nrows: Optional[int] = None,
       sigma: float = WEIGHT_SIGMA, n_threads: Optional[int] = None) -> Tuple[np.ndarray, np.ndarray]:
    """Rows [row0, row0+nrows) of a quantised N(0, sigma) [rows x cols] matrix.

    Returns (q int8 [nrows, cols], s uint16 fp16-bits [nrows, ceil(cols/32)]); when
    cols % 32 != 0 the last block of each row is partial."""
    nrows = rows - row0 if nrows is None else nrows
    if row0 < 0 or nrows < 0 or row0 + nrows > rows:
        raise ValueError("row range out of bounds")
    q = np.empty((nrows, cols), dtype=np.int8)
    s = np.empty((nrows, (cols + 31) // 32), dtype=np.uint16)
    rc = _load().synth_q8(k, cols, row0, nrows, sigma, _ptr(q), _ptr(s), n_threads or n_threads_default())
    if rc != 0:
        raise RuntimeError("synth_q8 failed")
    return q, s


def normal_f32(k: int, start: int, count: int, sigma: float, mean: float = 0.0) -> np.ndarray:
    out = np.empty(count, dtype=np.float32)
    _load().synth_normal_f32(k, start, count, sigma, mean, _ptr(out))
    return out


def quantize(w: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Block-32 quantiser over the last axis of a float32 array (last block may be partial)."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    cols = w.shape[-1]
    q = np.empty(w.shape, dtype=np.int8)
    s = np.empty(w.shape[:-1] + ((cols + 31) // 32,), dtype=np.uint16)
    _load().synth_quantize(_ptr(w), w.size // cols, cols, _ptr(q), _ptr(s))
    return q, s


def uniform_int(k: int, start: int, count: int, n: int) -> np.ndarray:
    out = np.empty(count, dtype=np.int32)
    _load().synth_uniform_int(k, start, count, n, _ptr(out))
    return out


def f32_to_f16_bits(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().synth_f32_to_f16(_ptr(x), x.size, _ptr(out))
    return out


# ----------------------------------------------------------------------------- weight sets

@dataclass
class Q8:
    """An int8 block-32 matrix: q [rows, cols] int8, s [rows, ceil(cols/32)] fp16 bits (uint16)."""
    q: np.ndarray
    s: np.ndarray

    @property
    def rows(self) -> int:
        return self.q.shape[0]

    @property
    def cols(self) -> int:
        return self.q.shape[1]


@dataclass
class LayerWeights:
    attn_norm: np.ndarray
    ffn_norm: np.ndarray
    wq: Q8
    wk: Q8
    wv: Q8
    wo: Q8
    w_gate: Optional[Q8] = None
    w_up: Optional[Q8] = None
    w_down: Optional[Q8] = None
    router: Optional[Q8] = None
    e_gate: List[Q8] = field(default_factory=list)
    e_up: List[Q8] = field(default_factory=list)
    e_down: List[Q8] = field(default_factory=list)
    shared_score: Optional[Q8] = None  # [1 x hidden], the shared expert's scalar gate
    shared_gate: Optional[Q8] = None
    shared_up: Optional[Q8] = None
    shared_down: Optional[Q8] = None


@dataclass
class StageWeights:
    """Exactly the tensors a stage over blocks [begin, end) owns."""
    cfg: ModelCfg
    begin: int
    end: int
    layers: List[LayerWeights]
    embed: Optional[Q8] = None
    final_norm: Optional[np.ndarray] = None
    lm_head: Optional[Q8] = None


def gamma(seed: int, cfg: ModelCfg, layer: int, tensor: int, mode: str) -> np.ndarray:
    """RMSNorm gain: all ones ("ones") or 1 + N(0, 0.1) ("seeded")."""
    if mode == "ones":
        return np.ones(cfg.hidden, dtype=np.float32)
    if mode == "seeded":
        return normal_f32(tensor_key(seed, cfg.cfg_id, layer, tensor), 0, cfg.hidden, GAMMA_SIGMA, 1.0)
    raise ValueError(mode)


def layer_weights(cfg: ModelCfg, layer: int, seed: int = DEFAULT_SEED, gamma_mode: str = "ones",
                  n_threads: Optional[int] = None) -> LayerWeights:
    c, l = cfg, layer

    def mat(t, rows, cols, e=0):
        return Q8(*q8(tensor_key(seed, c.cfg_id, l, t, e), rows, cols, n_threads=n_threads))

    lw = LayerWeights(
        attn_norm=gamma(seed, c, l, T_ATTN_NORM, gamma_mode),
        ffn_norm=gamma(seed, c, l, T_FFN_NORM, gamma_mode),
        wq=mat(T_WQ, c.q_dim, c.hidden), wk=mat(T_WK, c.kv_dim, c.hidden), wv=mat(T_WV, c.kv_dim, c.hidden),
        wo=mat(T_WO, c.hidden, c.q_dim))
    if c.is_moe:
        lw.router = mat(T_ROUTER, c.n_experts, c.hidden)
        for e in range(c.n_experts):
            lw.e_gate.append(mat(T_EGATE, c.expert_ffn, c.hidden, e))
            lw.e_up.append(mat(T_EUP, c.expert_ffn, c.hidden, e))
            lw.e_down.append(mat(T_EDOWN, c.hidden, c.expert_ffn, e))
        if c.shared_ffn:
            lw.shared_score = mat(T_SSCORE, 1, c.hidden)
            lw.shared_gate = mat(T_SGATE, c.shared_ffn, c.hidden)
            lw.shared_up = mat(T_SUP, c.shared_ffn, c.hidden)
            lw.shared_down = mat(T_SDOWN, c.hidden, c.shared_ffn)
    else:
        lw.w_gate = mat(T_GATE, c.ffn, c.hidden)
        lw.w_up = mat(T_UP, c.ffn, c.hidden)
        lw.w_down = mat(T_DOWN, c.hidden, c.ffn)
    return lw


def stage_weights(cfg: ModelCfg, begin: int, end: int, seed: int = DEFAULT_SEED, gamma_mode: str = "ones",
                  n_threads: Optional[int] = None, with_layers: bool = True) -> StageWeights:
    """The weights a stage over blocks [begin, end) owns (embedding if begin == 0; final
    norm and readout if end == n_layers).  Nothing outside that range is generated."""
    if not (0 <= begin < end <= cfg.n_layers):
        raise ValueError("bad layer range")
    sw = StageWeights(cfg, begin, end, [])
    if with_layers:
        sw.layers = [layer_weights(cfg, l, seed, gamma_mode, n_threads) for l in range(begin, end)]
    if begin == 0:
        sw.embed = Q8(*q8(tensor_key(seed, cfg.cfg_id, 0, T_EMBED), cfg.vocab, cfg.hidden, n_threads=n_threads))
    if end == cfg.n_layers:
        sw.final_norm = gamma(seed, cfg, 0, T_FINAL_NORM, gamma_mode)
        sw.lm_head = Q8(*q8(tensor_key(seed, cfg.cfg_id, 0, T_HEAD), cfg.vocab, cfg.hidden, n_threads=n_threads))
    return sw


def prompt_tokens(cfg: ModelCfg, seq: int, n: int, seed: int = DEFAULT_SEED) -> np.ndarray:
    """Seeded prompt ids, uniform in [0, vocab)."""
    return uniform_int(tensor_key(seed, cfg.cfg_id, 0, T_PROMPT, seq), 0, n, cfg.vocab)


def ragged_lengths(n_seqs: int, lo: int, hi: int, seed: int = DEFAULT_SEED, cfg_id: int = 4) -> np.ndarray:
    """Per-sequence context lengths uniform in [lo, hi]."""
    return lo + uniform_int(tensor_key(seed, cfg_id, 0, T_KVFILL, 1 << 20), 0, n_seqs, hi - lo + 1)


def reduced(cfg: ModelCfg, n_layers: int, **kw) -> ModelCfg:
    """Same shapes with fewer blocks (parity runs of the large models)."""
    return replace(cfg, n_layers=n_layers, **kw)
