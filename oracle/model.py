"""Float64 CPU oracle of the quantised decoder stage.  TEST INFRASTRUCTURE ONLY.

Pages cited (by title and section):
  [RFC]   "RFC: pipeline placement across multiple GPUs for models larger than one device"
  [TS]    "Multi-node layer splitting and tensor parallelism"
  [BOOK]  "41. Many GPUs: tensor, pipeline, expert and data parallelism"

Arithmetic is float64 inside every op.  Values are rounded to float32 wherever the
stage materialises a float32 tensor (x, h, q, k, v, o, the SwiGLU product a,
logits) and K/V are rounded to float16 when stored.  Where the pages leave a step
open the plainest reading is taken; each such reading is marked "Reading:".

Parity status: every function here is pinned by a test in tests/test_oracle_*.py
against a closed form, an invariant, a special case or a brute-force loop, and
Stage.forward as a whole by weights that reduce a block to a closed form
(tests/test_oracle_block_reductions.py: identity blocks, uniform attention, an
identity SwiGLU in float32 and bf16, identical experts, an identity readout).  The
end-to-end logits and greedy tokens of a seeded model are pinned only through
those parts and through the staged-vs-unstaged invariant (no page prints values
for a seeded model).
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

F64 = np.float64

__all__ = [
    "f32", "f16", "bf16", "dequant", "rmsnorm", "rope_rotate", "rope_inv_freq", "attention_partial",
    "merge_partials", "attention", "silu", "swiglu", "moe_route", "moe_ffn", "shared_expert", "Stage", "Pipeline",
    "greedy", "matvec",
]


# ----------------------------------------------------------------------------- rounding

def f32(x) -> np.ndarray:
    """Round to float32 (RNE) and continue in float64."""
    return np.asarray(x, dtype=F64).astype(np.float32).astype(F64)


def f16(x) -> np.ndarray:
    """Round to float16 (RNE), returned as float16."""
    return np.asarray(x, dtype=F64).astype(np.float16)


def bf16(x) -> np.ndarray:
    """Round to float32, then to bfloat16 (RNE on the upper 16 bits); returned in float64.

    This is the rounding of a float32 value to a bf16 GEMM operand."""
    a = np.ascontiguousarray(np.asarray(x, dtype=F64).astype(np.float32))
    u = a.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).astype(F64)


# ----------------------------------------------------------------------------- weights

def dequant(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """W = scale_b * q for every block b of 32 consecutive weights along the input axis.

    q: int8 [rows, cols]; s: float16 bit patterns (uint16) [rows, ceil(cols/32)].  When
    cols is not a multiple of 32 the last block of each row holds cols % 32 weights.
    Reading: the pages name only an 8-bit format ("Q8", [RFC] "Larger-than-single-card
    proof"); the block-32 int8 + fp16-scale layout is the one this stage stores.  The
    product of an 11-bit fp16 significand and a 7-bit integer is exact in float32 and
    float64 alike."""
    rows, cols = q.shape
    nb = (cols + 31) // 32
    scale = np.asarray(s, dtype=np.uint16).view(np.float16).astype(F64)
    assert scale.shape == (rows, nb)
    out = np.empty((rows, cols), dtype=F64)
    for b in range(nb):
        lo, hi = 32 * b, min(cols, 32 * b + 32)
        out[:, lo:hi] = q[:, lo:hi].astype(F64) * scale[:, b:b + 1]
    return out


def matvec(w: np.ndarray, x: np.ndarray) -> np.ndarray:
    """x @ w.T for x [n, cols] -- the plain linear map (a library matmul as one step)."""
    return np.asarray(x, dtype=F64) @ np.asarray(w, dtype=F64).T


# ----------------------------------------------------------------------------- layer ops

def rmsnorm(x: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """h = x / sqrt(mean(x^2) + eps) * gamma over the last axis.

    [BOOK] "Pipeline parallelism": each block applies add_norm before attention and
    before the MLP, and the final norm after the last block.  Reading: add_norm adds
    the pending delta (if any) to the residual x and returns (norm(x), x); norm is
    RMSNorm with eps = 1e-5 unless the model says otherwise."""
    x = np.asarray(x, dtype=F64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(gamma, dtype=F64)


def rope_inv_freq(head_dim: int, theta: float) -> np.ndarray:
    """theta^(-2i/D) for i in [0, D/2)."""
    return np.asarray(theta, dtype=F64) ** (-2.0 * np.arange(head_dim // 2, dtype=F64) / head_dim)


def rope_rotate(v: np.ndarray, positions: np.ndarray, theta: float) -> np.ndarray:
    """Rotary position embedding, rotate-half pairing: element i pairs with i + D/2.

    v: [n, heads, D]; positions: [n].  [BOOK] "Pipeline parallelism" computes
    rope(positions) once per forward and applies it inside attention.  Reading: the
    common rotate-half form with angle pos * theta^(-2i/D), theta = 10000."""
    v = np.asarray(v, dtype=F64)
    d = v.shape[-1]
    half = d // 2
    ang = np.asarray(positions, dtype=F64)[:, None] * rope_inv_freq(d, theta)[None, :]
    cos, sin = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    x1, x2 = v[..., :half], v[..., half:]
    return np.concatenate([x1 * cos - x2 * sin, x2 * cos + x1 * sin], axis=-1)


def attention_partial(q: np.ndarray, k: np.ndarray, v: np.ndarray, q_pos: np.ndarray,
                      k_pos: np.ndarray, scale: float) -> Tuple[np.ndarray, np.ndarray]:
    """Causal attention of one head: q [Tq, D] over k, v [Tk, D] -> (out [Tq, D], lse [Tq]).

    [BOOK] "Ring attention for very long contexts", attention_partial: scores are
    q.k * scale, masked where the key position exceeds the query position; a row that
    sees no key gets lse = -inf and an all-zero output."""
    q, k, v = (np.asarray(a, dtype=F64) for a in (q, k, v))
    s = (q @ k.T) * scale
    s = np.where(np.asarray(k_pos)[None, :] > np.asarray(q_pos)[:, None], -np.inf, s)
    out = np.zeros((q.shape[0], v.shape[1]), dtype=F64)
    lse = np.full(q.shape[0], -np.inf, dtype=F64)
    for i in range(q.shape[0]):
        row = s[i]
        if np.all(np.isneginf(row)):
            continue
        m = np.max(row)
        e = np.exp(row - m)
        tot = np.sum(e)
        lse[i] = m + np.log(tot)
        out[i] = (e / tot) @ v
    return out, lse


def merge_partials(outs: Sequence[np.ndarray], lses: Sequence[np.ndarray]) -> Tuple[np.ndarray, np.ndarray]:
    """Combine partial attentions over disjoint key sets.

    [BOOK] "Ring attention for very long contexts": each partial carries its
    log-sum-exp; o = sum_s exp(l_s - l) o_s with l = log sum_s exp(l_s).  Partials with
    l_s = -inf contribute nothing."""
    lses = [np.asarray(l, dtype=F64) for l in lses]
    outs = [np.asarray(o, dtype=F64) for o in outs]
    top = np.max(np.stack(lses), axis=0)
    top = np.where(np.isneginf(top), 0.0, top)
    w = [np.exp(l - top) for l in lses]
    total = np.sum(np.stack(w), axis=0)
    merged = sum(o * wi[..., None] for o, wi in zip(outs, w)) / np.where(total > 0, total, 1.0)[..., None]
    lse = np.where(total > 0, top + np.log(np.where(total > 0, total, 1.0)), -np.inf)
    return merged, lse


def attention(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray, seq_ids: np.ndarray,
              positions: np.ndarray, n_kv_heads: int) -> np.ndarray:
    """Grouped-query attention of n tokens over the stage's fp16 cache.

    q: [n, Hq, D] (float64); k_cache, v_cache: [max_seqs, Hkv, max_len, D] float16.
    Token t of sequence seq_ids[t] at position positions[t] attends to cached positions
    0..positions[t] of its own sequence (causal).  Query head j reads KV head
    floor(j / (Hq / Hkv)): [BOOK] "Tensor parallelism" (32 query heads share 8 KV heads,
    each KV head serving a contiguous group).  Scale 1/sqrt(D) as in attention_partial.
    Reading: the current token's k/v are read back from the fp16 cache like every other
    cached row."""
    n, hq, d = q.shape
    group = hq // n_kv_heads
    out = np.zeros((n, hq, d), dtype=F64)
    scale = 1.0 / np.sqrt(d)
    for t in range(n):
        s_id, p = int(seq_ids[t]), int(positions[t])
        for j in range(hq):
            g = j // group
            keys = k_cache[s_id, g, : p + 1].astype(F64)
            vals = v_cache[s_id, g, : p + 1].astype(F64)
            o, _ = attention_partial(q[t, j][None, :], keys, vals, np.array([p]), np.arange(p + 1), scale)
            out[t, j] = o[0]
    return out


def silu(z: np.ndarray) -> np.ndarray:
    """z * sigmoid(z) = z / (1 + e^-z)."""
    z = np.asarray(z, dtype=F64)
    return z / (1.0 + np.exp(-z))


def swiglu(h: np.ndarray, w_gate: np.ndarray, w_up: np.ndarray, w_down: np.ndarray,
           gemm_round=None) -> np.ndarray:
    """down(silu(gate(h)) * up(h)) -- [BOOK] "MoE layers under tensor parallelism"
    (local_experts and the shared expert apply F.linear(F.silu(gate) * up, down)).

    The intermediate a = silu(g) * u is materialised in float32.  ``gemm_round`` (e.g.
    bf16) rounds the GEMM operands h and a when the stage runs its GEMMs in that type."""
    rnd = gemm_round or (lambda t: t)
    hh = rnd(h)
    g = matvec(w_gate, hh)
    u = matvec(w_up, hh)
    a = f32(silu(g) * u)
    return matvec(w_down, rnd(a))


def moe_route(logits: np.ndarray, top_k: int) -> Tuple[np.ndarray, np.ndarray]:
    """Top-k routing of one token: p = softmax(router logits); the k largest p in
    descending order (ties to the lower expert id); weights p[idx] / sum p[idx].

    [BOOK] "MoE layers under tensor parallelism": the gate returns (weights, experts)
    per token.  Reading: softmax over all experts, then top-k, then renormalise over the
    selected k (A3B-style); a shared expert, when the model has one, is added outside the
    routed mix (shared_expert)."""
    z = np.asarray(logits, dtype=F64)
    p = np.exp(z - np.max(z))
    p = p / np.sum(p)
    order = np.argsort(-p, kind="stable")
    idx = order[:top_k]
    w = p[idx] / np.sum(p[idx])
    return idx, w


def shared_expert(h: np.ndarray, score: np.ndarray, w_gate: np.ndarray, w_up: np.ndarray, w_down: np.ndarray,
                  gemm_round=None) -> np.ndarray:
    """The shared expert of a MoE layer for tokens h [n, H]: sigmoid(score . h_t) *
    SwiGLU_shared(h_t).  [BOOK] "MoE layers under tensor parallelism" and "Expert parallelism
    with all-to-all": the layer output adds sigmoid(shared_gate(x)) times shared(x) to the
    routed experts' sum.  ``score`` is the scalar gate's weights [1, H]; its logit is
    materialised in float32 like the router logits.  Returns [n, H] float64."""
    s = f32(matvec(score, h))[:, 0].astype(F64)
    with np.errstate(over="ignore"):  # exp(-s) = inf for s << 0 gives the exact limit 0
        sig = 1.0 / (1.0 + np.exp(-s))
    return sig[:, None] * swiglu(h, w_gate, w_up, w_down, gemm_round)


def moe_ffn(h: np.ndarray, router: np.ndarray, e_gate: Sequence[np.ndarray], e_up: Sequence[np.ndarray],
            e_down: Sequence[np.ndarray], top_k: int, gemm_round=None) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Routed-expert FFN for tokens h [n, H]: out_t = sum_j w_j * SwiGLU_{e_j}(h_t), summed in
    slot order.  [BOOK] "MoE layers under tensor parallelism", local_experts: each used
    expert runs SwiGLU on its tokens and the result is added with the router weight.

    ``e_*`` are callables or arrays indexed by expert id (dequantised on demand).
    Returns (out [n, H] float64, ids [n, k], weights [n, k])."""
    rnd = gemm_round or (lambda t: t)
    logits = f32(matvec(router, h))
    n = h.shape[0]
    out = np.zeros((n, h.shape[1]), dtype=F64)
    ids = np.zeros((n, top_k), dtype=np.int64)
    ws = np.zeros((n, top_k), dtype=F64)
    for t in range(n):
        idx, w = moe_route(logits[t], top_k)
        ids[t], ws[t] = idx, w
        acc = np.zeros(h.shape[1], dtype=F64)
        for j in range(top_k):
            e = int(idx[j])
            g, u, dn = (m(e) if callable(m) else m[e] for m in (e_gate, e_up, e_down))
            acc = acc + w[j] * swiglu(h[t][None, :], g, u, dn, rnd)[0]
        out[t] = acc
    return out, ids, ws


def greedy(logits: np.ndarray) -> np.ndarray:
    """Greedy token per row: argmax, lowest index on ties (Reading: the pages do not say)."""
    return np.argmax(np.asarray(logits), axis=-1).astype(np.int32)


# ----------------------------------------------------------------------------- the stage

class Stage:
    """One pipeline stage: decoder blocks [begin, end) of ``cfg`` with their weights and KV.

    [RFC] "What I found": a stage owns its resident weights and its model state (KV);
    only the hidden activation crosses the boundary; the first stage embeds, the last
    applies norm and readout.  [TS] "Supported stage executors": the dense pipeline
    transfers F32 hidden activations, each node loads only its layer weights and KV,
    the first stage embeds and the last computes logits.  [BOOK] "Pipeline parallelism":
    the per-block loop and the single residual tensor that crosses each boundary.

    ``weights`` has the fields of synth.StageWeights (embed/lm_head/final_norm present
    only if owned; layers[l - begin] for each owned block).  Matrices are (q, s) pairs
    exposed as objects with ``.q`` and ``.s``.
    """

    def __init__(self, cfg, begin: int, end: int, weights, max_seqs: int = 1, max_len: int = 256,
                 cache_dequant: bool = True):
        if not (0 <= begin < end <= cfg.n_layers):
            raise ValueError("bad layer range")
        self.cfg, self.begin, self.end = cfg, begin, end
        self.first, self.last = begin == 0, end == cfg.n_layers
        self.w = weights
        self.max_seqs, self.max_len = max_seqs, max_len
        shape = (end - begin, max_seqs, cfg.n_kv_heads, max_len, cfg.head_dim)
        self.k_cache = np.zeros(shape, dtype=np.float16)
        self.v_cache = np.zeros(shape, dtype=np.float16)
        self.features: Optional[np.ndarray] = None
        self._deq_cache: Dict[int, np.ndarray] = {}
        self.cache_dequant = cache_dequant

    # dequantised matrices (cached by identity; the oracle is allowed to be slow, not wasteful)
    def _deq(self, m) -> np.ndarray:
        key = id(m)
        if key not in self._deq_cache:
            self._deq_cache[key] = dequant(m.q, m.s)
        return self._deq_cache[key]

    def forget_dequant(self) -> None:
        self._deq_cache.clear()

    def forward(self, seq_ids, positions, tokens=None, hidden_in=None, gemm: str = "f32",
                cache_dequant: Optional[bool] = None) -> np.ndarray:
        """Run n tokens through this stage's blocks; returns the float32 hidden [n, H].

        The first stage embeds ``tokens``; any other stage takes ``hidden_in`` (float32
        [n, H]) unchanged -- it is a residual with nothing pending to add ([BOOK]
        "Pipeline parallelism").  The last stage returns the final features
        f = rmsnorm(x) * gamma_f and keeps them for ``logits``.

        gemm = "f32" keeps GEMM operands in float32; "bf16" rounds every GEMM operand
        (activations and dequantised weights) to bfloat16, accumulating in float64; the
        residual, norms and handoff stay float32 (the prefill numerics)."""
        c = self.cfg
        seq_ids = np.asarray(seq_ids, dtype=np.int64)
        positions = np.asarray(positions, dtype=np.int64)
        n = len(positions)
        rnd = bf16 if gemm == "bf16" else (lambda t: t)
        if cache_dequant is None:
            cache_dequant = self.cache_dequant
        deq = (lambda m: rnd(self._deq(m))) if cache_dequant else (lambda m: rnd(dequant(m.q, m.s)))
        if self.first:
            if tokens is None or hidden_in is not None:
                raise ValueError("the first stage embeds tokens")
            x = dequant(self.w.embed.q[np.asarray(tokens)], self.w.embed.s[np.asarray(tokens)])
        else:
            if hidden_in is None or tokens is not None:
                raise ValueError("a later stage takes the hidden activation")
            x = np.asarray(hidden_in, dtype=np.float32).astype(F64)
        x = f32(x)
        assert x.shape == (n, c.hidden)
        for li in range(self.end - self.begin):
            lw = self.w.layers[li]
            # attention sub-block: h = norm(x); q,k,v; rope; append K/V; attend; x += W_o o
            h = f32(rmsnorm(x, lw.attn_norm, c.rms_eps))
            hh = rnd(h)
            q = f32(matvec(deq(lw.wq), hh)).reshape(n, c.n_q_heads, c.head_dim)
            k = f32(matvec(deq(lw.wk), hh)).reshape(n, c.n_kv_heads, c.head_dim)
            v = f32(matvec(deq(lw.wv), hh)).reshape(n, c.n_kv_heads, c.head_dim)
            q = f32(rope_rotate(q, positions, c.rope_theta))
            k = rope_rotate(k, positions, c.rope_theta)
            for t in range(n):
                self.k_cache[li, seq_ids[t], :, positions[t]] = f16(k[t])
                self.v_cache[li, seq_ids[t], :, positions[t]] = f16(v[t])
            o = f32(attention(q, self.k_cache[li], self.v_cache[li], seq_ids, positions, c.n_kv_heads))
            x = f32(x + matvec(deq(lw.wo), rnd(o.reshape(n, c.q_dim))))
            # FFN sub-block: h = norm(x); x += FFN(h)
            h = f32(rmsnorm(x, lw.ffn_norm, c.rms_eps))
            if c.is_moe:
                ffn, _, _ = moe_ffn(h, deq(lw.router) if gemm != "bf16" else self._deq(lw.router), lambda e: deq(lw.e_gate[e]),
                                    lambda e: deq(lw.e_up[e]), lambda e: deq(lw.e_down[e]), c.top_k, rnd)
                if getattr(c, "shared_ffn", 0):
                    ffn = ffn + shared_expert(h, self._deq(lw.shared_score), deq(lw.shared_gate), deq(lw.shared_up),
                                              deq(lw.shared_down), rnd)
            else:
                ffn = swiglu(h, deq(lw.w_gate), deq(lw.w_up), deq(lw.w_down), rnd)
            x = f32(x + ffn)
        if self.last:
            f = f32(rmsnorm(x, self.w.final_norm, c.rms_eps))
            self.features = f
            return f.astype(np.float32)
        return x.astype(np.float32)

    def route(self, li: int, h: np.ndarray):
        """Router decision of owned block ``li`` for normed inputs h (diagnostics for tests)."""
        lw = self.w.layers[li]
        logits = f32(matvec(self._deq(lw.router), h))
        return [moe_route(l, self.cfg.top_k) for l in logits], logits

    def logits(self, rows: Optional[Sequence[int]] = None) -> np.ndarray:
        """Readout of the last stage: logits = W_head f for the requested rows of the last
        forward ([RFC] "What I found": the last stage does norm / readout)."""
        if not self.last:
            raise ValueError("only the last stage owns the readout")
        f = self.features if rows is None else self.features[np.asarray(rows)]
        return f32(matvec(self._deq(self.w.lm_head), f)).astype(np.float32)


class Pipeline:
    """Stages chained in order, one hidden activation handed across each boundary.

    Counts the handoff traffic per boundary the way the book's communicator counts
    sends ([BOOK] "The communicator" and "Measured": calls and bytes)."""

    def __init__(self, stages: List[Stage]):
        for a, b in zip(stages, stages[1:]):
            if a.end != b.begin:
                raise ValueError("stages must be contiguous")
        if stages[0].begin != 0 or not stages[-1].last:
            raise ValueError("stages must cover the model")
        self.stages = stages
        self.handoff_calls = [0] * (len(stages) - 1)
        self.handoff_bytes = [0] * (len(stages) - 1)

    def forward(self, seq_ids, positions, tokens, gemm: str = "f32") -> np.ndarray:
        h = None
        for i, st in enumerate(self.stages):
            if i == 0:
                h = st.forward(seq_ids, positions, tokens=tokens, gemm=gemm)
            else:
                h = st.forward(seq_ids, positions, hidden_in=h, gemm=gemm)
            if i + 1 < len(self.stages):
                assert h.dtype == np.float32
                self.handoff_calls[i] += 1
                self.handoff_bytes[i] += h.nbytes
        return h

    def logits(self, rows=None) -> np.ndarray:
        return self.stages[-1].logits(rows)

    def generate(self, prompts: List[np.ndarray], n_new: int, prefill_gemm: str = "f32",
                 decode_gemm: str = "f32") -> Tuple[np.ndarray, List[np.ndarray]]:
        """Greedy generation for several sequences: one prefill step over all prompt tokens
        (logits of each sequence's last token), then n_new - 1 decode steps feeding the
        greedy token back at the next position.  Returns (tokens [seqs, n_new], logits per step)."""
        seqs = len(prompts)
        seq_ids = np.concatenate([np.full(len(p), s) for s, p in enumerate(prompts)])
        positions = np.concatenate([np.arange(len(p)) for p in prompts])
        toks = np.concatenate(prompts)
        self.forward(seq_ids, positions, toks, gemm=prefill_gemm)
        last_rows = np.cumsum([len(p) for p in prompts]) - 1
        lg = self.logits(last_rows)
        out = [greedy(lg)]
        all_logits = [lg]
        lens = np.array([len(p) for p in prompts])
        for _ in range(n_new - 1):
            self.forward(np.arange(seqs), lens.copy(), out[-1], gemm=decode_gemm)
            lens += 1
            lg = self.logits()
            all_logits.append(lg)
            out.append(greedy(lg))
        return np.stack(out, axis=1), all_logits
