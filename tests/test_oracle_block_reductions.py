"""Whole-block pins of the oracle: weights that reduce a decoder block to a closed form.

The per-function pins check each step alone; these check how Stage.forward composes them
([BOOK] "Pipeline parallelism": the per-block loop, one residual tensor through the stage;
[RFC] "What I found": a stage keeps its own KV state between calls).
  - W_o = 0 and W_down = 0: both sub-blocks add exactly zero, so the stage returns its input
    bit for bit (a dropped or doubled residual fails), while the KV cache is still written.
  - W_q = 0: every score is 0, so softmax weighs the visible rows equally and attention is the
    plain mean of the cached V rows of the token's own sequence at positions up to its own
    (causal window, per-sequence cache, rows kept from an earlier call).  With W_v picking the
    first Hkv*D coordinates of the normed input and W_o = I, a block becomes
        x <- x + [mean_{j <= p} fp16(h_j)[kv(g)] for each q head g],  kv(g) = g // (Hq / Hkv),
    so a wrong head-to-group map, an off-by-one window or another sequence's rows show up.
    The result must not depend on W_k at all.
  - a last stage with such an identity block and the readout W_head = I: the logits of a row
    are its final features rmsnorm(x) * gamma_f followed by zeros.
  - W_o = 0 with identity gate, twice-identity up and identity down: a block adds
    silu(h) * 2h with h the FFN-normed residual, element by element.
  - a MoE stage whose experts are all one SwiGLU equals the dense stage with it, whatever the
    router selects.
  - the identity FFN with the GEMMs in bf16: exactly the bf16 roundings of h and of the SwiGLU
    output, nothing else.
"""
import numpy as np

import oracle
import synth

CFG = synth.CONFIGS[0]  # H 256, 4 q heads, 2 KV heads of 64, FFN 688
ONE = np.uint16(0x3C00)  # fp16 1.0


def zero_q8(rows, cols):
    return synth.Q8(np.zeros((rows, cols), np.int8), np.zeros((rows, (cols + 31) // 32), np.uint16))


def eye_q8(rows, cols):
    q = np.zeros((rows, cols), np.int8)
    n = min(rows, cols)
    q[np.arange(n), np.arange(n)] = 1
    return synth.Q8(q, np.full((rows, (cols + 31) // 32), ONE, np.uint16))


def stage(layers, max_seqs=2):
    sw = synth.StageWeights(CFG, 1, 3, layers)
    return oracle.Stage(CFG, 1, 3, sw, max_seqs=max_seqs, max_len=32)


def hidden(n, seed):
    return np.random.default_rng(seed).standard_normal((n, CFG.hidden)).astype(np.float32)


def test_zero_output_projections_make_the_stage_the_identity():
    layers = []
    for l in (1, 2):
        lw = synth.layer_weights(CFG, l, gamma_mode="seeded")
        lw.wo = zero_q8(CFG.hidden, CFG.q_dim)
        lw.w_down = zero_q8(CFG.hidden, CFG.ffn)
        layers.append(lw)
    st = stage(layers)
    x = hidden(7, 1)
    y = st.forward(np.zeros(7, int), np.arange(7), hidden_in=x)
    assert y.dtype == np.float32 and np.array_equal(y.view(np.uint32), x.view(np.uint32))
    assert np.abs(st.k_cache[:, 0, :, :7].astype(np.float64)).min(axis=-1).max() > 0  # rows written
    assert not st.k_cache[:, 0, :, 7:].any() and not st.k_cache[:, 1].any()


def uniform_attention_layers(wk_seed):
    layers = []
    for l in (1, 2):
        lw = synth.layer_weights(CFG, l, gamma_mode="seeded")
        lw.wq = zero_q8(CFG.q_dim, CFG.hidden)
        lw.wk = synth.layer_weights(CFG, l, seed=wk_seed).wk
        lw.wv = eye_q8(CFG.kv_dim, CFG.hidden)
        lw.wo = eye_q8(CFG.hidden, CFG.q_dim)
        lw.w_down = zero_q8(CFG.hidden, CFG.ffn)
        layers.append(lw)
    return layers


def expected(layers, calls):
    """The closed form above, call after call, in float64 with the stage's float32/fp16
    roundings at the points where it stores a tensor."""
    G, D = CFG.n_q_heads // CFG.n_kv_heads, CFG.head_dim
    cache = {}  # (block, seq) -> {position: fp16 V row}
    outs = []
    for seq_ids, positions, x in calls:
        x = x.astype(np.float64)
        for b, lw in enumerate(layers):
            g = lw.attn_norm.astype(np.float64)
            h = (x / np.sqrt(np.mean(x * x, axis=1, keepdims=True) + CFG.rms_eps) * g).astype(np.float32)
            v = h[:, :CFG.kv_dim].astype(np.float16)
            for t, (s, p) in enumerate(zip(seq_ids, positions)):
                cache.setdefault((b, s), {})[p] = v[t].astype(np.float64)
            o = np.empty_like(x)
            for t, (s, p) in enumerate(zip(seq_ids, positions)):
                rows = np.stack([r for q, r in cache[(b, s)].items() if q <= p])
                mean = rows.mean(axis=0).reshape(CFG.n_kv_heads, D)
                o[t] = np.concatenate([mean[hq // G] for hq in range(CFG.n_q_heads)])
            x = (x + o.astype(np.float32)).astype(np.float32).astype(np.float64)
        outs.append(x.astype(np.float32))
    return outs


def test_zero_queries_give_the_causal_mean_of_the_sequence_values():
    # prefill of two ragged sequences interleaved in one call, then one decode token each
    seq0 = [0, 1, 0, 0, 1, 0, 1, 0]
    pos0 = [0, 0, 1, 2, 1, 3, 2, 4]
    calls = [(seq0, pos0, hidden(8, 2)), ([1, 0], [3, 5], hidden(2, 3))]
    st = stage(uniform_attention_layers(wk_seed=11))
    got = [st.forward(s, p, hidden_in=x) for s, p, x in calls]
    want = expected(uniform_attention_layers(wk_seed=11), calls)
    for g, w, (_, _, x) in zip(got, want, calls):
        scale = np.abs(w - x).max()
        assert scale > 0.05  # attention added something
        assert np.abs(g - w).max() <= 2e-3 * scale + 1e-6
    # the keys cannot matter when every query is zero: bit for bit with other W_k
    st2 = stage(uniform_attention_layers(wk_seed=12))
    got2 = [st2.forward(s, p, hidden_in=x) for s, p, x in calls]
    assert not np.array_equal(st.k_cache, st2.k_cache)
    for a, b in zip(got, got2):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_the_closed_form_separates_the_plausible_mistakes():
    """The expected values above differ by far more than the tolerance from what a block
    with the q-head -> KV-head map g % Hkv, or with the window one row short, would give."""
    seq0 = [0, 0, 0, 0]
    pos0 = [0, 1, 2, 3]
    x = hidden(4, 4)
    st = stage(uniform_attention_layers(wk_seed=11), max_seqs=1)
    got = st.forward(seq0, pos0, hidden_in=x)
    lw = uniform_attention_layers(wk_seed=11)[0]
    G, D = CFG.n_q_heads // CFG.n_kv_heads, CFG.head_dim
    x64 = x.astype(np.float64)
    h = (x64 / np.sqrt(np.mean(x64 * x64, axis=1, keepdims=True) + CFG.rms_eps) * lw.attn_norm).astype(np.float32)
    v = h[:, :CFG.kv_dim].astype(np.float16).astype(np.float64).reshape(4, CFG.n_kv_heads, D)
    right = np.stack([np.concatenate([v[:t + 1].mean(0)[hq // G] for hq in range(CFG.n_q_heads)]) for t in range(4)])
    wrong_map = np.stack([np.concatenate([v[:t + 1].mean(0)[hq % CFG.n_kv_heads] for hq in range(CFG.n_q_heads)])
                          for t in range(4)])
    short = np.stack([np.concatenate([v[:max(t, 1)].mean(0)[hq // G] for hq in range(CFG.n_q_heads)])
                      for t in range(4)])
    assert np.abs(right - wrong_map).max() > 0.1 and np.abs(right[1:] - short[1:]).max() > 0.1
    # one block's attention output is the first block's x increment: check it in isolation
    st1 = oracle.Stage(CFG, 1, 2, synth.StageWeights(CFG, 1, 2, [lw]), max_seqs=1, max_len=32)
    y1 = st1.forward(seq0, pos0, hidden_in=x).astype(np.float64)
    assert np.abs((y1 - x64) - right).max() <= 2e-3 * np.abs(right).max()
    assert got.shape == x.shape


def test_last_stage_with_identity_blocks_and_readout_gives_the_normed_input_as_logits():
    """A last stage whose block adds zero and whose readout is I (V x H, V > H): the final
    features are rmsnorm(x) * gamma_f, the logits of a row are those features followed by
    V - H zeros, and greedy picks the largest feature ([RFC] "What I found": the last stage
    applies the norm and the readout)."""
    lw = synth.layer_weights(CFG, 3, gamma_mode="seeded")
    lw.wo = zero_q8(CFG.hidden, CFG.q_dim)
    lw.w_down = zero_q8(CFG.hidden, CFG.ffn)
    sw = synth.StageWeights(CFG, 3, 4, [lw], final_norm=synth.gamma(synth.DEFAULT_SEED, CFG, 0, 99, "seeded"),
                            lm_head=eye_q8(CFG.vocab, CFG.hidden))
    st = oracle.Stage(CFG, 3, 4, sw, max_seqs=1, max_len=32)
    x = hidden(5, 5)
    f = st.forward(np.zeros(5, int), np.arange(5), hidden_in=x)
    x64 = x.astype(np.float64)
    want = x64 / np.sqrt(np.mean(x64 * x64, axis=1, keepdims=True) + CFG.rms_eps) * sw.final_norm
    assert np.abs(f - want).max() <= 1e-6 * np.abs(want).max()
    rows = [4, 1]
    lg = st.logits(rows)
    assert lg.shape == (2, CFG.vocab) and not lg[:, CFG.hidden:].any()
    assert np.array_equal(lg[:, :CFG.hidden], f[rows])
    assert list(oracle.greedy(lg)) == [int(np.argmax(f[r])) for r in rows]


def test_moe_stage_with_identical_experts_equals_the_dense_stage():
    """Every expert holding the same gate/up/down: whatever the router picks, the renormalised
    top-k weights sum to 1 over copies of one SwiGLU, so a MoE stage must return what the dense
    stage with those matrices returns ("41. Many GPUs: tensor, pipeline, expert and data
    parallelism", the MoE layer: top-k experts mixed with renormalised router weights).  The
    router is seeded and random, so the selected experts differ from token to token."""
    shape = dict(hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64, vocab=512)
    moe = synth.reduced(synth.CONFIGS[2], 4, n_experts=8, top_k=2, expert_ffn=64, **shape)
    dense = synth.reduced(synth.CONFIGS[0], 4, ffn=64, **shape)
    layers_m, layers_d = [], []
    for l in (1, 2):
        lm = synth.layer_weights(moe, l, gamma_mode="seeded")
        ld = synth.layer_weights(dense, l, gamma_mode="seeded")
        for name in ("attn_norm", "ffn_norm", "wq", "wk", "wv", "wo"):
            setattr(ld, name, getattr(lm, name))
        lm.e_gate = [lm.e_gate[0]] * moe.n_experts
        lm.e_up = [lm.e_up[0]] * moe.n_experts
        lm.e_down = [lm.e_down[0]] * moe.n_experts
        ld.w_gate, ld.w_up, ld.w_down = lm.e_gate[0], lm.e_up[0], lm.e_down[0]
        layers_m.append(lm)
        layers_d.append(ld)
    x = hidden(6, 7)
    sm = oracle.Stage(moe, 1, 3, synth.StageWeights(moe, 1, 3, layers_m), max_seqs=1, max_len=16)
    sd = oracle.Stage(dense, 1, 3, synth.StageWeights(dense, 1, 3, layers_d), max_seqs=1, max_len=16)
    ym = sm.forward(np.zeros(6, int), np.arange(6), hidden_in=x).astype(np.float64)
    yd = sd.forward(np.zeros(6, int), np.arange(6), hidden_in=x).astype(np.float64)
    assert np.abs(ym - yd).max() <= 1e-6 * np.abs(yd).max()
    # the router does select different experts for different inputs
    picks = {tuple(sorted(r[0])) for r in sm.route(0, oracle.f32(x))[0]}
    assert len(picks) > 1


def scaled_eye_q8(rows, cols, k):
    m = eye_q8(rows, cols)
    m.q[np.arange(min(rows, cols)), np.arange(min(rows, cols))] = k
    return m


def test_zero_attention_and_identity_ffn_give_the_swiglu_of_the_normed_input():
    """W_o = 0 removes the attention half; W_gate = I, W_up = 2 I, W_down = I (exact int8 rows,
    F > H so the extra gate/up rows are zero and silu(0) * 0 = 0) reduce the FFN half to
        x <- x + silu(h) * 2 h,   h = x / sqrt(mean(x^2) + eps) * gamma_2,
    element by element, block after block ("41. Many GPUs: tensor, pipeline, expert and data
    parallelism", section "Pipeline parallelism": add_norm, then the MLP on the normed
    residual).  Gate and up swapped would give silu(2h) * h; the attention norm's gain in
    place of gamma_2, or a lost residual, fail too."""
    layers = []
    for l in (1, 2):
        lw = synth.layer_weights(CFG, l, gamma_mode="seeded")
        lw.wo = zero_q8(CFG.hidden, CFG.q_dim)
        lw.w_gate = eye_q8(CFG.ffn, CFG.hidden)
        lw.w_up = scaled_eye_q8(CFG.ffn, CFG.hidden, 2)
        lw.w_down = eye_q8(CFG.hidden, CFG.ffn)
        layers.append(lw)
    assert CFG.ffn > CFG.hidden
    st = stage(layers)
    x = hidden(5, 8)
    y = st.forward(np.zeros(5, int), np.arange(5), hidden_in=x).astype(np.float64)
    want = x.astype(np.float64)
    for lw in layers:
        h = (want / np.sqrt(np.mean(want * want, axis=1, keepdims=True) + CFG.rms_eps) * lw.ffn_norm)
        h = h.astype(np.float32).astype(np.float64)
        a = (h / (1.0 + np.exp(-h)) * 2.0 * h).astype(np.float32).astype(np.float64)
        want = (want + a).astype(np.float32).astype(np.float64)
    assert np.abs(y - want).max() <= 1e-5 * np.abs(want).max()
    swapped = x.astype(np.float64)
    for lw in layers:
        h = swapped / np.sqrt(np.mean(swapped * swapped, axis=1, keepdims=True) + CFG.rms_eps) * lw.ffn_norm
        swapped = swapped + 2.0 * h / (1.0 + np.exp(-2.0 * h)) * h
    assert np.abs(want - swapped).max() > 100 * 1e-5 * np.abs(want).max()


def bf16_round(v):
    u = np.asarray(v, np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000).astype(np.uint32)
    return r.view(np.float32).astype(np.float64)


def test_bf16_mode_rounds_the_gemm_operands_of_the_identity_ffn():
    """The same reduction with the stage's GEMMs in bf16 (prefill numerics): the GEMM operands
    -- the normed input h and the SwiGLU output a -- are rounded to bf16 (ties to even), the
    weights (0, 1, 2) are exact, and the residual stays float32:
        x <- x + bf16(f32(silu(bf16(h)) * 2 bf16(h)))."""
    layers = []
    for l in (1, 2):
        lw = synth.layer_weights(CFG, l, gamma_mode="seeded")
        lw.wo = zero_q8(CFG.hidden, CFG.q_dim)
        lw.w_gate = eye_q8(CFG.ffn, CFG.hidden)
        lw.w_up = scaled_eye_q8(CFG.ffn, CFG.hidden, 2)
        lw.w_down = eye_q8(CFG.hidden, CFG.ffn)
        layers.append(lw)
    st = stage(layers)
    x = hidden(5, 9)
    y = st.forward(np.zeros(5, int), np.arange(5), hidden_in=x, gemm="bf16").astype(np.float64)
    want = x.astype(np.float64)
    unrounded = x.astype(np.float64)
    for lw in layers:
        h = (want / np.sqrt(np.mean(want * want, axis=1, keepdims=True) + CFG.rms_eps) * lw.ffn_norm)
        hb = bf16_round(h.astype(np.float32))
        a = (hb / (1.0 + np.exp(-hb)) * 2.0 * hb).astype(np.float32)
        want = (want + bf16_round(a)).astype(np.float32).astype(np.float64)
        h2 = unrounded / np.sqrt(np.mean(unrounded * unrounded, axis=1, keepdims=True) + CFG.rms_eps) * lw.ffn_norm
        unrounded = unrounded + h2 / (1.0 + np.exp(-h2)) * 2.0 * h2
    assert np.abs(y - want).max() <= 1e-6 * np.abs(want).max()
    assert np.abs(unrounded - want).max() > 1e-4 * np.abs(want).max()  # the roundings are visible
