"""Pins of the oracle's shared expert ("41. Many GPUs: tensor, pipeline, expert and data
parallelism", sections "MoE layers under tensor parallelism" and "Expert parallelism with
all-to-all": the MoE layer adds sigmoid(shared_gate(x)) * shared(x) to the routed experts).

- the sigmoid at closed-form points: a zero gate halves the shared SwiGLU exactly, a
  saturated gate passes it whole or drops it;
- the wiring inside a block: with every routed expert silenced, a stage with a shared expert
  whose gate is zero adds exactly half of what a dense stage adds whose FFN is that expert
  (same attention, same input), the residual itself being what the stage without the shared
  expert returns."""
import copy

import numpy as np

import oracle
import synth


def rand_mat(rng, rows, cols):
    return rng.normal(0, 0.05, (rows, cols))


def test_zero_gate_halves_the_shared_swiglu():
    rng = np.random.default_rng(900)
    H, F, n = 64, 40, 5
    h = rng.normal(0, 1, (n, H))
    g, u, d = rand_mat(rng, F, H), rand_mat(rng, F, H), rand_mat(rng, H, F)
    got = oracle.shared_expert(h, np.zeros((1, H)), g, u, d)
    assert np.array_equal(got, 0.5 * oracle.swiglu(h, g, u, d))


def test_saturated_gate_passes_or_drops_the_shared_swiglu():
    rng = np.random.default_rng(901)
    H, F = 64, 40
    h = rng.normal(0, 1, (1, H))
    g, u, d = rand_mat(rng, F, H), rand_mat(rng, F, H), rand_mat(rng, H, F)
    big = 2000.0 * h / float((h @ h.T)[0, 0])  # score . h = 2000 (exp(-2000) is 0 in float64)
    assert np.array_equal(oracle.shared_expert(h, big, g, u, d), oracle.swiglu(h, g, u, d))
    assert np.array_equal(oracle.shared_expert(h, -big, g, u, d), np.zeros_like(h))


def test_block_adds_the_gated_shared_expert():
    # two blocks: the stage over block 0 is not the last one, so it returns the residual itself
    moe = synth.reduced(synth.CONFIGS[2], 2, hidden=128, n_q_heads=4, n_kv_heads=2, head_dim=64, vocab=256,
                        n_experts=4, top_k=2, expert_ffn=48, shared_ffn=56)
    plain = synth.reduced(moe, 2, shared_ffn=0)
    dense = synth.reduced(moe, 2, n_experts=0, top_k=0, expert_ffn=0, ffn=56, shared_ffn=0)
    w_moe = synth.stage_weights(moe, 0, 1, gamma_mode="seeded")
    lw = w_moe.layers[0]
    for m in lw.e_down:                     # silence every routed expert
        m.q[:] = 0
    lw.shared_score.q[:] = 0                # gate logit 0: weight 1/2
    w_plain = copy.deepcopy(w_moe)
    w_plain.layers[0].shared_score = w_plain.layers[0].shared_gate = None
    w_plain.layers[0].shared_up = w_plain.layers[0].shared_down = None
    w_dense = copy.deepcopy(w_moe)          # same embedding, norms and attention
    ld = w_dense.layers[0]
    ld.w_gate, ld.w_up, ld.w_down = lw.shared_gate, lw.shared_up, lw.shared_down
    ld.router, ld.e_gate, ld.e_up, ld.e_down = None, [], [], []
    ld.shared_score = ld.shared_gate = ld.shared_up = ld.shared_down = None
    toks = synth.prompt_tokens(moe, 3, 6)
    out = {}
    for name, cfg, w in (("moe", moe, w_moe), ("plain", plain, w_plain), ("dense", dense, w_dense)):
        st = oracle.Stage(cfg, 0, 1, w, max_len=16)
        out[name] = st.forward(np.zeros(6, dtype=np.int64), np.arange(6), tokens=toks).astype(np.float64)
    x1 = out["plain"]                       # the residual after attention (no expert adds anything)
    shared_half = out["moe"] - x1
    dense_full = out["dense"] - x1
    assert np.abs(dense_full).max() > 1e-3  # the shared expert does something
    # equal up to the float32 rounding of the materialised residuals
    tol = 4 * np.finfo(np.float32).eps * np.abs(x1).max()
    assert np.abs(shared_half - 0.5 * dense_full).max() <= tol
