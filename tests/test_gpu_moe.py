"""GPU parity of the routed-expert (MoE) stage: router GEMV, top-k, gathered expert
gate/up with SwiGLU scaled by the routing weight, gathered expert down with the residual.

Tolerances as in test_gpu_stage.py.  Routing decisions are compared only where the
oracle's gap between the k-th and (k+1)-th router logit exceeds 1e-4 (float rounding
cannot flip those); the seeds below are checked to have no closer gap.
"""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

LOGIT_ATOL = 2e-2


def small_moe():
    return synth.reduced(synth.CONFIGS[2], 2, hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64, vocab=512,
                         n_experts=8, top_k=2, expert_ffn=64)


def pipelines(model, bounds, max_len=64, gamma_mode="seeded"):
    from layer_range_stage_gb300.pipeline import StagePipeline
    gp = StagePipeline(model, bounds, lambda l: synth.layer_weights(model, l, gamma_mode=gamma_mode),
                       lambda a, b: synth.stage_weights(model, a, b, gamma_mode=gamma_mode, with_layers=False),
                       max_seqs=1, max_seq_len=max_len, max_tokens=32)
    op = oracle.Pipeline([oracle.Stage(model, a, b, synth.stage_weights(model, a, b, gamma_mode=gamma_mode),
                                       max_len=max_len, cache_dequant=False) for a, b in zip(bounds, bounds[1:])])
    return gp, op


def run_gpu(gp, model, prompt, n_new):
    n = len(prompt)
    lg = torch.empty((1, model.vocab), dtype=torch.float32, device="cuda")
    tok = gp.step(True, np.zeros(n), np.arange(n), prompt, rows=[n - 1], logits_out=lg)
    toks, logits = [int(tok[0])], [lg.cpu().numpy().copy()]
    for t in range(n_new - 1):
        tok = gp.step(False, [0], [n + t], [toks[-1]], rows=[0], logits_out=lg)
        toks.append(int(tok[0]))
        logits.append(lg.cpu().numpy().copy())
    return np.array(toks), logits


def run(gp, op, model, prompt, n_new):
    toks_o, logits_o = op.generate([prompt], n_new)
    toks, logits = run_gpu(gp, model, prompt, n_new)
    return toks, logits, toks_o[0], logits_o


def route_gaps(model, bounds, prompt, gamma_mode="seeded"):
    """Router-logit gaps at the top-k boundary for the prompt tokens (oracle, float32 logits)."""
    gaps = []
    op = oracle.Pipeline([oracle.Stage(model, a, b, synth.stage_weights(model, a, b, gamma_mode=gamma_mode),
                                       max_len=64, cache_dequant=False) for a, b in zip(bounds, bounds[1:])])
    st = op.stages[0]
    n = len(prompt)
    x = oracle.dequant(st.w.embed.q[prompt], st.w.embed.s[prompt])
    lw = st.w.layers[0]
    h = oracle.f32(oracle.rmsnorm(oracle.f32(x), lw.ffn_norm, model.rms_eps))
    _, logits = st.route(0, h)
    for row in logits:
        s = np.sort(row)[::-1]
        gaps.append(s[model.top_k - 1] - s[model.top_k])
    return min(gaps)


def test_small_moe_matches_oracle_and_is_split_invariant(cuda):
    model = small_moe()
    prompt = synth.prompt_tokens(model, 0, 12)
    gp, op = pipelines(model, [0, 1, 2])
    with gp:
        toks, logits, toks_o, logits_o = run(gp, op, model, prompt, 5)
    for a, b in zip(logits, logits_o):
        assert np.abs(a - b).max() <= LOGIT_ATOL
    assert toks.tolist() == toks_o.tolist()
    gm, _ = pipelines(model, [0, 2])
    with gm:
        toks_m, logits_m = run_gpu(gm, model, prompt, 5)
    assert np.array_equal(toks_m, toks)
    for a, b in zip(logits_m, logits):
        assert np.array_equal(a, b)


def test_moe_full_width_two_blocks(cuda):
    """128 experts top-8, expert FFN 768, hidden 2048, 32q/4kv heads, vocab 151936: two
    blocks split 1/1."""
    model = synth.reduced(synth.CONFIGS[2], 2)
    prompt = synth.prompt_tokens(model, 0, 6)
    assert route_gaps(model, [0, 1, 2], prompt, "ones") > 1e-4
    gp, op = pipelines(model, [0, 1, 2], gamma_mode="ones")
    with gp:
        toks, logits, toks_o, logits_o = run(gp, op, model, prompt, 3)
    for a, b in zip(logits, logits_o):
        assert np.abs(a - b).max() <= LOGIT_ATOL
    assert toks.tolist() == toks_o.tolist()


def test_small_moe_with_shared_expert_matches_oracle(cuda):
    """A shared expert beside the routed ones (its scalar gate as the router's last row,
    its SwiGLU and down projection after the routed experts'): logits and greedy tokens
    against the oracle; such stages decode on the GEMV path (no persistent kernel)."""
    from layer_range_stage_gb300 import binding as B
    model = synth.reduced(small_moe(), 2, shared_ffn=96)
    prompt = synth.prompt_tokens(model, 0, 12)
    gp, op = pipelines(model, [0, 1, 2])
    with gp:
        assert B.stage_gemm_mode(gp.stages[0], 1) == 0
        toks, logits, toks_o, logits_o = run(gp, op, model, prompt, 5)
    for a, b in zip(logits, logits_o):
        assert np.abs(a - b).max() <= LOGIT_ATOL
    assert toks.tolist() == toks_o.tolist()
