"""Stage-level pins of the oracle: the pages' staged == unstaged invariant, the handoff
traffic the book prints, and prefill/decode consistency."""
import json
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def build_pipeline(cfg, bounds, seed=synth.DEFAULT_SEED, gamma_mode="ones", max_seqs=1, max_len=128):
    stages = []
    for a, b in zip(bounds, bounds[1:]):
        w = synth.stage_weights(cfg, a, b, seed=seed, gamma_mode=gamma_mode)
        stages.append(oracle.Stage(cfg, a, b, w, max_seqs=max_seqs, max_len=max_len))
    return oracle.Pipeline(stages)


@pytest.fixture(scope="module")
def tiny_runs():
    """cfg 0 shapes, seeded non-unit gains, prompt 24 + 6 greedy steps, every split."""
    cfg = synth.CONFIGS[0]
    prompt = synth.prompt_tokens(cfg, 0, 24)
    runs = {}
    for bounds in ([0, 4], [0, 1, 4], [0, 2, 4], [0, 3, 4], [0, 1, 2, 3, 4]):
        p = build_pipeline(cfg, bounds, gamma_mode="seeded")
        toks, logits = p.generate([prompt], 6)
        kv = np.concatenate([s.k_cache for s in p.stages]), np.concatenate([s.v_cache for s in p.stages])
        runs[tuple(bounds)] = (toks, logits, p.stages[-1].features.copy(), kv)
    return runs


def test_staged_equals_unstaged_bit_for_bit(tiny_runs):
    """'Numerical correctness proof' of the RFC page: split and unsplit runs match
    bit-for-bit in logits, final features, KV state and generated-token feedback."""
    ref = tiny_runs[(0, 4)]
    for bounds, run in tiny_runs.items():
        assert np.array_equal(run[0], ref[0]), bounds
        for a, b in zip(run[1], ref[1]):
            assert np.array_equal(a, b), bounds
        assert np.array_equal(run[2], ref[2]), bounds
        assert np.array_equal(run[3][0], ref[3][0]) and np.array_equal(run[3][1], ref[3][1]), bounds


def test_tiny_run_is_not_degenerate(tiny_runs):
    _, logits, feats, _ = tiny_runs[(0, 4)]
    assert all(np.isfinite(l).all() for l in logits)
    assert np.allclose((feats.astype(np.float64) ** 2).mean(axis=1), 1.0, rtol=0.5)
    # greedy decoding of a random model may repeat one token; the per-position
    # predictions of the prompt must still vary
    cfg = synth.CONFIGS[0]
    p = build_pipeline(cfg, [0, 2, 4], gamma_mode="seeded")
    prompt = synth.prompt_tokens(cfg, 0, 24)
    p.forward(np.zeros(24, int), np.arange(24), prompt)
    assert len(set(oracle.greedy(p.logits()).tolist())) > 1


def test_book_pipeline_traffic_golden():
    """Handoff traffic of the book's CPU pipeline run: one f32 hidden vector per token per
    step crosses each boundary; 16 sends and 1.29 MB for 8 x 64-token prompts + 16 tokens."""
    g = json.load(open(os.path.join(GOLDEN, "book_pipeline_traffic.json")))
    w = g["workload"]
    cfg = synth.BOOK_CPU
    assert (cfg.n_layers, cfg.hidden, cfg.n_q_heads, cfg.n_kv_heads, cfg.vocab) == (
        w["n_layers"], w["hidden"], w["n_q_heads"], w["n_kv_heads"], w["vocab"])
    prompts = [synth.prompt_tokens(cfg, s, w["prompt_len"]) for s in range(w["prompts"])]
    tokens = {}
    for ranks, exp in g["pipeline"].items():
        n = int(ranks)
        bounds = [round(i * cfg.n_layers / n) for i in range(n + 1)]    # the book's default split
        assert bounds == exp["bounds"]
        p = build_pipeline(cfg, bounds, max_seqs=w["prompts"], max_len=96)
        tokens[n], _ = p.generate(prompts, w["new_tokens"])
        for calls, nbytes in zip(p.handoff_calls, p.handoff_bytes):
            assert calls == exp["rank0_send_calls"]
            assert round(nbytes / 1e6, 2) == exp["rank0_send_MB"]
    p1 = build_pipeline(cfg, [0, 4], max_seqs=w["prompts"], max_len=96)
    tokens[1], _ = p1.generate(prompts, w["new_tokens"])
    assert g["same_tokens"] and np.array_equal(tokens[1], tokens[2]) and np.array_equal(tokens[1], tokens[4])


def test_prefill_matches_token_by_token_decode():
    cfg = synth.CONFIGS[0]
    prompt = synth.prompt_tokens(cfg, 3, 12)
    a = build_pipeline(cfg, [0, 2, 4])
    ha = a.forward(np.zeros(12, int), np.arange(12), prompt)
    b = build_pipeline(cfg, [0, 2, 4])
    hb = np.concatenate([b.forward([0], [t], prompt[t:t + 1]) for t in range(12)])
    assert np.linalg.norm(ha - hb) <= 1e-6 * np.linalg.norm(ha)
    for sa, sb in zip(a.stages, b.stages):
        ka, kb = sa.k_cache.astype(np.float64), sb.k_cache.astype(np.float64)
        assert np.abs(ka - kb).max() <= 1e-3 * np.abs(ka).max()


def test_bf16_gemm_mode_stays_close():
    cfg = synth.CONFIGS[0]
    prompt = synth.prompt_tokens(cfg, 1, 16)
    a = build_pipeline(cfg, [0, 4])
    b = build_pipeline(cfg, [0, 4])
    fa = a.forward(np.zeros(16, int), np.arange(16), prompt)
    fb = b.forward(np.zeros(16, int), np.arange(16), prompt, gemm="bf16")
    rel = np.linalg.norm(fa - fb) / np.linalg.norm(fa)
    assert 1e-5 < rel < 5e-2        # bf16 operands move the result, but not far


def test_moe_stage_routes_and_runs():
    cfg = synth.reduced(synth.CONFIGS[2], 2, hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64,
                        vocab=512, n_experts=8, top_k=2, expert_ffn=64)
    prompt = synth.prompt_tokens(cfg, 0, 6)
    p = build_pipeline(cfg, [0, 1, 2])
    toks, logits = p.generate([prompt], 3)
    u = build_pipeline(cfg, [0, 2])
    toks_u, logits_u = u.generate([prompt], 3)
    assert np.array_equal(toks, toks_u)
    for a, b in zip(logits, logits_u):
        assert np.array_equal(a, b)


def test_batched_ragged_decode_equals_each_sequence_alone():
    """A decode step of several sequences at their own positions (ragged contexts, listed out
    of order) computes, row for row, what each sequence's step computes alone: the batched
    70B-shape parity rests on the oracle keeping the rows of a batch independent."""
    cfg = synth.CONFIGS[0]
    lens = [5, 17, 11]
    prompts = [synth.prompt_tokens(cfg, 20 + s, n) for s, n in enumerate(lens)]

    def prefilled():
        p = build_pipeline(cfg, [0, 2, 4], gamma_mode="seeded", max_seqs=3)
        for s, pr in enumerate(prompts):
            p.forward(np.full(len(pr), s), np.arange(len(pr)), pr)
        return p

    order = [2, 0, 1]
    toks = [int(prompts[s][-1]) for s in order]
    batched = prefilled().forward(order, [lens[s] for s in order], toks)
    for row, s in enumerate(order):
        alone = prefilled().forward([s], [lens[s]], [toks[row]])
        assert np.allclose(batched[row], alone[0], rtol=1e-12, atol=1e-12), s
