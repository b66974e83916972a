"""GPU parity of the stage forward against the CPU oracle, through the C ABI.

Tolerances (stated for the float32 path): final hidden / features relative L2 <= 1e-3,
logits max-abs <= 2e-2, identical greedy tokens on the tiny config; staged and
monolithic GPU runs bit-exact (logits, features, KV, committed positions, tokens).
"""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

HIDDEN_RTOL = 1e-3
LOGIT_ATOL = 2e-2


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def gpu_pipeline(model, bounds, gamma_mode="ones", **kw):
    from layer_range_stage_gb300.pipeline import StagePipeline
    return StagePipeline(model, bounds, lambda l: synth.layer_weights(model, l, gamma_mode=gamma_mode),
                         lambda a, b: synth.stage_weights(model, a, b, gamma_mode=gamma_mode, with_layers=False), **kw)


def oracle_pipeline(model, bounds, gamma_mode="ones", max_seqs=1, max_len=256):
    return oracle.Pipeline([oracle.Stage(model, a, b, synth.stage_weights(model, a, b, gamma_mode=gamma_mode),
                                         max_seqs=max_seqs, max_len=max_len) for a, b in zip(bounds, bounds[1:])])


def run_gpu_greedy(gp, model, prompt, n_new):
    """Prefill + n_new - 1 decode steps through stage_pipeline_step; returns tokens,
    per-step logits and the last-step final features."""
    n = len(prompt)
    lg = torch.empty((1, model.vocab), dtype=torch.float32, device="cuda")
    tok = gp.step(True, np.zeros(n), np.arange(n), prompt, rows=[n - 1], logits_out=lg)
    toks, logits = [int(tok[0])], [lg.cpu().numpy().copy()]
    for t in range(n_new - 1):
        tok = gp.step(False, [0], [n + t], [toks[-1]], rows=[0], logits_out=lg)
        toks.append(int(tok[0]))
        logits.append(lg.cpu().numpy().copy())
    return np.array(toks), logits


@pytest.fixture(scope="module")
def tiny_oracle():
    model = synth.CONFIGS[0]
    prompt = synth.prompt_tokens(model, 0, 64)
    op = oracle_pipeline(model, [0, 2, 4], gamma_mode="seeded")
    toks, logits = op.generate([prompt], 17)
    kv = [(s.k_cache, s.v_cache) for s in op.stages]
    return model, prompt, toks[0], logits, op.stages[-1].features.copy(), kv


def test_tiny_matches_oracle_and_greedy_tokens(cuda, tiny_oracle):
    model, prompt, toks_o, logits_o, feat_o, kv_o = tiny_oracle
    with gpu_pipeline(model, [0, 2, 4], gamma_mode="seeded", max_seq_len=128, max_tokens=64) as gp:
        toks, logits = run_gpu_greedy(gp, model, prompt, 17)
        import layer_range_stage_gb300 as L
        # KV of block 1 (stage 0) and block 3 (stage 1) against the oracle's fp16 cache
        n_pos = 64 + 16
        for st, gl, (ko, vo), li in ((gp.stages[0], 1, kv_o[0], 1), (gp.stages[1], 3, kv_o[1], 1)):
            k, v = L.stage_read_kv(st, gl, 0, n_pos, model.n_kv_heads, model.head_dim)
            assert rel_l2(k.astype(np.float64), ko[li, 0, :, :n_pos].astype(np.float64)) <= HIDDEN_RTOL
            assert rel_l2(v.astype(np.float64), vo[li, 0, :, :n_pos].astype(np.float64)) <= HIDDEN_RTOL
    for a, b in zip(logits, logits_o):
        assert np.abs(a - b).max() <= LOGIT_ATOL
    assert toks.tolist() == toks_o.tolist()


def test_tiny_final_features_match_oracle(cuda, tiny_oracle):
    model, prompt, _, _, _, _ = tiny_oracle
    op = oracle_pipeline(model, [0, 2, 4], gamma_mode="seeded")
    n = len(prompt)
    f_o = op.forward(np.zeros(n), np.arange(n), prompt)
    # direct stage calls: stage 0 then stage 1, hidden buffers owned by the test
    from layer_range_stage_gb300 import binding as B
    cfgc = B.make_cfg(model, 1, 128, 64)
    st0 = B.stage_create(cfgc, 0, 2, synth.stage_weights(model, 0, 2, gamma_mode="seeded"))
    st1 = B.stage_create(cfgc, 2, 4, synth.stage_weights(model, 2, 4, gamma_mode="seeded"))
    try:
        h = torch.empty((n, model.hidden), dtype=torch.float32, device="cuda")
        f = torch.empty_like(h)
        B.stage_prefill(st0, np.zeros(n), np.arange(n), tokens=prompt, hidden_out=h)
        # the handoff after stage 0 against the oracle's stage 0 output
        h_o = oracle_pipeline(model, [0, 2, 4], gamma_mode="seeded").stages[0].forward(np.zeros(n), np.arange(n), prompt)
        assert rel_l2(h.cpu().numpy(), h_o) <= HIDDEN_RTOL
        B.stage_prefill(st1, np.zeros(n), np.arange(n), hidden_in=h, hidden_out=f)
        torch.cuda.synchronize()
        assert rel_l2(f.cpu().numpy(), f_o) <= HIDDEN_RTOL
    finally:
        B.stage_destroy(st0)
        B.stage_destroy(st1)


def test_staged_equals_monolithic_bit_exact(cuda):
    model = synth.CONFIGS[0]
    prompt = synth.prompt_tokens(model, 5, 40)
    import layer_range_stage_gb300 as L
    runs = {}
    for bounds in ([0, 4], [0, 2, 4], [0, 1, 2, 3, 4], [0, 3, 4]):
        with gpu_pipeline(model, bounds, gamma_mode="seeded", max_seq_len=128, max_tokens=64) as gp:
            toks, logits = run_gpu_greedy(gp, model, prompt, 8)
            kv = []
            for gl in range(4):
                si = max(i for i, b in enumerate(bounds[:-1]) if b <= gl)
                kv.append(L.stage_read_kv(gp.stages[si], gl, 0, 40 + 7, model.n_kv_heads, model.head_dim))
            runs[tuple(bounds)] = (toks, logits, kv, gp.committed(0))
    ref = runs[(0, 4)]
    for b, r in runs.items():
        assert np.array_equal(r[0], ref[0]), b
        for x, y in zip(r[1], ref[1]):
            assert np.array_equal(x, y), b
        for (k1, v1), (k2, v2) in zip(r[2], ref[2]):
            assert np.array_equal(k1.view(np.uint16), k2.view(np.uint16)) and np.array_equal(v1.view(np.uint16), v2.view(np.uint16)), b
        assert set(r[3]) == {40 + 7}, b


def test_graph_generate_matches_step_by_step(cuda):
    model = synth.CONFIGS[0]
    prompt = synth.prompt_tokens(model, 7, 20)
    import layer_range_stage_gb300 as L
    out = {}
    for mode in ("steps", "graph", "nograph"):
        with gpu_pipeline(model, [0, 2, 4], max_seq_len=128, max_tokens=64) as gp:
            n = len(prompt)
            first = gp.step(True, np.zeros(n), np.arange(n), prompt, rows=[n - 1])
            if mode == "steps":
                toks = [int(first[0])]
                for t in range(10):
                    toks.append(int(gp.step(False, [0], [n + t], [toks[-1]], rows=[0])[0]))
                gen = np.array(toks[1:])
            else:
                gen = gp.generate([0], first, 10, use_graph=(mode == "graph"))[:, 0]
            k, v = L.stage_read_kv(gp.stages[1], 3, 0, n + 10, model.n_kv_heads, model.head_dim)
            out[mode] = (gen, k.view(np.uint16).copy(), gp.committed(0))
    for mode in ("graph", "nograph"):
        assert np.array_equal(out[mode][0], out["steps"][0])
        assert np.array_equal(out[mode][1], out["steps"][1])
        assert out[mode][2] == out["steps"][2] == [len(prompt) + 10] * 2


def test_batched_ragged_decode_matches_oracle(cuda):
    model = synth.CONFIGS[0]
    lens = [5, 33, 17]
    prompts = [synth.prompt_tokens(model, 10 + i, n) for i, n in enumerate(lens)]
    op = oracle_pipeline(model, [0, 2, 4], max_seqs=3, max_len=128)
    toks_o, logits_o = op.generate(prompts, 4)
    with gpu_pipeline(model, [0, 2, 4], max_seqs=3, max_seq_len=128, max_tokens=64) as gp:
        seq = np.concatenate([np.full(n, s) for s, n in enumerate(lens)])
        pos = np.concatenate([np.arange(n) for n in lens])
        lg = torch.empty((3, model.vocab), dtype=torch.float32, device="cuda")
        rows = np.cumsum(lens) - 1
        tok = gp.step(True, seq, pos, np.concatenate(prompts), rows=rows, logits_out=lg)
        got = [tok.copy()]
        assert np.abs(lg.cpu().numpy() - logits_o[0]).max() <= LOGIT_ATOL
        cur = np.array(lens)
        for t in range(3):
            tok = gp.step(False, [0, 1, 2], cur, got[-1], rows=[0, 1, 2], logits_out=lg)
            cur = cur + 1
            got.append(tok.copy())
            assert np.abs(lg.cpu().numpy() - logits_o[t + 1]).max() <= LOGIT_ATOL
    assert np.array_equal(np.stack(got, axis=1), toks_o)


def test_dense_8b_shape_two_blocks_matches_oracle(cuda):
    """Full width of the 8B-shape model (hidden 4096, FFN 14336, vocab 32000, 32q/8kv x 128)
    at reduced depth, split 1/1."""
    model = synth.reduced(synth.CONFIGS[1], 2)
    prompt = synth.prompt_tokens(model, 0, 12)
    op = oracle_pipeline(model, [0, 1, 2], max_len=64)
    toks_o, logits_o = op.generate([prompt], 3)
    f_o = op.stages[-1].features
    with gpu_pipeline(model, [0, 1, 2], max_seq_len=64, max_tokens=16) as gp:
        toks, logits = run_gpu_greedy(gp, model, prompt, 3)
    for a, b in zip(logits, logits_o):
        assert np.abs(a - b).max() <= LOGIT_ATOL
    assert toks.tolist() == toks_o[0].tolist()


# ----------------------------------------------------------------------------- host-side checks on a live stage

@pytest.fixture()
def tiny_pair(cuda):
    from layer_range_stage_gb300 import binding as B
    model = synth.CONFIGS[0]
    cfgc = B.make_cfg(model, 2, 64, 32)
    st0 = B.stage_create(cfgc, 0, 2, synth.stage_weights(model, 0, 2))
    st1 = B.stage_create(cfgc, 2, 4, synth.stage_weights(model, 2, 4))
    yield model, B, st0, st1
    B.stage_destroy(st0)
    B.stage_destroy(st1)


def test_handoff_and_position_checks(tiny_pair):
    model, B, st0, st1 = tiny_pair
    h = torch.zeros((4, model.hidden), dtype=torch.float32, device="cuda")
    toks = synth.prompt_tokens(model, 0, 4)
    with pytest.raises(B.StageError) as e:                         # tokens to a non-first stage
        B.stage_prefill(st1, np.zeros(4), np.arange(4), tokens=toks, hidden_out=h)
    assert e.value.code == B.STAGE_E_HANDOFF
    with pytest.raises(B.StageError) as e:                         # hidden to the first stage
        B.stage_prefill(st0, np.zeros(4), np.arange(4), tokens=toks, hidden_in=h, hidden_out=h)
    assert e.value.code == B.STAGE_E_HANDOFF
    wrong = torch.zeros((4, model.hidden + 32), dtype=torch.float32, device="cuda")
    with pytest.raises(B.StageError) as e:                         # wrong width
        B.stage_prefill(st1, np.zeros(4), np.arange(4), hidden_in=wrong, hidden_out=h)
    assert e.value.code == B.STAGE_E_HANDOFF
    with pytest.raises(B.StageError) as e:                         # wrong n
        B.stage_prefill(st1, np.zeros(3), np.arange(3), hidden_in=h, hidden_out=h)
    assert e.value.code == B.STAGE_E_HANDOFF
    with pytest.raises(B.StageError) as e:                         # does not start at committed length
        B.stage_prefill(st0, np.zeros(4), np.arange(1, 5), tokens=toks, hidden_out=h)
    assert e.value.code == B.STAGE_E_POSITION
    with pytest.raises(B.StageError) as e:                         # non-contiguous
        B.stage_prefill(st0, np.zeros(4), [0, 1, 3, 4], tokens=toks, hidden_out=h)
    assert e.value.code == B.STAGE_E_POSITION
    B.stage_prefill(st0, np.zeros(4), np.arange(4), tokens=toks, hidden_out=h)
    B.stage_commit(st0, [0], [4])
    with pytest.raises(B.StageError) as e:                         # commit beyond what was written
        B.stage_commit(st0, [0], [6])
    assert e.value.code == B.STAGE_E_STATE
    h1 = h[:1].contiguous()
    with pytest.raises(B.StageError) as e:                         # past max_seq_len
        B.stage_truncate(st0, 0, 4)
        for p in range(4, 65):
            B.stage_decode(st0, [0], [p], tokens=[1], hidden_out=h1)
            B.stage_commit(st0, [0], [p + 1])
    assert e.value.code == B.STAGE_E_POSITION and B.stage_committed_len(st0, 0) == 64
    with pytest.raises(B.StageError) as e:
        B.stage_logits(st0, [0])
    assert e.value.code == B.STAGE_E_NOT_LAST
    with pytest.raises(B.StageError) as e:
        B.stage_decode(st0, [1, 1], [0, 0], tokens=[1, 1], hidden_out=h[:2].contiguous())
    assert e.value.code == B.STAGE_E_INVALID


def test_busy_refusal(tiny_pair):
    model, B, st0, st1 = tiny_pair
    h = torch.zeros((1, model.hidden), dtype=torch.float32, device="cuda")
    B.stage_debug_inject(st0, 1, 1)
    with pytest.raises(B.StageError) as e:
        B.stage_decode(st0, [0], [0], tokens=[3], hidden_out=h)
    assert e.value.code == B.STAGE_E_BUSY and B.stage_committed_len(st0, 0) == 0
    B.stage_debug_inject(st0, 1, 0)
    B.stage_decode(st0, [0], [0], tokens=[3], hidden_out=h)


def test_injected_failure_publishes_nothing_and_retry_is_identical(cuda):
    from layer_range_stage_gb300 import binding as B
    model = synth.CONFIGS[0]
    prompt = synth.prompt_tokens(model, 3, 10)
    with gpu_pipeline(model, [0, 2, 4], max_seq_len=64, max_tokens=16) as gp:
        lg = torch.empty((1, model.vocab), dtype=torch.float32, device="cuda")
        gp.step(True, np.zeros(10), np.arange(10), prompt, rows=[9], logits_out=lg)
        ref = lg.cpu().numpy().copy()
        # fail the second stage of the next step: no stage may advance
        B.stage_debug_inject(gp.stages[1], 2, B.STAGE_E_INJECTED)
        with pytest.raises(B.StageError) as e:
            gp.step(False, [0], [10], [5], rows=[0], logits_out=lg)
        assert e.value.code == B.STAGE_E_INJECTED
        assert gp.committed(0) == [10, 10]
        gp.step(False, [0], [10], [5], rows=[0], logits_out=lg)
        a = lg.cpu().numpy().copy()
        assert gp.committed(0) == [11, 11]
        # refill: truncate both stages back and redo the same step -> the same bits
        for st in gp.stages:
            B.stage_truncate(st, 0, 10)
        gp.step(False, [0], [10], [5], rows=[0], logits_out=lg)
        assert np.array_equal(a, lg.cpu().numpy())
        # reset and replay the prefill: identical logits
        for st in gp.stages:
            B.stage_reset(st)
        gp.step(True, np.zeros(10), np.arange(10), prompt, rows=[9], logits_out=lg)
        assert np.array_equal(ref, lg.cpu().numpy())
        calls, nbytes = gp.handoff_stats(0)
        # four handoffs: the failed step ran no stage (every stage's call is validated
        # before the first launch)
        assert calls == 4 and nbytes == (10 + 1 + 1 + 10) * model.hidden * 4
