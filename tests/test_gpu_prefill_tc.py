"""GPU parity of the tensor-core prefill (bf16 operands, f32 accumulation) against the
oracle's bf16 GEMM mode, through the C ABI.

A stage created with gemm_bf16_min_tokens = m runs every projection of a call with at
least m tokens as a tcgen05 GEMM ("41. Many GPUs: tensor, pipeline, expert and data
parallelism", section "Pipeline parallelism": prefill is the block loop over all prompt
tokens); shorter calls stay on the float32 GEMV.  The oracle rounds the same operands to
bf16 and accumulates in float64.

Tolerances, from the arithmetic.  The tensor-core GEMM itself is held to the oracle at
relative L2 5e-7 sqrt(K) (the tcgen05 GEMM tests).  A block output is not: a value that
differs by a relative d before it is rounded to fp16 (K/V) or bf16 (the next GEMM
operand) lands on the other side of a rounding boundary with probability ~ d / ulp, so
every rounding turns a difference d into noise ~ sqrt(d ulp), and a block chains four of
them.  Perturbing the oracle's own GEMM outputs by 1e-7 already moves a bf16 block of the
8B-shape model by ~1e-3 (2e-5 in float32 mode).  So:
  - K/V of a first block (identical GEMM operands on both sides, one fp16 rounding):
    relative L2 <= 2 sqrt(5e-7 sqrt(K) 2^-11);
  - a block output, or features after several blocks: one bf16 ulp, 2^-8, and closer to
    the bf16 oracle than to the float32 one by a factor of 2 at least;
  - logits from teacher-forced features: max-abs <= 2e-2; staged and monolithic runs
    bit-exact.
"""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

LOGIT_ATOL = 2e-2
BF16_NOISE = 2.0 ** -8   # one bf16 ulp, relative


def kv_tol(K):
    """fp16 rounding noise of K/V computed from identical operands with float32 accumulation."""
    return 2.0 * np.sqrt(5e-7 * np.sqrt(K) * 2.0 ** -11)


def rel_l2(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def gpu_pipeline(model, bounds, gamma_mode="seeded", **kw):
    from layer_range_stage_gb300.pipeline import StagePipeline
    return StagePipeline(model, bounds, lambda l: synth.layer_weights(model, l, gamma_mode=gamma_mode),
                         lambda a, b: synth.stage_weights(model, a, b, gamma_mode=gamma_mode, with_layers=False), **kw)


def oracle_pipeline(model, bounds, gamma_mode="seeded", max_len=256):
    return oracle.Pipeline([oracle.Stage(model, a, b, synth.stage_weights(model, a, b, gamma_mode=gamma_mode),
                                         max_seqs=1, max_len=max_len) for a, b in zip(bounds, bounds[1:])])


def test_gemm_mode_selection(cuda):
    from layer_range_stage_gb300 import binding as B
    dense, moe = synth.CONFIGS[0], synth.reduced(synth.CONFIGS[2], 1)
    st = B.stage_create(B.make_cfg(dense, 1, 64, 32, 8), 0, 4, synth.stage_weights(dense, 0, 4))
    try:
        # single-token calls take the persistent decode kernel (2)
        assert [B.stage_gemm_mode(st, n) for n in (1, 2, 7, 8, 32)] == [2, 0, 0, 1, 1]
    finally:
        B.stage_destroy(st)
    st = B.stage_create(B.make_cfg(dense, 1, 64, 32, 0), 0, 4, synth.stage_weights(dense, 0, 4))
    try:
        assert B.stage_gemm_mode(st, 32) == 0
    finally:
        B.stage_destroy(st)
    # MoE stages keep the GEMV (the expert gather) for several tokens; a single token takes
    # the persistent decode kernel (router and top-k inside it)
    st = B.stage_create(B.make_cfg(moe, 1, 64, 32, 8), 0, 1, synth.stage_weights(moe, 0, 1))
    try:
        assert B.stage_gemm_mode(st, 32) == 0 and B.stage_gemm_mode(st, 1) == 2
    finally:
        B.stage_destroy(st)


def test_tiny_bf16_blocks_teacher_forced(cuda):
    """Each block on its own (one-block stages), fed the GPU's own input: the block output
    and its K/V against the oracle's bf16 block on that same input (and against the
    float32 block, which must be farther away).  The first block's GEMM operands are
    identical on both sides (embedding rows), so its K/V agree to fp16 rounding noise."""
    model = synth.CONFIGS[0]
    n = 64
    prompt = synth.prompt_tokens(model, 0, n)
    from layer_range_stage_gb300 import binding as B
    cfgc = B.make_cfg(model, 1, 128, 64, 16)
    hin = None
    for li in range(4):
        st = B.stage_create(cfgc, li, li + 1, synth.stage_weights(model, li, li + 1, gamma_mode="seeded"))
        ost = oracle.Stage(model, li, li + 1, synth.stage_weights(model, li, li + 1, gamma_mode="seeded"),
                           max_seqs=1, max_len=128)
        try:
            out = torch.empty((n, model.hidden), dtype=torch.float32, device="cuda")
            if li == 0:
                B.stage_prefill(st, np.zeros(n), np.arange(n), tokens=prompt, hidden_out=out)
                kw = dict(tokens=prompt)
            else:
                B.stage_prefill(st, np.zeros(n), np.arange(n), hidden_in=hin, hidden_out=out)
                kw = dict(hidden_in=hin.cpu().numpy())
            ref = ost.forward(np.zeros(n), np.arange(n), gemm="bf16", **kw)
            kref = ost.k_cache[0, 0, :, :n].astype(np.float64), ost.v_cache[0, 0, :, :n].astype(np.float64)
            ref32 = oracle.Stage(model, li, li + 1, synth.stage_weights(model, li, li + 1, gamma_mode="seeded"),
                                 max_seqs=1, max_len=128).forward(np.zeros(n), np.arange(n), gemm="f32", **kw)
            torch.cuda.synchronize()
            k, v = B.stage_read_kv(st, li, 0, n, model.n_kv_heads, model.head_dim)
            tol = kv_tol(model.hidden) if li == 0 else BF16_NOISE
            assert rel_l2(k.astype(np.float64), kref[0]) <= tol, li
            assert rel_l2(v.astype(np.float64), kref[1]) <= tol, li
            got = out.cpu().numpy()
            assert rel_l2(got, ref) <= BF16_NOISE, li
            assert rel_l2(got, ref32) > 2 * rel_l2(got, ref), li
            hin = out
        finally:
            B.stage_destroy(st)


def test_tiny_bf16_prefill_then_f32_decode(cuda):
    """64-token prefill on the tensor cores, then greedy decode on the GEMV, through the
    pipeline.  Over four blocks the prefill logits are held to one bf16 ulp (relative L2)
    and to max-abs 2e-2, every decode step's logits too while the greedy tokens agree, and
    greedy tokens must agree wherever the oracle's top-2 logit margin exceeds that noise."""
    model = synth.CONFIGS[0]
    prompt = synth.prompt_tokens(model, 0, 64)
    n = len(prompt)
    op = oracle_pipeline(model, [0, 2, 4])
    toks_o, logits_o = op.generate([prompt], 17, prefill_gemm="bf16", decode_gemm="f32")
    import layer_range_stage_gb300 as L
    with gpu_pipeline(model, [0, 2, 4], max_seq_len=128, max_tokens=64, gemm_bf16_min_tokens=16) as gp:
        assert L.stage_gemm_mode(gp.stages[0], 64) == 1 and L.stage_gemm_mode(gp.stages[0], 1) == 2
        lg = torch.empty((1, model.vocab), dtype=torch.float32, device="cuda")
        tok = gp.step(True, np.zeros(n), np.arange(n), prompt, rows=[n - 1], logits_out=lg)
        toks, logits = [int(tok[0])], [lg.cpu().numpy().copy()]
        for t in range(16):
            tok = gp.step(False, [0], [n + t], [toks[-1]], rows=[0], logits_out=lg)
            toks.append(int(tok[0]))
            logits.append(lg.cpu().numpy().copy())
    assert rel_l2(logits[0], logits_o[0]) <= BF16_NOISE
    for t, (a, b) in enumerate(zip(logits, logits_o)):
        assert rel_l2(a, b) <= BF16_NOISE, t
        assert np.abs(a - b).max() <= LOGIT_ATOL, t
        if toks[t] != toks_o[0][t]:
            top2 = np.sort(b[0])[-2:]
            assert top2[1] - top2[0] <= 4 * BF16_NOISE * np.abs(b).max(), t
            break


def test_tiny_bf16_staged_equals_monolithic_bit_exact(cuda):
    model = synth.CONFIGS[0]
    prompt = synth.prompt_tokens(model, 5, 40)
    import layer_range_stage_gb300 as L
    runs = {}
    for bounds in ([0, 4], [0, 2, 4], [0, 1, 2, 3, 4]):
        with gpu_pipeline(model, bounds, max_seq_len=128, max_tokens=64, gemm_bf16_min_tokens=16) as gp:
            lg = torch.empty((2, model.vocab), dtype=torch.float32, device="cuda")
            gp.step(True, np.zeros(40), np.arange(40), prompt, rows=[0, 39], logits_out=lg)
            kv = []
            for gl in range(4):
                si = max(i for i, b in enumerate(bounds[:-1]) if b <= gl)
                k, v = L.stage_read_kv(gp.stages[si], gl, 0, 40, model.n_kv_heads, model.head_dim)
                kv.append((k.view(np.uint16).copy(), v.view(np.uint16).copy()))
            runs[tuple(bounds)] = (lg.cpu().numpy().copy(), kv)
    ref = runs[(0, 4)]
    for b, r in runs.items():
        assert np.array_equal(r[0], ref[0]), b
        for (k1, v1), (k2, v2) in zip(r[1], ref[1]):
            assert np.array_equal(k1, k2) and np.array_equal(v1, v2), b


def test_dense_8b_width_prefill_300_tokens(cuda):
    """Full width of the 8B-shape model at depth 2, split 1/1: a 300-token prefill spans two
    256-token GEMM tiles with a ragged tail; every projection shape of the model runs."""
    model = synth.reduced(synth.CONFIGS[1], 2)
    n = 300
    prompt = synth.prompt_tokens(model, 1, n)
    rows = [0, 137, 255, 256, n - 1]
    op = oracle_pipeline(model, [0, 1, 2], max_len=320)
    h_o = op.stages[0].forward(np.zeros(n), np.arange(n), tokens=prompt, gemm="bf16")
    kv_o = op.stages[0].k_cache[0, 0, :, :n], op.stages[0].v_cache[0, 0, :, :n]
    from layer_range_stage_gb300 import binding as B
    cfgc = B.make_cfg(model, 1, 320, n, 64)
    st0 = B.stage_create(cfgc, 0, 1, synth.stage_weights(model, 0, 1, gamma_mode="seeded"))
    st1 = B.stage_create(cfgc, 1, 2, synth.stage_weights(model, 1, 2, gamma_mode="seeded"))
    try:
        assert B.stage_gemm_mode(st0, n) == 1
        h = torch.empty((n, model.hidden), dtype=torch.float32, device="cuda")
        f = torch.empty_like(h)
        B.stage_prefill(st0, np.zeros(n), np.arange(n), tokens=prompt, hidden_out=h)
        B.stage_prefill(st1, np.zeros(n), np.arange(n), hidden_in=h, hidden_out=f)
        lg = torch.empty((len(rows), model.vocab), dtype=torch.float32, device="cuda")
        B.stage_logits(st1, rows, lg)
        torch.cuda.synchronize()
        k, v = B.stage_read_kv(st0, 0, 0, n, model.n_kv_heads, model.head_dim)
        hg, fg = h.cpu().numpy(), f.cpu().numpy()
        assert rel_l2(k.astype(np.float64), kv_o[0].astype(np.float64)) <= kv_tol(model.hidden)
        assert rel_l2(v.astype(np.float64), kv_o[1].astype(np.float64)) <= kv_tol(model.hidden)
        assert rel_l2(hg, h_o) <= BF16_NOISE
        h_f32 = oracle_pipeline(model, [0, 1, 2], max_len=320).stages[0].forward(
            np.zeros(n), np.arange(n), tokens=prompt, gemm="f32")
        assert rel_l2(hg, h_f32) > 2 * rel_l2(hg, h_o)
        # stage 1 teacher-forced on the GPU's handoff; the readout of its features
        f_o = op.stages[1].forward(np.zeros(n), np.arange(n), hidden_in=hg, gemm="bf16")
        assert rel_l2(fg, f_o) <= BF16_NOISE
        assert np.abs(lg.cpu().numpy() - op.logits(rows)).max() <= LOGIT_ATOL
    finally:
        B.stage_destroy(st0)
        B.stage_destroy(st1)


def test_dense_8b_prefill_4x512_one_call(cuda):
    """The prefill workload of the benchmark at full width: four seeded prompts of 512 tokens
    in one tensor-core call through two 8B-shape blocks (split 1/1), so the attention's
    query tiles meet sequence boundaries inside the launch.  Against the bf16-mode oracle:
    block 0's output and its K/V at sampled positions of every sequence, block 1
    teacher-forced on the GPU's handoff, and the readout of each sequence's last row
    (logits max-abs <= 2e-2).  The achieved relative L2 of the features is printed beside
    the float32 path's 1e-3."""
    from layer_range_stage_gb300 import binding as B
    model = synth.reduced(synth.CONFIGS[1], 2)
    ns, plen = 4, 512
    n = ns * plen
    prompt = np.concatenate([synth.prompt_tokens(model, 100 + q, plen) for q in range(ns)])
    seq, pos = np.repeat(np.arange(ns), plen), np.tile(np.arange(plen), ns)
    rows = list(np.arange(1, ns + 1) * plen - 1)
    cfgc = B.make_cfg(model, ns, plen, n, 64)
    st0 = B.stage_create(cfgc, 0, 1, synth.stage_weights(model, 0, 1, gamma_mode="seeded"))
    st1 = B.stage_create(cfgc, 1, 2, synth.stage_weights(model, 1, 2, gamma_mode="seeded"))
    try:
        assert B.stage_gemm_mode(st0, n) == 1
        h = torch.empty((n, model.hidden), dtype=torch.float32, device="cuda")
        f = torch.empty_like(h)
        B.stage_prefill(st0, seq, pos, tokens=prompt, hidden_out=h)
        B.stage_prefill(st1, seq, pos, hidden_in=h, hidden_out=f)
        lg = torch.empty((ns, model.vocab), dtype=torch.float32, device="cuda")
        B.stage_logits(st1, rows, lg)
        torch.cuda.synchronize()
        kv = [B.stage_read_kv(st0, 0, q, plen, model.n_kv_heads, model.head_dim) for q in range(ns)]
        hg, fg, lgg = h.cpu().numpy(), f.cpu().numpy(), lg.cpu().numpy()
    finally:
        B.stage_destroy(st0)
        B.stage_destroy(st1)
    o0 = oracle.Stage(model, 0, 1, synth.stage_weights(model, 0, 1, gamma_mode="seeded"), max_seqs=ns, max_len=plen)
    h_o = o0.forward(seq, pos, tokens=prompt, gemm="bf16")
    err_h = rel_l2(hg, h_o)
    assert err_h <= BF16_NOISE
    rng = np.random.default_rng(512)
    ps = np.unique(np.concatenate([[0, 15, 16, 63, 64, plen - 1], rng.integers(0, plen, 26)]))
    for q in range(ns):
        k, v = kv[q]
        assert rel_l2(k[:, ps].astype(np.float64), o0.k_cache[0, q][:, ps].astype(np.float64)) <= kv_tol(model.hidden), q
        assert rel_l2(v[:, ps].astype(np.float64), o0.v_cache[0, q][:, ps].astype(np.float64)) <= kv_tol(model.hidden), q
    o1 = oracle.Stage(model, 1, 2, synth.stage_weights(model, 1, 2, gamma_mode="seeded"), max_seqs=ns, max_len=plen)
    f_o = o1.forward(seq, pos, hidden_in=hg, gemm="bf16")
    err_f = rel_l2(fg, f_o)
    assert err_f <= BF16_NOISE
    lo = o1.logits(rows)
    err_l = float(np.abs(lgg - lo).max())
    print(f"4x512 bf16 prefill: block output rel L2 {err_h:.3e}, final features rel L2 {err_f:.3e} "
          f"(float32 path tolerance 1e-3), logits max-abs {err_l:.3e} (tolerance {LOGIT_ATOL})")
    assert err_l <= LOGIT_ATOL
