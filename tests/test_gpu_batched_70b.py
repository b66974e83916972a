"""The 70B-shape batched decode at full width against the oracle, through the C ABI.

Hidden 8192, 64 q / 8 kv heads x 128, SwiGLU 28672, vocab 128256, int8 block-32 weights;
64 sequences whose KV lengths are uniform in [128, 4096]; 4 stages chained, one block each
(the model's depth is reduced to 4 blocks: every block has the same shapes).  The caches
start from seeded fp16 N(0, 1) rows written through stage_write_kv (and into the oracle's
caches; every block gets the same rows), then one decode step of 64 tokens -- one per
sequence, at its own position -- runs through the 4 stages.  Every stage is checked against
the oracle's block fed the GPU's own input to that stage (teacher-forced: relative L2 <= 1e-3,
the float32 tolerance); the readout against the oracle's on
sampled vocabulary rows (max-abs <= 2e-2) and the greedy tokens against the oracle's full
argmax wherever its top-2 margin exceeds that tolerance.

Both decode paths of a 64-token call: the float32 GEMV path, and the tensor-core path (the
stage's GEMM threshold set to 64: every projection a tcgen05 GEMM with bf16 operands and f32
accumulation) against the oracle with every GEMM operand rounded to bf16, where a block
output is held to one bf16 ulp (2^-8) in relative L2 -- the bf16 tolerance of the prefill
tests.  A call of at most 64 tokens takes the weight-streaming GEMM (128 weight rows against
the call's tokens, K split over several CTAs where the weight tiles are few).  The readout is
the float32 GEMV on the f32 path and that bf16 GEMM on the tensor-core path; like every GEMM
of that path it is checked against the oracle with its operands (features and dequantised head)
rounded to bf16, to the same logit tolerance.
"""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

HIDDEN_RTOL = {"f32": 1e-3, "bf16": 2.0 ** -8}
LOGIT_ATOL = 2e-2
NSEQ = 64


def rel_l2(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def kv_rows(model, seq, n):
    """Seeded fp16 K and V rows [Hkv, n, D] of one sequence."""
    shape = (model.n_kv_heads, n, model.head_dim)
    size = model.n_kv_heads * n * model.head_dim
    k = synth.normal_f32(synth.key(4400, seq, 0), 0, size, 1.0).reshape(shape).astype(np.float16)
    v = synth.normal_f32(synth.key(4400, seq, 1), 0, size, 1.0).reshape(shape).astype(np.float16)
    return k, v


@pytest.mark.parametrize("path", ["f32", "bf16"])
def test_70b_shape_batched_decode_ragged_64(cuda, path):
    from layer_range_stage_gb300 import binding as B
    model = synth.reduced(synth.CONFIGS[4], 4)
    lens = np.random.default_rng(4401).integers(128, 4097, NSEQ)
    max_len = int(lens.max()) + 1
    cfgc = B.make_cfg(model, NSEQ, max_len, NSEQ, NSEQ if path == "bf16" else 0)
    seqs = np.arange(NSEQ)
    toks = np.random.default_rng(4402).integers(0, model.vocab, NSEQ)
    stages, ws = [], [synth.stage_weights(model, li, li + 1) for li in range(4)]
    kv = [kv_rows(model, s, int(lens[s])) for s in range(NSEQ)]
    try:
        hs = []
        for li in range(4):
            st = B.stage_create(cfgc, li, li + 1, ws[li])
            stages.append(st)
            assert B.stage_gemm_mode(st, NSEQ) == (1 if path == "bf16" else 0)
            for s in range(NSEQ):
                B.stage_write_kv(st, li, s, 0, kv[s][0], kv[s][1])
            B.stage_commit(st, seqs, lens)
            h = torch.empty((NSEQ, model.hidden), dtype=torch.float32, device="cuda")
            if li == 0:
                B.stage_decode(st, seqs, lens, tokens=toks, hidden_out=h)
            else:
                B.stage_decode(st, seqs, lens, hidden_in=hs[-1], hidden_out=h)
            hs.append(h)
        lg = torch.empty((NSEQ, model.vocab), dtype=torch.float32, device="cuda")
        am = torch.empty((NSEQ,), dtype=torch.int32, device="cuda")
        B.stage_logits(stages[-1], np.arange(NSEQ), lg, am)
        torch.cuda.synchronize()
        hg = [h.cpu().numpy() for h in hs]
        logits, argmax = lg.cpu().numpy(), am.cpu().numpy()
    finally:
        for st in stages:
            B.stage_destroy(st)

    # the oracle on every stage, each fed the GPU's input to that stage
    for li in range(4):
        w = ws[li]
        ost = oracle.Stage(model, li, li + 1, w, max_seqs=NSEQ, max_len=max_len, cache_dequant=False)
        for s in range(NSEQ):
            ost.k_cache[0, s, :, :lens[s]] = kv[s][0]
            ost.v_cache[0, s, :, :lens[s]] = kv[s][1]
        if li == 0:
            ref = ost.forward(seqs, lens, tokens=toks, gemm=path)
        else:
            ref = ost.forward(seqs, lens, hidden_in=hg[li - 1], gemm=path)
        assert rel_l2(hg[li], ref) <= HIDDEN_RTOL[path], li
        if li == 3:
            head = w.lm_head
            # the readout of the GPU's own features; on the tensor-core path the readout is a
            # GEMM like the others, so its operands are rounded to bf16 on the oracle's side too
            feats = hg[3].astype(np.float64)
            rd = (lambda m: oracle.bf16(m)) if path == "bf16" else (lambda m: m)
            feats = rd(feats)
            rng = np.random.default_rng(4403)
            sample = np.unique(np.concatenate([rng.integers(0, model.vocab, 512), argmax]))
            lo = oracle.matvec(rd(oracle.dequant(head.q[sample], head.s[sample])), feats)
            assert np.abs(logits[:, sample] - lo).max() <= LOGIT_ATOL
            # full argmax of the oracle, in chunks of vocabulary rows
            best = np.full(NSEQ, -np.inf)
            second = np.full(NSEQ, -np.inf)
            arg = np.zeros(NSEQ, dtype=np.int64)
            for r0 in range(0, model.vocab, 8192):
                r1 = min(model.vocab, r0 + 8192)
                chunk = oracle.matvec(rd(oracle.dequant(head.q[r0:r1], head.s[r0:r1])), feats)
                for t in range(NSEQ):
                    c = chunk[t]
                    j = int(np.argmax(c))
                    top2 = np.sort(c)[-2:]
                    if c[j] > best[t]:
                        second[t] = max(best[t], top2[0])
                        best[t], arg[t] = c[j], r0 + j
                    else:
                        second[t] = max(second[t], c[j])
            for t in range(NSEQ):
                if best[t] - second[t] > 2 * LOGIT_ATOL:
                    assert argmax[t] == arg[t], t
