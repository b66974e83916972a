"""Dequantisation and indexing on the GPU, bit for bit, and the greedy tie rule.

Where the arithmetic around a dequantised weight is exact, the GPU must reproduce the
oracle's scale * q (or its bf16 rounding) exactly, not within a tolerance:
  - the embedding rows of the first stage ("RFC: pipeline placement across multiple GPUs for
    models larger than one device", section "What I found": the first stage embeds) are
    scale * q, a product that is exact in float32;
  - a GEMV of a one-hot input e_k returns column k of the dequantised matrix: one nonzero
    product (exact: an 11-bit scale times a 7-bit integer) and sums of zeros;
  - a bf16 tensor-core GEMM of one-hot rows returns columns of bf16(scale * q), the operand
    the GEMM dequantises into shared memory, times 1.0.
The greedy token is the lowest index among equal maxima ("41. Many GPUs: tensor, pipeline,
expert and data parallelism", section "Measured": near-ties decide whether greedy tokens
diverge): two identical readout rows that hold the maximum must give the lower index.
"""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def packed(B, q, s):
    rows, cols = q.shape
    qb, sb = B.stage_op_q8_device_bytes(rows, cols)
    qd = torch.empty(qb, dtype=torch.uint8, device="cuda")
    sd = torch.empty(sb, dtype=torch.uint8, device="cuda")
    B.stage_op_q8_pack(synth.Q8(q, s), qd, sd)
    return qd, sd


@pytest.mark.parametrize("rows,cols", [(32000, 4096), (1024, 256), (1000, 688)])
def test_embedding_rows_equal_dequant(cuda, rows, cols):
    from layer_range_stage_gb300 import binding as B
    q, s = synth.q8(synth.key(501, rows, cols), rows, cols)
    qd, sd = packed(B, q, s)
    rng = np.random.default_rng(rows)
    tok = np.unique(np.concatenate([[0, 1, rows - 2, rows - 1], rng.integers(0, rows, 40)])).astype(np.int32)
    out = torch.full((len(tok), cols), float("nan"), dtype=torch.float32, device="cuda")
    B.stage_op_embed(qd, sd, rows, cols, torch.from_numpy(tok).cuda(), out)
    torch.cuda.synchronize()
    want = oracle.dequant(q[tok], s[tok]).astype(np.float32)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("rows,cols", [(4096, 4096), (4096, 14336), (1001, 688)])
def test_gemv_one_hot_inputs_give_dequantised_columns(cuda, rows, cols):
    from layer_range_stage_gb300 import binding as B
    q, s = synth.q8(synth.key(502, rows, cols), rows, cols)
    qd, sd = packed(B, q, s)
    ks = np.array([0, 1, 31, 32, cols // 2 + 5, cols - 1])
    x = np.zeros((len(ks), cols), dtype=np.float32)
    x[np.arange(len(ks)), ks] = 1.0
    y = torch.full((len(ks), rows), float("nan"), dtype=torch.float32, device="cuda")
    B.stage_op_gemv(qd, sd, rows, cols, torch.from_numpy(x).cuda(), y)
    torch.cuda.synchronize()
    want = oracle.dequant(q, s)[:, ks].T.astype(np.float32)
    assert np.array_equal(y.cpu().numpy().view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("rows,cols,M", [(4096, 4096, 300), (1000, 688, 64)])
def test_bf16_gemm_one_hot_rows_give_bf16_dequantised_columns(cuda, rows, cols, M):
    from layer_range_stage_gb300 import binding as B
    q, s = synth.q8(synth.key(503, rows, cols), rows, cols)
    qd, sd = packed(B, q, s)
    kp = (cols + 255) // 256 * 256
    rng = np.random.default_rng(cols)
    ks = rng.integers(0, cols, M)
    ks[:4] = [0, 31, 32, cols - 1]
    a = np.zeros((M, kp), dtype=np.uint16)
    a[np.arange(M), ks] = 0x3F80  # bf16 1.0
    y = torch.full((M, rows), float("nan"), dtype=torch.float32, device="cuda")
    B.stage_op_gemm_bf16(torch.from_numpy(a.view(np.int16)).cuda(), qd, sd, rows, cols, y)
    torch.cuda.synchronize()
    want = oracle.bf16(oracle.dequant(q, s))[:, ks].T.astype(np.float32)
    assert np.array_equal(y.cpu().numpy().view(np.uint32), want.view(np.uint32))


def test_greedy_ties_go_to_the_lower_index(cuda):
    """The tiny model with a readout whose rows are all zero except two identical rows a < b,
    each 127 * sign(f_c) at the column c where the oracle's final features are largest: the
    logits of a and b are equal and the largest, so the greedy token must be a (and the
    oracle says so too).  Run for two pairs, one of them near the end of the vocabulary."""
    from layer_range_stage_gb300.pipeline import StagePipeline
    model = synth.CONFIGS[0]
    prompt = synth.prompt_tokens(model, 4, 24)
    n = len(prompt)
    ost = [oracle.Stage(model, a, b, synth.stage_weights(model, a, b), max_len=64) for a, b in ((0, 2), (2, 4))]
    f = ost[1].forward(np.zeros(n), np.arange(n), hidden_in=ost[0].forward(np.zeros(n), np.arange(n), tokens=prompt))
    f_last = f[-1].astype(np.float64)
    col = int(np.argmax(np.abs(f_last)))
    for a, b in ((5, 9), (model.vocab - 7, model.vocab - 1)):
        def endpoints(lo, hi, a=a, b=b):
            sw = synth.stage_weights(model, lo, hi, with_layers=False)
            if sw.lm_head is not None:
                q = np.zeros_like(sw.lm_head.q)
                q[[a, b], col] = 127 if f_last[col] > 0 else -127
                sc = sw.lm_head.s.copy()
                sc[b] = sc[a]  # identical rows: the same bytes and the same scales
                sw.lm_head = synth.Q8(q, sc)
            return sw
        with StagePipeline(model, [0, 2, 4], lambda l: synth.layer_weights(model, l), endpoints, max_seq_len=64,
                           max_tokens=32) as gp:
            lg = torch.empty((1, model.vocab), dtype=torch.float32, device="cuda")
            tok = gp.step(True, np.zeros(n), np.arange(n), prompt, rows=[n - 1], logits_out=lg)
            got = lg.cpu().numpy()[0]
        assert got[a] == got[b] and got[a] == got.max() and got[a] > 0
        assert int(tok[0]) == a
        assert int(oracle.greedy(got[None, :])[0]) == a
