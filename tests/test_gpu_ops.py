"""Kernel-level parity at full workload sizes, through the C ABI (include/stage_ops.h).

GEMV: the 8B-shape projections (and ragged shapes) against the oracle's dequantised
dot products on sampled rows -- the oracle regenerates just those rows from the seeded
generator.  Attention: every head of a context-2048 decode step in the launch
configuration the benchmark uses (19 chunks), plus a ragged multi-sequence batch.
Tolerance (float32 accumulation against float64): per sampled row |err| <= 1e-5 |h| |w|,
relative L2 <= 2e-5 over a whole matrix; attention relative L2 <= 1e-4.
"""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def rel_l2(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def packed(B, key, rows, cols):
    q, s = synth.q8(key, rows, cols)
    qb, sb = B.stage_op_q8_device_bytes(rows, cols)
    qd = torch.empty(qb, dtype=torch.uint8, device="cuda")
    sd = torch.empty(sb, dtype=torch.uint8, device="cuda")
    B.stage_op_q8_pack(synth.Q8(q, s), qd, sd)
    return qd, sd


@pytest.mark.parametrize("name,rows,cols,ntok,norm", [
    ("qkv", 6144, 4096, 1, True),
    ("gate", 14336, 4096, 1, True),
    ("down", 4096, 14336, 1, False),
    ("head", 32000, 4096, 1, False),
    ("ragged", 1000, 688, 1, False),
    ("ragged-multi", 1001, 688, 3, True),
    ("multi", 4096, 4096, 5, False),
])
def test_gemv_sampled_rows_match_oracle(cuda, name, rows, cols, ntok, norm):
    from layer_range_stage_gb300 import binding as B
    key = synth.key(77, rows, cols)
    qd, sd = packed(B, key, rows, cols)
    x = np.stack([synth.normal_f32(synth.key(78, t, cols), 0, cols, 1.0) for t in range(ntok)])
    gamma = synth.normal_f32(synth.key(79, cols), 0, cols, 0.1, 1.0) if norm else None
    xd = torch.from_numpy(x).cuda()
    yd = torch.empty((ntok, rows), dtype=torch.float32, device="cuda")
    B.stage_op_gemv(qd, sd, rows, cols, xd, yd, None if gamma is None else torch.from_numpy(gamma).cuda(), 1e-5)
    torch.cuda.synchronize()
    y = yd.cpu().numpy()
    rng = np.random.default_rng(rows + cols)
    sample = np.unique(np.concatenate([[0, 1, rows - 2, rows - 1], rng.integers(0, rows, 60)]))
    h = oracle.rmsnorm(x.astype(np.float64), gamma, 1e-5) if norm else x.astype(np.float64)
    for r in sample:
        q, s = synth.q8(key, rows, cols, row0=int(r), nrows=1, n_threads=1)
        w = oracle.dequant(q, s)[0]
        # float32 accumulation error scales with |h| |w| (a row's sum may cancel to ~0)
        err = np.abs(y[:, r] - h @ w)
        assert (err <= 1e-5 * np.linalg.norm(h, axis=1) * np.linalg.norm(w)).all(), (name, r, err)


def test_gemv_vector_error_budget(cuda):
    """Over all rows of one full-size matrix the float32 result stays within 2e-5 of the
    float64 one (relative L2)."""
    from layer_range_stage_gb300 import binding as B
    rows, cols = 4096, 4096
    key = synth.key(80, rows, cols)
    qd, sd = packed(B, key, rows, cols)
    q, s = synth.q8(key, rows, cols)
    x = synth.normal_f32(synth.key(81), 0, cols, 1.0)[None, :]
    yd = torch.empty((1, rows), dtype=torch.float32, device="cuda")
    B.stage_op_gemv(qd, sd, rows, cols, torch.from_numpy(x).cuda(), yd)
    torch.cuda.synchronize()
    ref = oracle.matvec(oracle.dequant(q, s), x.astype(np.float64))
    assert rel_l2(yd.cpu().numpy(), ref) <= 2e-5


def kv_inputs(seqs, hkv, max_len, d, hq, n_tok, tag):
    k = synth.normal_f32(synth.key(90, tag, 0), 0, seqs * hkv * max_len * d, 1.0).reshape(seqs, hkv, max_len, d)
    v = synth.normal_f32(synth.key(90, tag, 1), 0, seqs * hkv * max_len * d, 1.0).reshape(seqs, hkv, max_len, d)
    q = synth.normal_f32(synth.key(90, tag, 2), 0, n_tok * hq * d, 1.0).reshape(n_tok, hq, d)
    return q, k.astype(np.float16), v.astype(np.float16)


def run_attention(B, q, k, v, seq, pos, n_chunks):
    n_tok, hq, d = q.shape
    hkv = k.shape[1]
    qd = torch.from_numpy(q).cuda()
    kd = torch.from_numpy(k).cuda()
    vd = torch.from_numpy(v).cuda()
    sd = torch.tensor(seq, dtype=torch.int32, device="cuda")
    pd = torch.tensor(pos, dtype=torch.int32, device="cuda")
    out = torch.empty_like(qd)
    nb = B.stage_op_attention_workspace_bytes(n_tok, hq, hkv, d, n_chunks)
    ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
    B.stage_op_attention_decode(qd, kd, vd, sd, pd, out, n_chunks, ws)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("n_chunks", [19, 1, 64])
def test_attention_context_2048_all_heads(cuda, n_chunks):
    from layer_range_stage_gb300 import binding as B
    m = synth.CONFIGS[1]
    q, k, v = kv_inputs(1, m.n_kv_heads, 2112, m.head_dim, m.n_q_heads, 1, 1)
    got = run_attention(B, q, k, v, [0], [2047], n_chunks)
    ref = oracle.attention(q.astype(np.float64), k, v, np.array([0]), np.array([2047]), m.n_kv_heads)
    assert rel_l2(got, ref) <= 1e-4


def test_attention_ragged_batch_gqa8(cuda):
    from layer_range_stage_gb300 import binding as B
    hq, hkv, d = 32, 4, 128                       # the MoE model's 8-way grouping
    seq, pos = [0, 1, 2, 1], [5, 130, 2047, 700]
    q, k, v = kv_inputs(3, hkv, 2100, d, hq, 4, 2)
    got = run_attention(B, q, k, v, seq, pos, 3)
    ref = oracle.attention(q.astype(np.float64), k, v, np.array(seq), np.array(pos), hkv)
    assert rel_l2(got, ref) <= 1e-4
    # first position only: the output is that row's V
    got1 = run_attention(B, q[:1], k, v, [2], [0], 4)
    assert np.allclose(got1[0, 0], v[2, 0, 0].astype(np.float32), rtol=1e-6, atol=1e-6)
