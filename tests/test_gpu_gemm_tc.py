"""The tcgen05 prefill GEMM through the C ABI against the oracle's bf16 arithmetic:
A rounded to bf16, W = bf16(f32(scale) * q), products accumulated (float64 in the oracle,
float32 in TMEM).  Tolerance from the arithmetic: the float32 accumulation of K products
has a relative error ~ 2^-24 sqrt(K) times a small constant, so relative L2 <= 5e-7 sqrt(K)
(3.2e-5 at K = 4096, 6e-5 at K = 14336).  Ragged M and N, padded K, and the full prefill
shape on sampled rows."""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def rel_l2(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def bf16_bits(x):
    """float32 -> bf16 bit patterns, round to nearest even (the operand rounding)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return (((u + 0x7FFF + ((u >> 16) & 1)) >> 16) & 0xFFFF).astype(np.uint16)


def run(M, N, K, sample_rows=None, tag=0):
    from layer_range_stage_gb300 import binding as B
    key = synth.key(61, M, N, K, tag)
    q, s = synth.q8(key, N, K)
    qb, sb = B.stage_op_q8_device_bytes(N, K)
    qd = torch.empty(qb, dtype=torch.uint8, device="cuda")
    sd = torch.empty(sb, dtype=torch.uint8, device="cuda")
    B.stage_op_q8_pack(synth.Q8(q, s), qd, sd)
    kp = (K + 255) // 256 * 256
    x = synth.normal_f32(synth.key(62, M, K, tag), 0, M * K, 1.0).reshape(M, K)
    abits = np.zeros((M, kp), np.uint16)
    abits[:, :K] = bf16_bits(x)
    ad = torch.from_numpy(abits.view(np.int16)).cuda()
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    B.stage_op_gemm_bf16(ad, qd, sd, N, K, y)
    torch.cuda.synchronize()
    got = y.cpu().numpy()
    a64 = oracle.bf16(x)
    rows = np.arange(N) if sample_rows is None else sample_rows
    w64 = oracle.bf16(oracle.dequant(q[rows], s[rows]))
    ref = a64 @ w64.T
    return got[:, rows], ref


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (300, 520, 4096), (37, 1000, 688), (512, 768, 14336)])
def test_gemm_matches_oracle_bf16(cuda, M, N, K):
    got, ref = run(M, N, K)
    assert np.isfinite(got).all()
    assert rel_l2(got, ref) <= 5e-7 * np.sqrt(K)


def test_gemm_prefill_qkv_shape_sampled_rows(cuda):
    rows = np.unique(np.concatenate([[0, 255, 256, 6143], np.random.default_rng(3).integers(0, 6144, 40)]))
    got, ref = run(2048, 6144, 4096, sample_rows=rows, tag=1)
    assert rel_l2(got, ref) <= 5e-7 * np.sqrt(4096)
