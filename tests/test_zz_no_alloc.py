"""The attention entry point that allocates nothing, against the one that takes a workspace.

Some callers cannot allocate device memory when they run attention (their host owns all
device memory through its own allocator, or their loop must never call cudaMalloc), so
the library offers stage_op_attention_decode_static, whose scratch is a fixed array
inside the library.  This file is collected last on purpose: if it fails, a run that
stops at the first failure has already run every other test.
"""
import numpy as np
import pytest

import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu



def inputs(tag, seqs, hkv, max_len, d, hq, n_tok):
    k = synth.normal_f32(synth.key(95, tag, 0), 0, seqs * hkv * max_len * d, 1.0).reshape(seqs, hkv, max_len, d)
    v = synth.normal_f32(synth.key(95, tag, 1), 0, seqs * hkv * max_len * d, 1.0).reshape(seqs, hkv, max_len, d)
    q = synth.normal_f32(synth.key(95, tag, 2), 0, n_tok * hq * d, 1.0).reshape(n_tok, hq, d)
    return (torch.from_numpy(q).cuda(), torch.from_numpy(k.astype(np.float16)).cuda(),
            torch.from_numpy(v.astype(np.float16)).cuda())


def test_static_scratch_matches_workspace_entry_point_twice(cuda):
    from layer_range_stage_gb300 import binding as B
    cases = [  # (tag, seqs, hkv, max_len, d, hq, seq ids, positions, n_chunks)
        (1, 1, 8, 2112, 128, 32, [0], [2047], 19),          # 8B-shape decode step at context 2048
        (2, 3, 4, 700, 128, 32, [2, 0, 1], [699, 17, 310], 5),  # ragged batch, 8-way groups
    ]
    for tag, seqs, hkv, max_len, d, hq, seq, pos, n_chunks in cases:
        q, k, v = inputs(tag, seqs, hkv, max_len, d, hq, len(seq))
        sd = torch.tensor(seq, dtype=torch.int32, device="cuda")
        pd = torch.tensor(pos, dtype=torch.int32, device="cuda")
        ws = torch.zeros(B.stage_op_attention_workspace_bytes(len(seq), hq, hkv, d, n_chunks), dtype=torch.uint8,
                         device="cuda")
        ref = torch.empty_like(q)
        B.stage_op_attention_decode(q, k, v, sd, pd, ref, n_chunks, ws)
        want = ref.cpu().numpy().view(np.uint32)
        # the same kernel, chunking and merge order: equal bit for bit, on two calls in a row
        # (the second reuses the array the first left behind)
        for call in range(2):
            got = torch.full_like(q, float("nan"))
            B.stage_op_attention_decode_static(q, k, v, sd, pd, got, n_chunks)
            torch.cuda.synchronize()
            assert np.array_equal(got.cpu().numpy().view(np.uint32), want), (tag, call)


def test_static_scratch_rejects_oversized_requests(cuda):
    from layer_range_stage_gb300 import binding as B
    q, k, v = inputs(3, 1, 8, 256, 128, 64, 64)
    sd = torch.zeros(64, dtype=torch.int32, device="cuda")
    pd = torch.full((64,), 255, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    assert B.stage_op_attention_workspace_bytes(64, 64, 8, 128, 64) > 4 << 20
    with pytest.raises(B.StageError) as e:
        B.stage_op_attention_decode_static(q, k, v, sd, pd, out, 64)
    assert e.value.code == B.STAGE_E_INVALID and "static scratch" in str(e.value)
