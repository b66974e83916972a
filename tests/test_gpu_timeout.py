"""A device-side wait that runs out, on purpose, and the call after it.

Every wait of the persistent decode is bounded (0.2 s); a wait that runs out sets the stage's
error word, the kernel waits (bounded) for its own copies in flight and every CTA leaves.
stage_debug_inject(st, 3, 1) makes the next single-token decode launch of a stage wait for a
tag that no step writes, so its attention waits run out -- nothing faults, traps or hangs.
The step must fail with STAGE_E_CUDA and publish nothing ("RFC: pipeline placement across
multiple GPUs for models larger than one device", section "What I found": a step succeeds or
fails as a whole), and the same step run again must match the oracle.
"""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

LOGIT_ATOL = 2e-2


@pytest.mark.parametrize("stalled_stage", [0, 1])
def test_timed_out_wait_fails_the_step_and_the_retry_matches_the_oracle(cuda, stalled_stage):
    from layer_range_stage_gb300 import binding as B
    from layer_range_stage_gb300.pipeline import StagePipeline
    model = synth.CONFIGS[0]
    bounds = [0, 2, 4]
    prompt = synth.prompt_tokens(model, 6, 20)
    n = len(prompt)
    op = oracle.Pipeline([oracle.Stage(model, a, b, synth.stage_weights(model, a, b), max_len=64)
                          for a, b in zip(bounds, bounds[1:])])
    toks_o, logits_o = op.generate([prompt], 3)
    with StagePipeline(model, bounds, lambda l: synth.layer_weights(model, l),
                       lambda a, b: synth.stage_weights(model, a, b, with_layers=False),
                       max_seq_len=64, max_tokens=32) as gp:
        assert B.stage_gemm_mode(gp.stages[stalled_stage], 1) == 2
        lg = torch.empty((1, model.vocab), dtype=torch.float32, device="cuda")
        tok = int(gp.step(True, np.zeros(n), np.arange(n), prompt, rows=[n - 1], logits_out=lg)[0])
        assert tok == toks_o[0][0]
        B.stage_debug_inject(gp.stages[stalled_stage], 3, 1)
        with pytest.raises(B.StageError) as e:
            gp.step(False, [0], [n], [tok], rows=[0], logits_out=lg)
        assert e.value.code == B.STAGE_E_CUDA
        assert gp.committed(0) == [n, n]  # nothing published
        got = []
        for t in range(2):  # the same step again, then one more
            nxt = int(gp.step(False, [0], [n + t], [tok], rows=[0], logits_out=lg)[0])
            assert np.abs(lg.cpu().numpy() - logits_o[t + 1]).max() <= LOGIT_ATOL, t
            got.append(nxt)
            tok = nxt
        assert got == list(toks_o[0][1:3])
