"""Chain of stages on one GPU and one stream, built block by block.

Each stage is created for its block range and then imports only its own tensors, one
block at a time, so host memory never holds more than one block ("RFC: pipeline
placement across multiple GPUs for models larger than one device", section
"Larger-than-single-card proof": weights go straight to their stage; the full model is
never materialised in one place).  All arithmetic happens in libstage.so.
"""
from __future__ import annotations

from typing import Callable, List, Optional, Sequence

import numpy as np

from . import binding as B


class StagePipeline:
    """Stages over the block ranges ``bounds`` (e.g. [0, 16, 32]) of one model.

    layer_weights(l) -> an object with the fields of stage_layer_w for block l.
    endpoint_weights(begin, end) -> an object with embed / final_norm / lm_head (None
    where the stage does not own them)."""

    def __init__(self, model, bounds: Sequence[int], layer_weights: Callable, endpoint_weights: Callable,
                 max_seqs: int = 1, max_seq_len: int = 256, max_tokens: int = 64, gemm_bf16_min_tokens: int = 0,
                 stream=None, budget: Optional[int] = None):
        if list(bounds) != sorted(set(bounds)) or bounds[0] != 0 or bounds[-1] != model.n_layers:
            raise ValueError("bounds must increase from 0 to n_layers")
        self.model = model
        self.bounds = list(bounds)
        self.cfg = B.make_cfg(model, max_seqs, max_seq_len, max_tokens, gemm_bf16_min_tokens)
        self.stages: List[int] = []
        self.handle = None
        try:
            for a, b in zip(bounds, bounds[1:]):
                st = B.stage_create(self.cfg, a, b, None, budget, stream)
                self.stages.append(st)
                if a == 0 or b == model.n_layers:
                    B.stage_load_endpoints(st, endpoint_weights(a, b))
                for l in range(a, b):
                    B.stage_load_layer(st, l, layer_weights(l))
            self.handle = B.stage_pipeline_create(self.stages)
        except Exception:
            self.close()
            raise

    # one step of all stages (+ readout of `rows` of the last stage)
    def step(self, is_prefill: bool, seq_ids, positions, tokens, rows=(), logits_out=None, want_tokens=True):
        return B.stage_pipeline_step(self.handle, is_prefill, seq_ids, positions, tokens, rows, logits_out, want_tokens)

    def generate(self, seq_ids, first_tokens, n_steps: int, use_graph: bool = True) -> np.ndarray:
        return B.stage_pipeline_generate(self.handle, seq_ids, first_tokens, n_steps, use_graph)

    def kernel_timing(self, enable: bool) -> None:
        B.stage_pipeline_kernel_timing(self.handle, enable)

    def kernel_time(self):
        return B.stage_pipeline_kernel_time(self.handle)

    def handoff_stats(self, boundary: int):
        return B.stage_pipeline_handoff_stats(self.handle, boundary)

    def committed(self, seq_id: int) -> List[int]:
        return [B.stage_committed_len(st, seq_id) for st in self.stages]

    def close(self) -> None:
        if self.handle is not None:
            B.stage_pipeline_destroy(self.handle)
            self.handle = None
        for st in self.stages:
            B.stage_destroy(st)
        self.stages = []

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
