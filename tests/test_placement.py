"""The placement planner (stage_plan_placement): contiguous block ranges, at least one block per
stage, every stage within its own device's budget ("RFC: pipeline placement across multiple
GPUs ...", section "Heterogeneous GPUs": required(stage_i) <= usable_budget(device_i) for
every device independently, never the summed memory), balancing resident bytes
("Multi-node layer splitting and tensor parallelism", section on layer-split placement).

Pinned against brute force over every contiguous split on small models: the planner's
placement is legal, reports each stage's stage_required_bytes, and reaches the smallest
possible largest required/budget ratio; it reports DoesNotFit exactly when no split is legal.
Host code only: runs without a GPU."""
import itertools

import numpy as np
import pytest

import synth
import layer_range_stage_gb300 as L
from layer_range_stage_gb300 import build as lbuild


@pytest.fixture(scope="module", autouse=True)
def built():
    lbuild.build()


def cfg_of(model, **kw):
    d = dict(max_seqs=2, max_seq_len=512, max_tokens=64)
    d.update(kw)
    return L.make_cfg(model, **d)


def splits(n, s):
    """Every bounds list of s contiguous non-empty ranges over n blocks."""
    for cuts in itertools.combinations(range(1, n), s - 1):
        yield [0, *cuts, n]


def brute(cfg, n, budgets):
    """Smallest largest required/budget ratio over the legal splits (None if none is legal)."""
    best = None
    for b in splits(n, len(budgets)):
        req = [L.stage_required_bytes(cfg, b[k], b[k + 1]) for k in range(len(budgets))]
        if any(r > bud for r, bud in zip(req, budgets)):
            continue
        cost = max(r / bud for r, bud in zip(req, budgets))
        best = cost if best is None else min(best, cost)
    return best


MODELS = [
    synth.CONFIGS[0],                                           # 4 dense blocks
    synth.reduced(synth.CONFIGS[1], 7),                         # 7 blocks of the 8B shape
    synth.reduced(synth.CONFIGS[2], 6, n_experts=16, top_k=4),  # 6 MoE blocks
]


@pytest.mark.parametrize("mi", range(len(MODELS)))
def test_planner_matches_brute_force(mi):
    model = MODELS[mi]
    cfg = cfg_of(model)
    n = model.n_layers
    whole = L.stage_required_bytes(cfg, 0, n)
    rng = np.random.default_rng(600 + mi)
    for s in (1, 2, 3):
        if s > n:
            continue
        for _ in range(12):
            # budgets from a fraction of the whole model up to all of it: some legal, some not
            budgets = [int(whole * f) for f in rng.uniform(0.25, 1.05, s)]
            want = brute(cfg, n, budgets)
            if want is None:
                with pytest.raises(L.StageError) as e:
                    L.stage_plan_placement(cfg, budgets)
                assert e.value.code == L.STAGE_E_DOES_NOT_FIT
                continue
            bounds, req = L.stage_plan_placement(cfg, budgets)
            assert bounds[0] == 0 and bounds[-1] == n and len(bounds) == s + 1
            assert all(a < b for a, b in zip(bounds, bounds[1:]))      # contiguous, >= 1 block each
            for k in range(s):
                assert req[k] == L.stage_required_bytes(cfg, bounds[k], bounds[k + 1])
                assert req[k] <= budgets[k]                               # every device on its own
            got = max(r / b for r, b in zip(req, budgets))
            assert abs(got - want) <= 1e-12 * max(1.0, want)


def test_equal_budgets_balance_the_8b_shape():
    """Two equal devices: the 32 dense blocks split 16/16 (the embedding on the first stage
    and the readout on the last weigh the same; the last stage's logits workspace is smaller
    than a block)."""
    model = synth.CONFIGS[1]
    cfg = cfg_of(model, max_seqs=1, max_seq_len=2048 + 64, max_tokens=64)
    big = L.stage_required_bytes(cfg, 0, 32)
    bounds, req = L.stage_plan_placement(cfg, [big, big])
    assert bounds == [0, 16, 32]
    block = L.stage_required_bytes(cfg, 0, 17) - L.stage_required_bytes(cfg, 0, 16)
    assert abs(req[0] - req[1]) < block


def test_asymmetric_budgets_choose_an_asymmetric_split():
    """A 2:1 pair of budgets: the even split does not fit the smaller device, the planner
    finds the asymmetric split that does (the page's 24 GB + 12 GB case)."""
    model = synth.CONFIGS[1]
    cfg = cfg_of(model, max_seqs=1, max_seq_len=2048 + 64, max_tokens=64)
    whole = L.stage_required_bytes(cfg, 0, 32)
    budgets = [int(whole * 0.70), int(whole * 0.35)]
    assert L.stage_required_bytes(cfg, 16, 32) > budgets[1]          # 16/16 is illegal here
    bounds, req = L.stage_plan_placement(cfg, budgets)
    assert bounds[1] > 16 and req[0] <= budgets[0] and req[1] <= budgets[1]


def test_summed_memory_never_makes_a_placement_legal():
    """Budgets whose sum exceeds the whole model, but with no split fitting both devices."""
    model = synth.CONFIGS[1]
    cfg = cfg_of(model, max_seqs=1, max_seq_len=2048 + 64, max_tokens=64)
    whole = L.stage_required_bytes(cfg, 0, 32)
    smallest_last = min(L.stage_required_bytes(cfg, a, 32) for a in range(1, 32))
    budgets = [whole * 2, smallest_last - 1]                          # sum > whole model
    with pytest.raises(L.StageError) as e:
        L.stage_plan_placement(cfg, budgets)
    assert e.value.code == L.STAGE_E_DOES_NOT_FIT


def test_invalid_requests():
    cfg = cfg_of(synth.CONFIGS[0])
    for budgets in ([], [1 << 40] * 5):                               # 0 devices, more devices than blocks
        with pytest.raises(L.StageError) as e:
            L.stage_plan_placement(cfg, budgets)
        assert e.value.code == L.STAGE_E_INVALID
