"""The C-ABI library loads, exports every declared symbol, and its host-side checks work
without a GPU (config validation, the device-budget fit rule, the byte plan)."""
import ctypes
import json
import os
import subprocess

import pytest

import synth
import layer_range_stage_gb300 as L
from layer_range_stage_gb300 import build as lbuild

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def built():
    lbuild.build()


def test_library_exports_every_declared_symbol():
    declared = L.declared_symbols()
    assert len(declared) >= 20
    out = subprocess.run(["nm", "-D", "--defined-only", lbuild.LIB], capture_output=True, text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    assert set(declared) <= exported, set(declared) - exported
    lib = L.lib()
    for name in declared:
        assert getattr(lib, name) is not None


def cfg_of(model, **kw):
    d = dict(max_seqs=1, max_seq_len=256, max_tokens=64)
    d.update(kw)
    return L.make_cfg(model, **d)


def test_required_bytes_covers_weights_and_kv():
    m = synth.CONFIGS[1]
    c = cfg_of(m, max_seq_len=2048 + 64, max_tokens=64)
    per_layer_params = (m.q_dim + 2 * m.kv_dim) * m.hidden + m.hidden * m.q_dim + 3 * m.ffn * m.hidden
    total = 0
    for a, b in ((0, 16), (16, 32)):
        req = L.stage_required_bytes(c, a, b)
        params = per_layer_params * (b - a) + (m.vocab * m.hidden if a == 0 else 0) + \
            (m.vocab * m.hidden if b == m.n_layers else 0)
        kv = 2 * (b - a) * m.n_kv_heads * (2048 + 64) * m.head_dim * 2
        assert req >= params * 1.0625 + kv
        assert req <= params * 1.0625 + kv + (256 << 20)     # workspace stays small at batch 1
        total += req
    assert L.stage_required_bytes(c, 0, 32) < total          # the split adds only workspace


def test_invalid_configs_are_rejected_before_any_device_call():
    m = synth.CONFIGS[0]
    for kw in (dict(max_seqs=0), dict(max_tokens=0)):
        c = cfg_of(m, **kw)
        assert L.stage_required_bytes(c, 0, 4) == 0
        with pytest.raises(L.StageError) as e:
            L.stage_create(c, 0, 4, budget=1 << 40, stream=0)
        assert e.value.code == L.STAGE_E_INVALID
    c = cfg_of(m)
    for a, b in ((2, 2), (3, 2), (-1, 2), (0, 5)):
        assert L.stage_required_bytes(c, a, b) == 0
        with pytest.raises(L.StageError) as e:
            L.stage_create(c, a, b, budget=1 << 40, stream=0)
        assert e.value.code == L.STAGE_E_INVALID
    bad = synth.reduced(m, 4, n_kv_heads=3)
    with pytest.raises(L.StageError) as e:
        L.stage_create(cfg_of(bad), 0, 4, budget=1 << 40, stream=0)
    assert e.value.code == L.STAGE_E_INVALID


def test_does_not_fit_is_per_device_not_summed():
    """The RFC's rule: a placement is legal only if every stage fits its own device's
    budget; the summed budget never counts.  With the page's numbers the whole model
    (40.396 GB) fits neither 22.76 GB device while the two stage charges fit."""
    g = json.load(open(os.path.join(GOLDEN, "rfc_fit_budgets.json")))
    budgets = g["device_budgets"]
    assert [g["single_device_required"] <= b for b in budgets] == g["expected"]["single_device_fits"]
    assert all(st["total_charge"] <= budgets[st["device"]] for st in g["stages"]) == g["expected"]["placement_fits"]
    assert (g["single_device_required"] <= sum(budgets)) == g["expected"]["summed_vram_would_fit"]
    # the same rule through stage_create: each stage against its own budget, checked
    # before anything is allocated
    m = synth.CONFIGS[2]
    c = cfg_of(m, max_seq_len=4096 + 64)
    whole = L.stage_required_bytes(c, 0, 40)
    s0, s1 = L.stage_required_bytes(c, 0, 21), L.stage_required_bytes(c, 21, 40)
    budget = max(s0, s1)
    assert whole > budget and s0 <= budget and s1 <= budget
    with pytest.raises(L.StageError) as e:
        L.stage_create(c, 0, 40, budget=budget, stream=0)
    assert e.value.code == L.STAGE_E_DOES_NOT_FIT and "DoesNotFit" in str(e.value)
    with pytest.raises(L.StageError) as e:
        L.stage_create(c, 0, 21, budget=s0 - 1, stream=0)
    assert e.value.code == L.STAGE_E_DOES_NOT_FIT


def test_error_codes_of_the_header_and_the_binding_agree():
    import re
    text = open(os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "stage.h")).read()
    codes = {name: int(val) for name, val in re.findall(r"\b(STAGE_(?:OK|E_[A-Z_]+))\s*=\s*(-?\d+)", text)}
    assert codes["STAGE_OK"] == 0 and len(codes) >= 11
    for name, val in codes.items():
        assert getattr(L, name) == val, name
        assert L.binding.ERROR_NAMES[val] == name


def test_a_failed_host_allocation_returns_an_error_instead_of_escaping():
    """A staging buffer of 2^62 bytes cannot be mapped in any 48- to 56-bit virtual address
    space, so the allocation fails before any byte is touched; the entry point must return
    STAGE_E_HOST (no C++ exception crosses the C ABI) and the library keeps working."""
    lib = L.lib()
    q = (ctypes.c_int8 * 32)()
    s = (ctypes.c_uint16 * 1)()
    h = L.binding.stage_q8(ctypes.cast(q, ctypes.c_void_p), ctypes.cast(s, ctypes.c_void_p), 1 << 42, 1 << 20)
    qb, sb = L.stage_op_q8_device_bytes(1 << 42, 1 << 20)
    assert qb == 1 << 62
    rc = lib.stage_op_q8_pack(ctypes.byref(h), ctypes.c_void_p(16), ctypes.c_void_p(16))
    assert rc == L.STAGE_E_HOST
    assert lib.stage_op_last_error().decode().startswith("host:")
    assert L.stage_op_q8_device_bytes(64, 100) == (64 * 256, 64 * 8 * 2)


def test_layer_counts_beyond_the_limits_are_rejected_before_any_allocation():
    m = synth.CONFIGS[0]
    c = cfg_of(m)
    c.n_layers = (1 << 16) + 1
    assert L.stage_required_bytes(c, 0, 4) == 0
    c.n_layers = 5000  # a valid model, but beyond the planner's 4096 blocks
    assert L.stage_required_bytes(c, 0, 4) > 0
    with pytest.raises(L.StageError) as e:
        L.stage_plan_placement(c, [1 << 40, 1 << 40])
    assert e.value.code == L.STAGE_E_INVALID


def test_binding_has_every_entry_point_under_its_c_name():
    from layer_range_stage_gb300 import binding as B
    for name in L.declared_symbols():
        assert callable(getattr(B, name, None)), name
        assert name in B._SIGS, name
    assert B.stage_create_error() == "" or isinstance(B.stage_create_error(), str)
    assert isinstance(B.stage_op_last_error(), str)


def test_entry_points_reject_bad_arguments_before_any_device_call():
    """The host-side checks the headers document, on a machine without a GPU: every call below
    must fail with STAGE_E_INVALID and a message before touching the device."""
    lib = L.lib()
    v = ctypes.c_void_p
    buf = (ctypes.c_float * 64)()
    p = ctypes.cast(buf, v)                                # 16-byte aligned host memory
    odd = v(p.value + 4)                                   # not 16-byte aligned
    tok = (ctypes.c_int32 * 4)()
    cases = [
        lambda: lib.stage_op_embed(None, p, 10, 64, ctypes.cast(tok, v), 1, p, None),
        lambda: lib.stage_op_embed(p, p, 10, 66, ctypes.cast(tok, v), 1, p, None),       # cols % 4
        lambda: lib.stage_op_embed(p, p, 10, 64, ctypes.cast(tok, v), 70000, p, None),   # n_tok
        lambda: lib.stage_op_gemv(p, p, 8, 64, odd, 1, None, ctypes.c_float(1e-5), p, None),
        lambda: lib.stage_op_gemv(p, p, 0, 64, p, 1, None, ctypes.c_float(1e-5), p, None),
        lambda: lib.stage_op_gemm_bf16(p, 100, 4, p, p, 8, 64, p, None),                  # lda < 256
        lambda: lib.stage_op_attention_decode(p, p, p, p, p, 1, 4, 2, 96, 16, 1, p, p, 1 << 20, None),
        lambda: lib.stage_op_attention_decode(p, p, p, p, p, 1, 4, 2, 64, 16, 65, p, p, 1 << 20, None),
        lambda: lib.stage_op_attention_decode(p, p, p, p, p, 1, 4, 2, 64, 16, 1, p, p, 16, None),
        lambda: lib.stage_op_attention_decode_static(p, p, p, p, p, 1, 4, 3, 64, 16, 1, p, None),
    ]
    for i, call in enumerate(cases):
        assert call() == L.STAGE_E_INVALID, i
        assert lib.stage_op_last_error().decode(), i
    assert lib.stage_op_attention_workspace_bytes(0, 4, 2, 64, 1) == 0
    out = v()
    assert lib.stage_pipeline_create(None, 2, ctypes.byref(out)) == L.STAGE_E_INVALID
    null_stages = (v * 2)()
    assert lib.stage_pipeline_create(null_stages, 2, ctypes.byref(out)) == L.STAGE_E_INVALID
    n = ctypes.c_int()
    assert lib.stage_committed_len(None, 0, ctypes.byref(n)) == L.STAGE_E_INVALID
    assert lib.stage_gemm_mode(None, 1, ctypes.byref(n)) == L.STAGE_E_INVALID
    assert lib.stage_last_error(None).decode() == "null stage"
    assert lib.stage_pipeline_last_error(None).decode() == "null pipeline"
    lib.stage_destroy(None)
    lib.stage_pipeline_destroy(None)
