"""Prefill chunk on the GPU against the fp64 oracle (parity), through the C ABI.

Every row of a prefill chunk must equal the oracle's layer output for that
token within the normwise tolerance, with the expert IDs of that token exact
(near-ties handled as in the decode tests), and the bf16 output must be the
round-to-nearest-even of the fp32 output. The IDs and weights checked are the
ones the chunk itself computed and combined with (moe_layer_selection).
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import quantized_routed_expert_moe_gb300 as moe
import seeded_inputs as si
from _parity import compare_chunk

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from quantized_routed_expert_moe_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def to_dev(X, spec):
    if spec.act == "bf16":
        return torch.from_numpy(np.ascontiguousarray(X).view(np.int16)).cuda()
    return torch.from_numpy(np.ascontiguousarray(X, dtype=np.float32)).cuda()


def run_prefill(ml, spec, X, T):
    H, k = spec.hidden, spec.top_k
    x = to_dev(X.reshape(-1), spec)
    yd = torch.bfloat16 if spec.act == "bf16" else torch.float32
    y = torch.empty(T * H, dtype=yd, device="cuda")
    y32 = torch.empty(T * H, dtype=torch.float32, device="cuda")
    ids = torch.empty(T * k, dtype=torch.int32, device="cuda")
    w = torch.empty(T * k, dtype=torch.float32, device="cuda")
    ml.prefill_chunk(x, T, y, y32)
    ml.selection(T, ids, w)
    torch.cuda.synchronize()
    st, bits = ml.check()
    assert st == 0, hex(bits)
    yb = y.view(torch.int16).cpu().numpy().view(np.uint16).reshape(T, H) if spec.act == "bf16" else None
    return (y32.cpu().numpy().reshape(T, H), ids.cpu().numpy().reshape(T, k), w.cpu().numpy().reshape(T, k), yb)


def check_rows(layer, X, y32, ids, w, yb):
    """Every row of the chunk against the oracle."""
    return compare_chunk(layer, X, y32, ids, w, y_bf16=yb)


SHAPES = {
    # name: (spec, T)
    "tiny_f32_T16": (si.CONFIGS["tiny"], 16),
    "bf16_T128_zipf": (si.LayerSpec(hidden=512, inter=256, n_experts=64, zipf_alpha=1.1), 128),
    "ragged_down_tile_T33": (si.LayerSpec(hidden=320, inter=192, n_experts=24, top_k=6), 33),
    "no_shared_T7": (si.LayerSpec(hidden=256, inter=128, n_experts=16, top_k=4, n_shared=0), 7),
    "top1_T50": (si.LayerSpec(hidden=192, inter=64, n_experts=9, top_k=1, act="f32"), 50),
    "k_equals_E_T2": (si.LayerSpec(hidden=128, inter=64, n_experts=8, top_k=8), 2),
    "E1024_T128": (si.LayerSpec(hidden=256, inter=128, n_experts=1024), 128),
    "q8_router_T64": (si.LayerSpec(hidden=1088, inter=704, n_experts=40, router_fmt="q8g64"), 64),
}


@pytest.mark.parametrize("name", list(SHAPES))
def test_prefill_shapes(name):
    spec, T = SHAPES[name]
    layer = si.gen_layer(21, 0, spec)
    X = si.gen_tokens(21, 0, T, spec)
    with moe.MoELayer(layer, max_tokens=T) as ml:
        y32, ids, w, yb = run_prefill(ml, spec, X, T)
    err, flags = check_rows(layer, X, y32, ids, w, yb)
    print(f"{name}: max normwise err {err:.3e}, near-tie tokens {flags}")


# Activations far from unit scale and with outlier channels: the chunk stages
# each token as x * 2^a in binary16 and each SwiGLU output row as h * 2^z, so
# large tokens do not overflow binary16 (65504) and tiny ones do not flush.
RANGE_CASES = {
    "outliers_x1000": lambda spec, T: si.gen_tokens_outliers(61, 0, T, spec, 1000.0),
    "tiny_1e-20": lambda spec, T: si.gen_tokens_scaled(62, 0, T, spec, 1e-20),
    "large_1e4": lambda spec, T: si.gen_tokens_scaled(63, 0, T, spec, 1e4),
    "large_1e5": lambda spec, T: si.gen_tokens_scaled(64, 0, T, spec, 1e5),
}


@pytest.mark.parametrize("case", list(RANGE_CASES))
@pytest.mark.parametrize("act", ["bf16", "f32"])
def test_prefill_dynamic_range(case, act):
    spec = si.LayerSpec(hidden=1024, inter=512, n_experts=32, act=act, zipf_alpha=1.1)
    layer = si.gen_layer(60, 0, spec)
    T = 40
    X = RANGE_CASES[case](spec, T)
    with moe.MoELayer(layer, max_tokens=T) as ml:
        y32, ids, w, yb = run_prefill(ml, spec, X, T)
    assert np.all(np.isfinite(y32))
    err, flags = check_rows(layer, X, y32, ids, w, yb)
    print(f"{case}/{act}: max normwise err {err:.3e}, near-tie tokens {flags}")


def test_prefill_matches_decode_rows():
    """Row t of a chunk equals decode of token t within tolerance (the chunk is an
    execution strategy, not a different function)."""
    spec = si.LayerSpec(hidden=512, inter=256, n_experts=32)
    layer = si.gen_layer(5, 0, spec)
    T = 24
    X = si.gen_tokens(5, 0, T, spec)
    with moe.MoELayer(layer, max_tokens=T) as ml:
        y32, _, _, _ = run_prefill(ml, spec, X, T)
        x = to_dev(X, spec)
        yd = torch.empty((T, spec.hidden), dtype=torch.float32, device="cuda")
        for t in range(T):
            ml.decode(x[t], None, yd[t])
        torch.cuda.synchronize()
    yd = yd.cpu().numpy().astype(np.float64)
    for t in range(T):
        err = np.max(np.abs(y32[t] - yd[t])) / np.max(np.abs(yd[t]))
        assert err <= 2e-3, (t, err)


def test_prefill_bit_reproducible():
    spec = si.LayerSpec(hidden=512, inter=256, n_experts=32, zipf_alpha=1.1)
    layer = si.gen_layer(6, 0, spec)
    T = 64
    X = si.gen_tokens(6, 0, T, spec)
    with moe.MoELayer(layer, max_tokens=T) as ml:
        a = run_prefill(ml, spec, X, T)[0]
        b = run_prefill(ml, spec, X, T)[0]
    assert np.array_equal(a, b)


def test_prefill_zero_input_exact():
    spec = si.LayerSpec(hidden=256, inter=128, n_experts=16)
    layer = si.gen_layer(3, 0, spec)
    T = 9
    X = np.zeros((T, 256), np.uint16)
    with moe.MoELayer(layer, max_tokens=T) as ml:
        y32, ids, w, _ = run_prefill(ml, spec, X, T)
    assert np.all(ids == np.arange(8)[None, :])
    assert np.all(w == np.float32(0.125))
    assert np.all(y32 == 0)


def dense_bias_layer(layer, experts):
    """The same layer with a router bias that sends every token to `experts`
    (the 'all tokens on the same experts' prefill case)."""
    E = layer.spec.n_experts
    bias = np.full(E, -30.0, np.float32)
    bias[list(experts)] = 30.0
    return dataclasses.replace(layer, router_bias=bias)


@pytest.fixture(scope="module")
def glm_layer():
    return si.gen_layer(0, 0, si.CONFIGS["glm_prefill"])


def test_glm_prefill_chunk(glm_layer):
    """Full-size chunk (GLM shape, 128 tokens, Zipf(1.1) bias) in the launch
    configuration the benchmark times; all 128 rows against the oracle."""
    spec = glm_layer.spec
    T = 128
    X = si.gen_tokens(3, 0, T, spec)
    with moe.MoELayer(glm_layer, max_tokens=T) as ml:
        y32, ids, w, yb = run_prefill(ml, spec, X, T)
    assert np.all(np.isfinite(y32))
    err, flags = check_rows(glm_layer, X, y32, ids, w, yb)
    print(f"glm prefill: max normwise err {err:.3e} over 128 rows, near-tie tokens {flags}")


def test_glm_prefill_dense_groups(glm_layer):
    """All 128 tokens on the same 8 experts: 9 groups of 128 rows (full MMA tiles)."""
    layer = dense_bias_layer(glm_layer, range(8))
    spec = layer.spec
    T = 128
    X = si.gen_tokens(4, 0, T, spec)
    with moe.MoELayer(layer, max_tokens=T) as ml:
        y32, ids, w, yb = run_prefill(ml, spec, X, T)
    assert np.all(np.sort(ids, axis=1) == np.arange(8)[None, :])
    err, flags = check_rows(layer, X, y32, ids, w, yb)
    print(f"glm prefill dense: max normwise err {err:.3e} over 128 rows")
