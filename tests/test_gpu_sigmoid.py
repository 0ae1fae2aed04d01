"""Sigmoid router scoring on the GPU against the fp64 oracle, through the C ABI.

Colibri README, "What's implemented" (DeepSeek-V3-style sigmoid router,
noaux_tc, routed_scaling_factor), with the readings in
tests/golden/sigmoid_router.txt: the selection keys are sigmoid scores plus a
per-expert bias, the weights are the selected scores renormalised and scaled.
Every call that selects is covered: decode (split path), the allocation-free
decode, moe_route, a prefill chunk and a streamed layer.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import quantized_routed_expert_moe_gb300 as moe
import seeded_inputs as si
from _parity import compare_token

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from quantized_routed_expert_moe_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def sig(spec, scale=2.5, bias_sd=0.05, **kw):
    import dataclasses
    return dataclasses.replace(spec, router_score="sigmoid", routed_scaling=scale, score_bias_sd=bias_sd, **kw)


SHAPES = {
    "tiny_f32": sig(si.CONFIGS["tiny"]),
    "bf16_no_bias": sig(si.LayerSpec(hidden=512, inter=256, n_experts=64), scale=1.0, bias_sd=None),
    "q8_router_ragged": sig(si.LayerSpec(hidden=320, inter=128, n_experts=40, router_fmt="q8g64")),
    "top1": sig(si.LayerSpec(hidden=192, inter=64, n_experts=9, top_k=1, act="f32"), scale=1.5),
    "E1024_wide_bias": sig(si.LayerSpec(hidden=256, inter=256, n_experts=1024), bias_sd=0.3),
    "no_shared": sig(si.LayerSpec(hidden=128, inter=192, n_experts=16, top_k=4, n_shared=0)),
}


def to_dev(X, spec):
    if spec.act == "bf16":
        return torch.from_numpy(np.ascontiguousarray(X).view(np.int16)).cuda()
    return torch.from_numpy(np.ascontiguousarray(X, dtype=np.float32)).cuda()


def run_decode(ml, spec, X, static=False):
    T, H, k = len(X), spec.hidden, spec.top_k
    xd = to_dev(X, spec)
    yd = torch.bfloat16 if spec.act == "bf16" else torch.float32
    y = torch.empty((T, H), dtype=yd, device="cuda")
    y32 = torch.empty((T, H), dtype=torch.float32, device="cuda")
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    for t in range(T):
        if static:   # the static-scratch decode is checked against the selection of moe_route
            ml.decode_static_scratch(xd[t], y[t], y32[t])
            ml.route(xd[t], 1, ids[t], w[t])
        else:        # the selection moe_decode itself combined with
            ml.decode(xd[t], y[t], y32[t])
            ml.selection(1, ids[t], w[t])
    torch.cuda.synchronize()
    yb = y.view(torch.int16).cpu().numpy().view(np.uint16) if spec.act == "bf16" else None
    return y32.cpu().numpy(), ids.cpu().numpy(), w.cpu().numpy(), yb


def check_rows(layer, X, y32, ids, w, yb):
    Wr = oracle.router_weights_f64(layer.router)
    errs, flags = [], 0
    for t in range(len(X)):
        err, fl = compare_token(layer, X[t], y32[t], ids[t], w[t], Wr=Wr, y_bf16=None if yb is None else yb[t])
        errs.append(err)
        flags += fl
    return max(errs), flags


@pytest.mark.parametrize("name", list(SHAPES))
def test_sigmoid_decode_and_route(name):
    spec = SHAPES[name]
    layer = si.gen_layer(41, 0, spec)
    T = 12
    X = si.gen_tokens(41, 0, T, spec)
    with moe.MoELayer(layer, max_tokens=T) as ml:
        y32, ids, w, yb = run_decode(ml, spec, X)
        st, bits = ml.check()
        assert st == 0, hex(bits)
    assert np.allclose(w.sum(axis=1), spec.routed_scaling, rtol=0, atol=1e-5)
    err, flags = check_rows(layer, X, y32, ids, w, yb)
    print(f"{name}: max normwise err {err:.3e}, near-tie tokens {flags}")


def test_sigmoid_static_scratch_matches_decode():
    spec = SHAPES["tiny_f32"]
    layer = si.gen_layer(42, 0, spec)
    X = si.gen_tokens(42, 0, 6, spec)
    with moe.MoELayer(layer, max_tokens=6) as ml:
        a = run_decode(ml, spec, X)
        b = run_decode(ml, spec, X, static=True)
    assert np.array_equal(a[0], b[0])
    check_rows(layer, X, *b)


@pytest.mark.parametrize("name", ["tiny_f32", "q8_router_ragged", "E1024_wide_bias"])
def test_sigmoid_prefill_chunk(name):
    spec = SHAPES[name]
    layer = si.gen_layer(43, 0, spec)
    T = 40
    X = si.gen_tokens(43, 0, T, spec)
    xd = to_dev(X.reshape(-1), spec)
    yd = torch.bfloat16 if spec.act == "bf16" else torch.float32
    y = torch.empty(T * spec.hidden, dtype=yd, device="cuda")
    y32 = torch.empty(T * spec.hidden, dtype=torch.float32, device="cuda")
    ids = torch.empty(T * spec.top_k, dtype=torch.int32, device="cuda")
    w = torch.empty(T * spec.top_k, dtype=torch.float32, device="cuda")
    with moe.MoELayer(layer, max_tokens=T) as ml:
        ml.prefill_chunk(xd, T, y, y32)
        ml.selection(T, ids, w)   # the selection the chunk itself combined with
        torch.cuda.synchronize()
        st, bits = ml.check()
        assert st == 0, hex(bits)
    yb = y.view(torch.int16).cpu().numpy().view(np.uint16).reshape(T, -1) if spec.act == "bf16" else None
    err, flags = check_rows(layer, X, y32.cpu().numpy().reshape(T, -1), ids.cpu().numpy().reshape(T, -1),
                            w.cpu().numpy().reshape(T, -1), yb)
    print(f"prefill {name}: max normwise err {err:.3e}, near-tie tokens {flags}")


@pytest.mark.parametrize("device", [False, True])
def test_sigmoid_streamed_layer_bit_identical(device):
    """A streamed layer selects in the router kernel's last block: same output
    as the resident layer, bit for bit, with the cache managed on the host or
    on the device."""
    spec = sig(si.LayerSpec(hidden=256, inter=128, n_experts=32))
    layer = si.gen_layer(44, 0, spec)
    T = 10
    X = si.gen_tokens(44, 0, T, spec)
    with moe.MoELayer(layer, max_tokens=T) as res:
        y_res = run_decode(res, spec, X)[0]
        n = moe.moe_expert_record_bytes(res.desc)
        recs = []
        for ex in layer.experts:
            buf = np.zeros(n, np.uint8)
            moe.moe_pack_expert_record(res.desc, ex, buf)
            recs.append(buf)
    xd = to_dev(X, spec)
    y = torch.empty((T, spec.hidden), dtype=torch.bfloat16, device="cuda")
    y32 = torch.empty((T, spec.hidden), dtype=torch.float32, device="cuda")
    if device:
        recs = [pinned_copy(r) for r in recs]
    with moe.MoELayer(layer, cache_slots=16, records=recs) as st:
        if device:
            st.set_option(moe.MOE_OPT_CACHE_DEVICE, 1)
        for t in range(T):
            st.decode(xd[t], y[t], y32[t])
            torch.cuda.synchronize()
        assert st.check() == (0, 0)
    assert np.array_equal(y32.cpu().numpy(), y_res)


def pinned_copy(r):
    """A record in page-locked host memory (the device-managed cache reads it
    through its mapping)."""
    t = torch.empty(len(r), dtype=torch.uint8).pin_memory()
    t.numpy()[:] = r
    return t


def test_sigmoid_option_errors():
    spec = SHAPES["tiny_f32"]
    layer = si.gen_layer(45, 0, spec)
    with moe.MoELayer(layer) as ml:   # the binding set sigmoid scoring
        for bad in (0.0, -1.0, float("inf"), float("nan")):
            with pytest.raises(moe.MoEError) as ei:
                ml.set_router_scoring(moe.MOE_SCORE_SIGMOID, bad)
            assert ei.value.status == 1
        with pytest.raises(moe.MoEError) as ei:
            ml.set_router_scoring(7, 1.0)
        assert ei.value.status == 1
        # switching back and forth is allowed
        ml.set_router_scoring(moe.MOE_SCORE_SOFTMAX, 1.0)
        ml.set_router_scoring(moe.MOE_SCORE_SIGMOID, 2.5)
