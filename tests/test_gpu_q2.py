"""2-bit experts (affine group-64, codes 0..3) on the GPU against the fp64 oracle.

Inferno README ("Model": 2-bit routed experts) and Colibri README ("What's
implemented": packed int2, dequant-on-use), with the storage reading in
tests/golden/q2g64_dequant.txt. Decode, the allocation-free decode, a
streamed layer, prefill chunks through the grouped tcgen05 GEMM (resident and
streamed through the cache) are covered.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import quantized_routed_expert_moe_gb300 as moe
import seeded_inputs as si
from _parity import compare_chunk, compare_token

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from quantized_routed_expert_moe_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def q2(spec):
    return dataclasses.replace(spec, expert_bits=2)


SHAPES = {
    "tiny_f32": q2(si.CONFIGS["tiny"]),
    "bf16_mid": q2(si.LayerSpec(hidden=512, inter=320, n_experts=64, zipf_alpha=1.1)),
    "q8_router_ragged": q2(si.LayerSpec(hidden=320, inter=128, n_experts=40, router_fmt="q8g64")),
    "top1": q2(si.LayerSpec(hidden=192, inter=64, n_experts=9, top_k=1, act="f32")),
    "E1024": q2(si.LayerSpec(hidden=256, inter=256, n_experts=1024)),
    "no_shared_wide": q2(si.LayerSpec(hidden=1088, inter=704, n_experts=24, top_k=6, n_shared=0)),
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
def test_q2_decode(name):
    spec = SHAPES[name]
    layer = si.gen_layer(51, 0, spec)
    X = si.gen_tokens(51, 0, 10, spec)
    with moe.MoELayer(layer) as ml:
        y32, ids, w, yb = run_decode(ml, spec, X)
        st, bits = ml.check()
        assert st == 0, hex(bits)
    err, flags = check_rows(layer, X, y32, ids, w, yb)
    print(f"{name}: max normwise err {err:.3e}, near-tie tokens {flags}")


def test_q2_static_scratch_and_reproducible():
    spec = SHAPES["bf16_mid"]
    layer = si.gen_layer(52, 0, spec)
    X = si.gen_tokens(52, 0, 6, spec)
    with moe.MoELayer(layer) as ml:
        a = run_decode(ml, spec, X)
        b = run_decode(ml, spec, X)
        c = run_decode(ml, spec, X, static=True)
    assert np.array_equal(a[0], b[0])
    check_rows(layer, X, *c)


@pytest.mark.parametrize("device", [False, True])
def test_q2_streamed_layer_bit_identical(device):
    spec = q2(si.LayerSpec(hidden=256, inter=128, n_experts=32, zipf_alpha=1.1))
    layer = si.gen_layer(53, 0, spec)
    X = si.gen_tokens(53, 0, 12, spec)
    with moe.MoELayer(layer) as res:
        want = run_decode(res, spec, X)[0]
        n = moe.moe_expert_record_bytes(res.desc)
        recs = []
        for ex in layer.experts:
            buf = np.zeros(n, np.uint8)
            moe.moe_pack_expert_record(res.desc, ex, buf)
            recs.append(buf)
    xd = to_dev(X, spec)
    y32 = torch.empty((len(X), spec.hidden), dtype=torch.float32, device="cuda")
    if device:   # the device-managed cache reads page-locked records through their mapping
        pinned = []
        for r in recs:
            t_ = torch.empty(len(r), dtype=torch.uint8).pin_memory()
            t_.numpy()[:] = r
            pinned.append(t_)
        recs = pinned
    with moe.MoELayer(layer, cache_slots=16, records=recs) as st:
        if device:
            st.set_option(moe.MOE_OPT_CACHE_DEVICE, 1)
        for t in range(len(X)):
            st.decode(xd[t], None, y32[t])
            torch.cuda.synchronize()
        assert st.check() == (0, 0)
    assert np.array_equal(y32.cpu().numpy(), want)


PREFILL = {
    # name: (spec, T) -- ragged K blocks (H = 320: 5 chunks of 64, I = 192: 3),
    # small and full groups, no shared expert, an 8-bit router
    "tiny_f32_T16": (q2(si.CONFIGS["tiny"]), 16),
    "bf16_T128_zipf": (q2(si.LayerSpec(hidden=512, inter=256, n_experts=64, zipf_alpha=1.1)), 128),
    "ragged_T33": (q2(si.LayerSpec(hidden=320, inter=192, n_experts=24, top_k=6)), 33),
    "no_shared_T7": (q2(si.LayerSpec(hidden=256, inter=128, n_experts=16, top_k=4, n_shared=0)), 7),
    "q8_router_T64": (q2(si.LayerSpec(hidden=1088, inter=704, n_experts=40, router_fmt="q8g64")), 64),
}


def run_prefill(ml, spec, X, T):
    xd = to_dev(X.reshape(-1), spec)
    yd = torch.bfloat16 if spec.act == "bf16" else torch.float32
    y = torch.empty(T * spec.hidden, dtype=yd, device="cuda")
    y32 = torch.empty(T * spec.hidden, dtype=torch.float32, device="cuda")
    ids = torch.empty(T * spec.top_k, dtype=torch.int32, device="cuda")
    w = torch.empty(T * spec.top_k, dtype=torch.float32, device="cuda")
    ml.prefill_chunk(xd, T, y, y32)
    ml.selection(T, ids, w)   # the selection the chunk itself combined with
    torch.cuda.synchronize()
    st, bits = ml.check()
    assert st == 0, hex(bits)
    yb = y.view(torch.int16).cpu().numpy().view(np.uint16).reshape(T, -1) if spec.act == "bf16" else None
    return (y32.cpu().numpy().reshape(T, -1), ids.cpu().numpy().reshape(T, -1), w.cpu().numpy().reshape(T, -1), yb)


@pytest.mark.parametrize("name", list(PREFILL))
def test_q2_prefill_chunk(name):
    """2-bit experts in the grouped tcgen05 GEMM: every row against the oracle."""
    spec, T = PREFILL[name]
    layer = si.gen_layer(55, 0, spec)
    X = si.gen_tokens(55, 0, T, spec)
    with moe.MoELayer(layer, max_tokens=T) as ml:
        y32, ids, w, yb = run_prefill(ml, spec, X, T)
    err, flags = compare_chunk(layer, X, y32, ids, w, y_bf16=yb)
    print(f"q2 prefill {name}: max normwise err {err:.3e}, near-tie tokens {flags}")


def test_q2_prefill_dense_groups():
    """Every token on the same experts: full 128-row tiles through the 2-bit dequantiser."""
    spec = q2(si.LayerSpec(hidden=1024, inter=512, n_experts=32))
    layer = si.gen_layer(56, 0, spec)
    bias = np.full(32, -30.0, np.float32)
    bias[:8] = 30.0
    layer = dataclasses.replace(layer, router_bias=bias)
    T = 128
    X = si.gen_tokens(56, 0, T, spec)
    with moe.MoELayer(layer, max_tokens=T) as ml:
        y32, ids, w, yb = run_prefill(ml, spec, X, T)
    assert np.all(np.sort(ids, axis=1) == np.arange(8)[None, :])
    err, _ = compare_chunk(layer, X, y32, ids, w, y_bf16=yb)
    print(f"q2 prefill dense: max normwise err {err:.3e}")


def test_q2_streamed_prefill_bit_identical():
    """A 2-bit chunk through a streamed 16-slot layer (staging waves) equals the
    resident layer's chunk bit for bit."""
    spec = q2(si.LayerSpec(hidden=512, inter=256, n_experts=64, zipf_alpha=1.1))
    layer = si.gen_layer(57, 0, spec)
    T = 48
    X = si.gen_tokens(57, 0, T, spec)
    with moe.MoELayer(layer, max_tokens=T) as res:
        want = run_prefill(res, spec, X, T)
        n = moe.moe_expert_record_bytes(res.desc)
        recs = []
        for ex in layer.experts:
            buf = np.zeros(n, np.uint8)
            moe.moe_pack_expert_record(res.desc, ex, buf)
            recs.append(buf)
    with moe.MoELayer(layer, max_tokens=T, cache_slots=16, records=recs) as st:
        got = run_prefill(st, spec, X, T)
    assert np.array_equal(got[0], want[0])
    assert np.array_equal(got[1], want[1])
