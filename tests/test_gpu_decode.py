"""Decode path on the GPU against the fp64 oracle (parity), through the C ABI.

The expert IDs and weights checked are the ones moe_decode itself used: the
selection its router kernel made, which its gate/up and down kernels read and
combined with (moe_layer_selection).
"""
import numpy as np
import pytest
import torch

import oracle
import quantized_routed_expert_moe_gb300 as moe
import seeded_inputs as si
from _parity import compare_token, f32_to_bf16_rne

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from quantized_routed_expert_moe_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def to_dev(x_np, spec):
    if spec.act == "bf16":
        return torch.from_numpy(np.ascontiguousarray(x_np).view(np.int16)).cuda()
    return torch.from_numpy(np.ascontiguousarray(x_np, dtype=np.float32)).cuda()


def decode_one(ml, spec, x_np, static=False):
    """One decode; returns (y32, ids, w, y_bf16 bits or None, y) with ids / w
    the selection the decode itself combined with."""
    H, k = spec.hidden, spec.top_k
    x = to_dev(x_np, spec)
    yd = torch.bfloat16 if spec.act == "bf16" else torch.float32
    y = torch.empty(H, dtype=yd, device="cuda")
    y32 = torch.empty(H, dtype=torch.float32, device="cuda")
    ids = torch.full((k,), -1, dtype=torch.int32, device="cuda")
    w = torch.full((k,), float("nan"), dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream()
    if static:
        ml.decode_static_scratch(x, y, y32, stream=s)
    else:
        ml.decode(x, y, y32, stream=s)
        ml.selection(1, ids, w, stream=s)
    torch.cuda.synchronize()
    yb = y.view(torch.int16).cpu().numpy().view(np.uint16) if spec.act == "bf16" else None
    return y32.cpu().numpy(), ids.cpu().numpy(), w.cpu().numpy(), yb, y


def check_layer(layer, tokens, seed=100, tokens_fn=None):
    spec = layer.spec
    Wr = oracle.router_weights_f64(layer.router)
    errs, flags = [], 0
    gen = tokens_fn or (lambda t: si.gen_tokens(seed, t, 1, spec)[0])
    with moe.MoELayer(layer) as ml:
        for t in range(tokens):
            x = gen(t)
            y32, ids, w, yb, _ = decode_one(ml, spec, x)
            err, flagged = compare_token(layer, x, y32, ids, w, Wr=Wr, y_bf16=yb)
            errs.append(err)
            flags += flagged
        st, bits = ml.check()
        assert st == 0, bits
    return max(errs), flags


def test_tiny_layer_decode():
    layer = si.gen_layer(0, 0, si.CONFIGS["tiny"])
    err, flags = check_layer(layer, 32)
    print(f"tiny: max normwise err {err:.3e}, near-tie tokens {flags}")


SHAPES = {
    "k_equals_E": si.LayerSpec(hidden=64, inter=64, n_experts=8, top_k=8, act="f32"),
    "no_shared_bf16": si.LayerSpec(hidden=128, inter=192, n_experts=16, top_k=4, n_shared=0),
    "q8_router_ragged": si.LayerSpec(hidden=320, inter=128, n_experts=40, router_fmt="q8g64"),
    "E1024": si.LayerSpec(hidden=256, inter=256, n_experts=1024),
    "top1": si.LayerSpec(hidden=192, inter=64, n_experts=9, top_k=1, act="f32"),
    "zipf_bias": si.LayerSpec(hidden=512, inter=320, n_experts=64, zipf_alpha=1.1),
    "ragged_lanes": si.LayerSpec(hidden=1088, inter=704, n_experts=24, top_k=6),
    # gate/up rows longer than one load block per lane (one pair per warp at a
    # time), with a ragged last block; down rows of two half-groups per lane
    "long_rows": si.LayerSpec(hidden=3136, inter=1088, n_experts=16, top_k=4),
}


@pytest.mark.parametrize("name", list(SHAPES))
def test_decode_shapes(name):
    layer = si.gen_layer(7, 1, SHAPES[name])
    err, flags = check_layer(layer, 6, seed=7)
    print(f"{name}: max normwise err {err:.3e}, near-tie tokens {flags}")


# Activations of very different magnitudes and with outlier channels: the
# decode stages them with a per-token power-of-two scale and 16-bit fixed point
# per run of 32 (an outlier sets the step of its 31 neighbours).
RANGE_CASES = {
    "outliers_x100": lambda spec, t: si.gen_tokens_outliers(31, t, 1, spec, 100.0)[0],
    "outliers_x1000": lambda spec, t: si.gen_tokens_outliers(32, t, 1, spec, 1000.0)[0],
    "tiny_1e-20": lambda spec, t: si.gen_tokens_scaled(33, t, 1, spec, 1e-20)[0],
    "large_1e4": lambda spec, t: si.gen_tokens_scaled(34, t, 1, spec, 1e4)[0],
    "large_1e5": lambda spec, t: si.gen_tokens_scaled(35, t, 1, spec, 1e5)[0],
}


@pytest.mark.parametrize("case", list(RANGE_CASES))
@pytest.mark.parametrize("act", ["bf16", "f32"])
def test_decode_dynamic_range(case, act):
    spec = si.LayerSpec(hidden=1024, inter=512, n_experts=32, act=act)
    layer = si.gen_layer(30, 0, spec)
    err, flags = check_layer(layer, 4, tokens_fn=lambda t: RANGE_CASES[case](spec, t))
    print(f"{case}/{act}: max normwise err {err:.3e}, near-tie tokens {flags}")


def test_zero_input_exact():
    spec = si.LayerSpec(hidden=256, inter=128, n_experts=16)
    layer = si.gen_layer(3, 0, spec)
    with moe.MoELayer(layer) as ml:
        y32, ids, w, yb, _ = decode_one(ml, spec, np.zeros(256, np.uint16))
    assert list(ids) == list(range(8))
    assert np.all(w == np.float32(0.125))
    assert np.all(y32 == 0)


def test_bit_reproducible():
    spec = si.CONFIGS["tiny"]
    layer = si.gen_layer(0, 0, spec)
    x = si.gen_tokens(5, 0, 1, spec)[0]
    with moe.MoELayer(layer) as ml:
        a = decode_one(ml, spec, x)[0]
        b = decode_one(ml, spec, x)[0]
    assert np.array_equal(a, b)


def test_route_matches_decode_selection():
    """moe_route and moe_decode select alike, bit for bit (both in the router
    kernel's last block)."""
    spec = si.LayerSpec(hidden=1024, inter=256, n_experts=128, zipf_alpha=1.1)
    layer = si.gen_layer(12, 0, spec)
    with moe.MoELayer(layer) as ml:
        for t in range(8):
            x_np = si.gen_tokens(12, t, 1, spec)[0]
            _, ids, w, _, _ = decode_one(ml, spec, x_np)
            ri = torch.empty(8, dtype=torch.int32, device="cuda")
            rw = torch.empty(8, dtype=torch.float32, device="cuda")
            ml.route(to_dev(x_np, spec), 1, ri, rw)
            torch.cuda.synchronize()
            assert np.array_equal(ri.cpu().numpy(), ids)
            assert np.array_equal(rw.cpu().numpy().view(np.uint32), w.view(np.uint32))


def test_shared_wait_runs_out_and_recovers():
    """Failure detection without a GPU fault: the gate/up kernel never counts
    itself in the shared-expert counter, the down kernel's bounded wait on it
    gives up, the host reads MOE_E_TIMEOUT, and the output is still right (the
    shared rows run after the ordinary wait instead); the next call is normal."""
    spec = si.LayerSpec(hidden=512, inter=256, n_experts=32)
    layer = si.gen_layer(8, 0, spec)
    x = si.gen_tokens(8, 0, 1, spec)[0]
    with moe.MoELayer(layer) as ml:
        ml.set_option(moe.MOE_OPT_TEST_STALL_SHARED, 1)
        y32, ids, w, yb, _ = decode_one(ml, spec, x)
        st, bits = ml.check()
        assert st == 5 and bits != 0  # MOE_E_TIMEOUT
        compare_token(layer, x, y32, ids, w, y_bf16=yb)
        ml.set_option(moe.MOE_OPT_TEST_STALL_SHARED, 0)
        y32b, ids, w, yb, _ = decode_one(ml, spec, x)
        assert ml.check() == (0, 0)
        assert np.array_equal(y32, y32b)
        compare_token(layer, x, y32b, ids, w, y_bf16=yb)


def test_host_buffer_entry_matches_device_path():
    spec = si.LayerSpec(hidden=512, inter=256, n_experts=32)
    layer = si.gen_layer(2, 0, spec)
    T = 5
    X = si.gen_tokens(9, 0, T, spec)
    yh = np.zeros((T, 512), np.uint16)
    with moe.MoELayer(layer) as ml:
        ml.decode_tokens_host(X, T, yh)
        for t in range(T):
            _, _, _, yb, _ = decode_one(ml, spec, X[t])
            assert np.array_equal(yb, yh[t])


def test_route_many_tokens():
    spec = si.LayerSpec(hidden=1024, inter=128, n_experts=128, zipf_alpha=1.1)
    layer = si.gen_layer(4, 0, spec)
    T = 128
    X = si.gen_tokens(4, 0, T, spec)
    x = to_dev(X.reshape(-1), spec)
    ids = torch.empty(T * 8, dtype=torch.int32, device="cuda")
    w = torch.empty(T * 8, dtype=torch.float32, device="cuda")
    Wr = oracle.router_weights_f64(layer.router)
    from _parity import check_selection, W_TOL
    with moe.MoELayer(layer, max_tokens=T) as ml:
        ml.route(x, T, ids, w)
        torch.cuda.synchronize()
    ids = ids.cpu().numpy().reshape(T, 8)
    w = w.cpu().numpy().reshape(T, 8)
    flagged = 0
    for t in range(T):
        use, fl = check_selection(layer, X[t], ids[t], Wr)
        flagged += fl
        l = oracle.router_logits(Wr, oracle.bf16_bits_to_f64(X[t]), layer.router_bias)
        assert np.allclose(w[t], oracle.routing_weights(l[use]), atol=W_TOL, rtol=0)
    print("near-tie tokens", flagged)


def test_argument_errors():
    spec = si.LayerSpec(hidden=128, inter=64, n_experts=8)
    layer = si.gen_layer(1, 0, spec)
    x = torch.zeros(128, dtype=torch.bfloat16, device="cuda")
    with moe.MoELayer(layer) as ml:
        with pytest.raises(moe.MoEError) as ei:
            ml.decode(x, None, None)
        assert ei.value.status == 1
        ids = torch.empty(16, dtype=torch.int32, device="cuda")
        w = torch.empty(16, dtype=torch.float32, device="cuda")
        with pytest.raises(moe.MoEError):
            ml.route(x, 2, ids, w)  # max_tokens is 1
        with pytest.raises(moe.MoEError):
            ml.selection(2, ids, w)  # max_tokens is 1
        with pytest.raises(moe.MoEError) as ei:
            ml.cache_stage(ids, 1)
        assert ei.value.status == 6
        with pytest.raises(moe.MoEError) as ei:
            ml.set_option(1, 0)   # no such option
        assert ei.value.status == 1


@pytest.fixture(scope="module")
def gemma_layer():
    return si.gen_layer(0, 0, si.CONFIGS["gemma_decode"])


def test_gemma_scale_decode(gemma_layer):
    err, flags = check_layer(gemma_layer, 16, seed=0)
    print(f"gemma: max normwise err {err:.3e}, near-tie tokens {flags}")


@pytest.fixture(scope="module")
def glm_layer():
    return si.gen_layer(0, 0, si.CONFIGS["glm_decode"])


@pytest.mark.slow
def test_glm_scale_decode(glm_layer):
    err, flags = check_layer(glm_layer, 4, seed=0)
    print(f"glm: max normwise err {err:.3e}, near-tie tokens {flags}")


def test_back_to_back_decodes_match_synchronised():
    """Many decodes queued back to back over two layer instances (the kernels
    of consecutive calls overlap through programmatic dependent launch, and
    each kernel reads the tagged words its predecessor publishes before that
    one completes) give bit-identical outputs to the same decodes with a
    synchronisation after every call."""
    spec = si.LayerSpec(hidden=1024, inter=512, n_experts=64, zipf_alpha=1.1)
    layer = si.gen_layer(41, 0, spec)
    T = 96
    X = si.gen_tokens(41, 0, T, spec)
    x = to_dev(X, spec)
    ya = torch.empty((T, spec.hidden), dtype=torch.bfloat16, device="cuda")
    yb = torch.empty((T, spec.hidden), dtype=torch.bfloat16, device="cuda")
    with moe.MoELayer(layer) as m0, moe.MoELayer(layer) as m1:
        mls = (m0, m1)
        for t in range(T):
            mls[t % 2].decode(x[t], ya[t])
        torch.cuda.synchronize()
        for t in range(T):
            mls[t % 2].decode(x[t], yb[t])
            torch.cuda.synchronize()
        assert m0.check() == (0, 0) and m1.check() == (0, 0)
    assert torch.equal(ya, yb)
