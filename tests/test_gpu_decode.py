"""Decode path on the GPU against the fp64 oracle (parity), through the C ABI."""
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


def decode_one(ml, spec, x_np):
    H, k = spec.hidden, spec.top_k
    x = to_dev(x_np, spec)
    yd = torch.bfloat16 if spec.act == "bf16" else torch.float32
    y = torch.empty(H, dtype=yd, device="cuda")
    y32 = torch.empty(H, dtype=torch.float32, device="cuda")
    ids = torch.empty(k, dtype=torch.int32, device="cuda")
    w = torch.empty(k, dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream()
    ml.decode(x, y, y32, stream=s)
    ml.route(x, 1, ids, w, stream=s)
    torch.cuda.synchronize()
    yb = y.view(torch.int16).cpu().numpy().view(np.uint16) if spec.act == "bf16" else None
    return y32.cpu().numpy(), ids.cpu().numpy(), w.cpu().numpy(), yb, y


PATHS = {"split": moe.MOE_PATH_SPLIT, "fused": moe.MOE_PATH_FUSED}


def check_layer(layer, tokens, seed=100, path="fused"):
    spec = layer.spec
    Wr = oracle.router_weights_f64(layer.router)
    errs, flags = [], 0
    with moe.MoELayer(layer) as ml:
        ml.set_option(moe.MOE_OPT_DECODE_PATH, PATHS[path])
        for t in range(tokens):
            x = si.gen_tokens(seed, t, 1, spec)[0]
            y32, ids, w, yb, _ = decode_one(ml, spec, x)
            err, flagged = compare_token(layer, x, y32, ids, w, Wr=Wr, y_bf16=yb)
            errs.append(err)
            flags += flagged
        st, bits = ml.check()
        assert st == 0, bits
    return max(errs), flags


@pytest.mark.parametrize("path", list(PATHS))
def test_tiny_layer_decode(path):
    layer = si.gen_layer(0, 0, si.CONFIGS["tiny"])
    err, flags = check_layer(layer, 32, path=path)
    print(f"tiny/{path}: max normwise err {err:.3e}, near-tie tokens {flags}")


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


# the fused decode's per-CTA buffers do not take the long rows (it refuses the
# layer with MOE_E_UNSUPPORTED); the split path covers them
SPLIT_ONLY = {"long_rows"}


@pytest.mark.parametrize("name,path", [(n, p) for p in PATHS for n in SHAPES if p == "split" or n not in SPLIT_ONLY])
def test_decode_shapes(name, path):
    layer = si.gen_layer(7, 1, SHAPES[name])
    err, flags = check_layer(layer, 6, seed=7, path=path)
    print(f"{name}/{path}: max normwise err {err:.3e}, near-tie tokens {flags}")


@pytest.mark.parametrize("path", list(PATHS))
def test_zero_input_exact(path):
    spec = si.LayerSpec(hidden=256, inter=128, n_experts=16)
    layer = si.gen_layer(3, 0, spec)
    with moe.MoELayer(layer) as ml:
        ml.set_option(moe.MOE_OPT_DECODE_PATH, PATHS[path])
        y32, ids, w, yb, _ = decode_one(ml, spec, np.zeros(256, np.uint16))
    assert list(ids) == list(range(8))
    assert np.all(w == np.float32(0.125))
    assert np.all(y32 == 0)


@pytest.mark.parametrize("path", list(PATHS))
def test_bit_reproducible(path):
    spec = si.CONFIGS["tiny"]
    layer = si.gen_layer(0, 0, spec)
    x = si.gen_tokens(5, 0, 1, spec)[0]
    with moe.MoELayer(layer) as ml:
        ml.set_option(moe.MOE_OPT_DECODE_PATH, PATHS[path])
        a = decode_one(ml, spec, x)[0]
        b = decode_one(ml, spec, x)[0]
    assert np.array_equal(a, b)


def test_fused_wait_runs_out_and_recovers():
    """Failure detection without a GPU fault: the routing flag is never set, every
    bounded wait on it gives up, the kernel drains out and the host reads
    MOE_E_TIMEOUT; the next call runs normally."""
    spec = si.LayerSpec(hidden=512, inter=256, n_experts=32)
    layer = si.gen_layer(8, 0, spec)
    x = si.gen_tokens(8, 0, 1, spec)[0]
    with moe.MoELayer(layer) as ml:
        ml.set_option(moe.MOE_OPT_DECODE_PATH, moe.MOE_PATH_FUSED)
        ml.set_option(moe.MOE_OPT_TEST_STALL_ROUTING, 1)
        decode_one(ml, spec, x)
        st, bits = ml.check()
        assert st == 5 and bits != 0  # MOE_E_TIMEOUT
        ml.set_option(moe.MOE_OPT_TEST_STALL_ROUTING, 0)
        y32, ids, w, yb, _ = decode_one(ml, spec, x)
        assert ml.check() == (0, 0)
        compare_token(layer, x, y32, ids, w, y_bf16=yb)


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
        with pytest.raises(moe.MoEError) as ei:
            ml.cache_stage(ids, 1)
        assert ei.value.status == 6


@pytest.fixture(scope="module")
def gemma_layer():
    return si.gen_layer(0, 0, si.CONFIGS["gemma_decode"])


@pytest.mark.parametrize("path", list(PATHS))
def test_gemma_scale_decode(gemma_layer, path):
    err, flags = check_layer(gemma_layer, 16, seed=0, path=path)
    print(f"gemma/{path}: max normwise err {err:.3e}, near-tie tokens {flags}")


@pytest.fixture(scope="module")
def glm_layer():
    return si.gen_layer(0, 0, si.CONFIGS["glm_decode"])


@pytest.mark.slow
@pytest.mark.parametrize("path", list(PATHS))
def test_glm_scale_decode(glm_layer, path):
    err, flags = check_layer(glm_layer, 4, seed=0, path=path)
    print(f"glm/{path}: max normwise err {err:.3e}, near-tie tokens {flags}")


def test_back_to_back_decodes_match_synchronised():
    """Many decodes queued back to back over two layer instances (the kernels
    of consecutive calls overlap through programmatic dependent launch) give
    bit-identical outputs to the same decodes with a synchronisation after
    every call."""
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
