"""moe_decode_static_scratch: decode with the library's fixed per-device
scratch region, for callers that may not allocate device memory while they
serve tokens (an allocation can synchronise the device and stall other
streams, and an engine that has already divided HBM has none to give).

The file name sorts last so that the GPU test also runs after every other test
in one session; it must pass alone as well. Every buffer the calls touch is
allocated before the first call.
"""
import re
from pathlib import Path

import numpy as np
import pytest
import torch

import quantized_routed_expert_moe_gb300 as moe
import seeded_inputs as si
from _parity import compare_token

HEADER = Path(__file__).resolve().parents[1] / "include" / "moe.h"


def test_scratch_limit_matches_header():
    m = re.search(r"#define MOE_STATIC_SCRATCH_BYTES \((\d+)u \* (\d+)u\)", HEADER.read_text())
    assert m and int(m.group(1)) * int(m.group(2)) == moe.MOE_STATIC_SCRATCH_BYTES


def _dev_x(x_np, spec):
    if spec.act == "bf16":
        return torch.from_numpy(np.ascontiguousarray(x_np).view(np.int16)).cuda()
    return torch.from_numpy(np.ascontiguousarray(x_np, dtype=np.float32)).cuda()


@pytest.fixture(scope="module")
def built():
    from quantized_routed_expert_moe_gb300 import build
    build.build()
    assert torch.cuda.is_available()


CASES = {
    "tiny_f32": si.CONFIGS["tiny"],
    "gemma_q8_router": si.CONFIGS["gemma_decode"],
    "no_shared_bf16": si.LayerSpec(hidden=128, inter=192, n_experts=16, top_k=4, n_shared=0),
}


@pytest.mark.gpu
@pytest.mark.parametrize("name", list(CASES))
def test_static_scratch_matches_decode(built, name):
    """Two calls in a row give, bit for bit, what moe_decode gives for the same
    tokens (the same kernels over other scratch), and that is within the
    tolerance of the fp64 oracle on the selection moe_decode combined with.
    After the first call (which looks up the region once), further calls leave
    the device's free memory unchanged: nothing is allocated."""
    spec = CASES[name]
    layer = si.gen_layer(11, 0, spec)
    H, k = spec.hidden, spec.top_k
    yd = torch.bfloat16 if spec.act == "bf16" else torch.float32
    X = [si.gen_tokens(11, t, 1, spec)[0] for t in range(2)]
    xs = [_dev_x(x, spec) for x in X]
    y_ref = [torch.empty(H, dtype=torch.float32, device="cuda") for _ in xs]
    ids = [torch.empty(k, dtype=torch.int32, device="cuda") for _ in xs]
    w = [torch.empty(k, dtype=torch.float32, device="cuda") for _ in xs]
    y_a = [torch.empty(H, dtype=torch.float32, device="cuda") for _ in xs]
    yb_a = [torch.empty(H, dtype=yd, device="cuda") for _ in xs]
    with moe.MoELayer(layer) as ml:
        s = torch.cuda.current_stream()
        for x, y, i, ww in zip(xs, y_ref, ids, w):
            ml.decode(x, None, y, stream=s)
            ml.selection(1, i, ww, stream=s)
        torch.cuda.synchronize()
        # two calls in a row on one stream, different tokens
        for x, y, yb in zip(xs, y_a, yb_a):
            ml.decode_static_scratch(x, yb, y, stream=s)
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        for _ in range(20):
            for x, y, yb in zip(xs, y_a, yb_a):
                ml.decode_static_scratch(x, yb, y, stream=s)
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free0
    for t, (y, yb, ref) in enumerate(zip(y_a, yb_a, y_ref)):
        assert torch.equal(y, ref)
        assert torch.equal(yb, y.to(yd))
        compare_token(layer, X[t], y.cpu().numpy(), ids[t].cpu().numpy(), w[t].cpu().numpy())


@pytest.mark.gpu
def test_static_scratch_rejects_oversized_layer(built):
    # (k + 1) * I * 4 bytes of SwiGLU outputs alone exceed the region, while
    # the layer itself is valid (its decode kernels fit in shared memory)
    spec = si.LayerSpec(hidden=64, inter=7296, n_experts=8, top_k=8)
    assert (spec.top_k + 1) * spec.inter * 4 > moe.MOE_STATIC_SCRATCH_BYTES
    layer = si.gen_layer(12, 0, spec)
    x = _dev_x(si.gen_tokens(12, 0, 1, spec)[0], spec)
    y = torch.full((spec.hidden,), 7.0, dtype=torch.float32, device="cuda")
    with moe.MoELayer(layer) as ml:
        with pytest.raises(moe.MoEError) as ei:
            ml.decode_static_scratch(x, None, y)
        assert ei.value.status == 1  # MOE_E_INVALID
        assert "static region holds" in str(ei.value)
        torch.cuda.synchronize()
    assert torch.all(y == 7.0)  # nothing ran
