"""C ABI: the library loads and exports what include/moe.h declares; host-side
logic (argument checks, record packing) behaves as documented. No GPU needed."""
import os
import re

import numpy as np
import pytest

import quantized_routed_expert_moe_gb300 as moe
import seeded_inputs as si
from conftest import ROOT


@pytest.fixture(scope="module", autouse=True)
def built():
    from quantized_routed_expert_moe_gb300 import build
    build.build()


def header_functions():
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)) - {"moe_expert_source"})


def test_every_declared_symbol_is_exported():
    names = header_functions()
    assert len(names) >= 12
    L = moe.lib()
    for n in names:
        assert hasattr(L, n), n
    assert sorted(moe.EXPORTS) == names


def header_constants():
    """Integer constants of include/moe.h: enumerators with explicit values and
    #defines of integer expressions."""
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    out = {n: int(v) for n, v in re.findall(r"\b(MOE_[A-Z0-9_]+)\s*=\s*(-?[0-9]+)\b", text)}
    for n, expr in re.findall(r"#define\s+(MOE_[A-Z0-9_]+)\s+([0-9()*+ u]+)\s*$", text, flags=re.M):
        out[n] = int(eval(expr.replace("u", "")))
    return out


def test_binding_constants_match_header():
    """The binding's constants (option ids, formats, limits) equal the
    header's, so a call from Python means what the header documents."""
    consts = header_constants()
    for must in ("MOE_OPT_CACHE_DEVICE", "MOE_OPT_TEST_STALL_SHARED", "MOE_W_Q2G64",
                 "MOE_MAX_TOP_K", "MOE_STATIC_SCRATCH_BYTES", "MOE_SCORE_SIGMOID"):
        assert must in consts, must
    checked = 0
    for name, value in consts.items():
        if hasattr(moe, name):
            assert getattr(moe, name) == value, (name, getattr(moe, name), value)
            checked += 1
    assert checked >= 15
    # the status values the tests compare against as literals
    assert (consts["MOE_OK"], consts["MOE_E_INVALID"], consts["MOE_E_UNSUPPORTED"], consts["MOE_E_TIMEOUT"],
            consts["MOE_E_STATE"], consts["MOE_E_SOURCE"]) == (0, 1, 2, 5, 6, 7)


def test_status_strings():
    for code, name in moe.STATUS.items():
        assert moe.moe_status_str(code) == name


def test_invalid_descriptors_rejected_before_cuda():
    spec = si.CONFIGS["tiny"]
    layer = si.gen_layer(0, 0, si.LayerSpec(hidden=64, inter=64, n_experts=8, act="f32"))
    bad = [
        dict(hidden=100), dict(inter=0), dict(top_k=9), dict(top_k=0), dict(n_experts=4),
        dict(max_tokens=129), dict(cache_slots=2),
    ]
    for kw in bad:
        args = dict(hidden=64, inter=64, n_experts=8, top_k=8, n_shared=1, router_fmt="f32",
                    act="f32", max_tokens=1, cache_slots=0)
        args.update(kw)
        d = moe.make_desc(**args)
        with pytest.raises(moe.MoEError) as ei:
            moe.moe_layer_create(d, layer.router, None, layer.shared, layer.experts, device=0)
        assert ei.value.status == 1, kw
    d = moe.make_desc(64, 64, 8, act="f32")
    d.abi_version = 99
    with pytest.raises(moe.MoEError):
        moe.moe_layer_create(d, layer.router, None, layer.shared, layer.experts)
    assert spec.hidden == 512


def test_router_scoring_null_layer_rejected():
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_layer_set_router_scoring(None, moe.MOE_SCORE_SIGMOID, 2.5)
    assert ei.value.status == 1


def test_no_cpu_fallback_without_gpu():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    layer = si.gen_layer(0, 0, si.LayerSpec(hidden=64, inter=64, n_experts=8, act="f32"))
    d = moe.make_desc(64, 64, 8, act="f32")
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_layer_create(d, layer.router, None, layer.shared, layer.experts)
    assert ei.value.status == 4  # MOE_E_CUDA: fails loudly, nothing runs on the CPU


def _expected_record(e, H, I):
    """The documented record layout, built independently with numpy."""
    def rowrec(q, n, K):
        codes = q.codes[n].tobytes()
        meta = np.stack([q.scale[n], q.bias[n]], axis=1).astype(np.uint16).tobytes()
        pad = (-(len(meta)) % 16)
        return codes + meta + b"\0" * pad
    parts = []
    for i in range(I):
        parts.append(rowrec(e.gate, i, H))
        parts.append(rowrec(e.up, i, H))
    for n in range(H):
        parts.append(rowrec(e.down, n, I))
    return b"".join(parts)


def _expected_record_q2(e, H, I):
    """The documented 2-bit kernel layout, built independently with numpy: per
    word of 16 codes, byte i holds elements 2i, 2i+1, 8+2i, 9+2i at bits 0, 2, 4, 6."""
    def rowrec(q, n, K):
        c = np.zeros(K, np.uint8)
        for j in range(4):
            c[j::4] = (q.codes[n] >> (2 * j)) & 3
        c = c.reshape(K // 16, 16)
        out = np.zeros((K // 16, 4), np.uint8)
        for i in range(4):
            out[:, i] = c[:, 2 * i] | (c[:, 2 * i + 1] << 2) | (c[:, 8 + 2 * i] << 4) | (c[:, 9 + 2 * i] << 6)
        meta = np.stack([q.scale[n], q.bias[n]], axis=1).astype(np.uint16).tobytes()
        return out.tobytes() + meta + b"\0" * (-(len(meta)) % 16)
    parts = []
    for i in range(I):
        parts.append(rowrec(e.gate, i, H))
        parts.append(rowrec(e.up, i, H))
    for n in range(H):
        parts.append(rowrec(e.down, n, I))
    return b"".join(parts)


@pytest.mark.parametrize("H,I", [(128, 64), (192, 320)])
def test_record_packing_q2(H, I):
    spec = si.LayerSpec(hidden=H, inter=I, n_experts=8, act="f32", expert_bits=2)
    e = si.gen_expert(5, 0, 1, spec)
    d = moe.desc_from_spec(spec)
    n = moe.moe_expert_record_bytes(d)
    want = _expected_record_q2(e, H, I)
    assert n == len(want)
    buf = np.zeros(n, np.uint8)
    moe.moe_pack_expert_record(d, e, buf)
    assert buf.tobytes() == want


@pytest.mark.parametrize("H,I", [(128, 64), (192, 320), (512, 256)])
def test_record_packing(H, I):
    spec = si.LayerSpec(hidden=H, inter=I, n_experts=8)
    e = si.gen_expert(1, 0, 2, spec)
    d = moe.desc_from_spec(spec)
    nb = moe.moe_expert_record_bytes(d)
    want = _expected_record(e, H, I)
    assert nb == len(want)
    dst = np.zeros(nb, np.uint8)
    moe.moe_pack_expert_record(d, e, dst)
    assert dst.tobytes() == want


def test_record_bytes_match_format():
    # cfg sizes: no padding when K/16 is a multiple of 16 bytes
    for name in ("tiny", "glm_decode"):
        spec = si.CONFIGS[name]
        assert moe.moe_expert_record_bytes(moe.desc_from_spec(spec)) == spec.expert_bytes()
    g = si.CONFIGS["gemma_decode"]
    # down rows of I = 704 carry 44 metadata bytes padded to 48
    assert moe.moe_expert_record_bytes(moe.desc_from_spec(g)) == g.expert_bytes() + 2816 * 4
