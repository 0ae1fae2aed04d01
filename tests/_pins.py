"""Checks that pin the fp64 oracle to facts fixed outside itself.

Each ``pin_*`` function raises AssertionError when the oracle disagrees with
a hand-worked table, a closed form, brute force or an independent pure-Python
restatement. ``tests/test_oracle_pins.py`` runs them on the oracle as it is,
and again with planted mistakes to show each mistake is caught.
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np

import oracle
import seeded_inputs as si
from seeded_inputs import LayerSpec, QMat, Expert, Router, Layer

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------------------
# golden-table readers
# ---------------------------------------------------------------------------

def _read_cases(path):
    cases, cur = [], None
    for raw in open(path):
        line = raw.strip()
        if not line or line.startswith("#"):
            continue
        tok = line.split()
        if tok[0] == "case":
            cur = {"name": tok[1], "bytes": {}, "groups": {}, "expect": {}}
            cases.append(cur)
        elif tok[0] == "bytes":
            for t in tok[1:]:
                i, h = t.split(":")
                cur["bytes"][int(i)] = int(h, 16)
        elif tok[0] == "group":
            g = int(tok[1])
            kv = dict(t.split("=") for t in tok[2:])
            cur["groups"][g] = (int(kv["scale"], 16), int(kv["bias"], 16))
        elif tok[0] == "expect":
            for t in tok[1:]:
                k, v = t.split("=")
                cur["expect"][int(k)] = Fraction(v)
    return cases


def read_sizes():
    out = {}
    for raw in open(os.path.join(GOLDEN, "format_sizes.txt")):
        line = raw.strip()
        if line and not line.startswith("#"):
            k, v = line.split()
            out[k] = float(v)
    return out


def read_lfu():
    slots, rows = None, []
    for raw in open(os.path.join(GOLDEN, "lfu_trace.txt")):
        line = raw.strip()
        if not line or line.startswith("#"):
            continue
        if line.startswith("slots"):
            slots = int(line.split()[1])
            continue
        tok, hits, fills = [p.strip() for p in line.split("|")]
        ids = [int(v) for v in tok.split()[1].split(",")]
        h = hits.split()[1]
        h = [] if h == "-" else [int(v) for v in h.split(",")]
        f = [tuple(int(v) for v in t.split(":")) for t in fills.split()[1:]]
        rows.append((ids, h, f))
    return slots, rows


def read_lfu_prefetch():
    """(slots, [(op, ids, hits_or_resident, fills)]) from lfu_prefetch.txt."""
    slots, rows = None, []
    for raw in open(os.path.join(GOLDEN, "lfu_prefetch.txt")):
        line = raw.strip()
        if not line or line.startswith("#"):
            continue
        if line.startswith("slots"):
            slots = int(line.split()[1])
            continue
        head, mid, fills = [p.strip() for p in line.split("|")]
        op, ids = head.split()
        m = mid.split()[1]
        m = [] if m == "-" else [int(v) for v in m.split(",")]
        f = [tuple(int(v) for v in t.split(":")) for t in fills.split()[1:]]
        rows.append((op, [int(v) for v in ids.split(",")], m, f))
    return slots, rows


def read_lfu_pinned():
    """(slots, [(op, args...)]) from lfu_pinned.txt: ("token", ids, hits,
    fills), ("pin", ids) or ("hottest", n, ids)."""
    slots, rows = None, []
    for raw in open(os.path.join(GOLDEN, "lfu_pinned.txt")):
        line = raw.strip()
        if not line or line.startswith("#"):
            continue
        if line.startswith("slots"):
            slots = int(line.split()[1])
            continue
        parts = [p.strip() for p in line.split("|")]
        op, arg = parts[0].split()
        ints = lambda v: [] if v == "-" else [int(u) for u in v.split(",")]
        if op == "pin":
            rows.append(("pin", ints(arg)))
        elif op == "hottest":
            rows.append(("hottest", int(arg), ints(parts[1])))
        else:
            h = ints(parts[1].split()[1])
            f = [tuple(int(u) for u in t.split(":")) for t in parts[2].split()[1:]]
            rows.append(("token", ints(arg), h, f))
    return slots, rows


# ---------------------------------------------------------------------------
# small layers built by hand
# ---------------------------------------------------------------------------

def const_qmat(N, K, code, scale_bits, bias_bits) -> QMat:
    byte = (code & 0xF) | ((code & 0xF) << 4)
    return QMat(np.full((N, K // 2), byte, np.uint8),
                np.full((N, K // 64), scale_bits, np.uint16),
                np.full((N, K // 64), bias_bits, np.uint16), 4, N, K)


def const_layer(H, I, E, k, code=9, scale_bits=0x2000, bias_bits=0xAC00, act="f32"):
    """Every weight equals (code - 8) * 2^-7 when bias = -8 * scale."""
    spec = LayerSpec(hidden=H, inter=I, n_experts=E, top_k=k, act=act)
    ex = Expert(const_qmat(I, H, code, scale_bits, bias_bits),
                const_qmat(I, H, code, scale_bits, bias_bits),
                const_qmat(H, I, code, scale_bits, bias_bits))
    rng = np.random.default_rng(5)
    router = Router("f32", w=(rng.standard_normal((E, H)) * 0.02).astype(np.float32))
    return Layer(spec, router, [ex] * E, ex)


def tiny_layer(seed=3, H=64, I=64, E=6, k=2, zipf=None, act="f32", router_fmt="f32"):
    spec = LayerSpec(hidden=H, inter=I, n_experts=E, top_k=k, act=act,
                     zipf_alpha=zipf, router_fmt=router_fmt)
    return si.gen_layer(seed, 0, spec)


# ---------------------------------------------------------------------------
# pins
# ---------------------------------------------------------------------------

def pin_dequant_q4_table():
    """Hand-worked 4-bit rows (golden/q4g64_dequant.txt) must come out exactly."""
    for case in _read_cases(os.path.join(GOLDEN, "q4g64_dequant.txt")):
        K = 128
        codes = np.zeros((1, K // 2), np.uint8)
        for i, v in case["bytes"].items():
            codes[0, i] = v
        sc = np.zeros((1, K // 64), np.uint16)
        bi = np.zeros((1, K // 64), np.uint16)
        for g, (s, b) in case["groups"].items():
            sc[0, g], bi[0, g] = s, b
        W = oracle.dequant_q4g64(codes, sc, bi)
        for k, v in case["expect"].items():
            assert Fraction(float(W[0, k])) == v, (case["name"], k, float(W[0, k]), float(v))


def pin_dequant_q2_table():
    """Hand-worked 2-bit rows (golden/q2g64_dequant.txt) must come out exactly."""
    for case in _read_cases(os.path.join(GOLDEN, "q2g64_dequant.txt")):
        K = 128
        codes = np.zeros((1, K // 4), np.uint8)
        for i, v in case["bytes"].items():
            codes[0, i] = v
        sc = np.zeros((1, K // 64), np.uint16)
        bi = np.zeros((1, K // 64), np.uint16)
        for g, (s, b) in case["groups"].items():
            sc[0, g], bi[0, g] = s, b
        W = oracle.dequant_q2g64(codes, sc, bi)
        for k, v in case["expect"].items():
            assert Fraction(float(W[0, k])) == v, (case["name"], k, float(W[0, k]), float(v))


def pin_q2_layer():
    """A tiny 2-bit layer equals the pure-Python restatement; constant codes
    give the closed form of the 4-bit case with code - 2 = 1 (code 3, bias -2s)."""
    spec = LayerSpec(hidden=128, inter=64, n_experts=6, top_k=2, act="f32", expert_bits=2)
    layer = si.gen_layer(17, 0, spec)
    for t in range(2):
        x = si.gen_tokens(17, t, 1, spec)[0]
        y, info = oracle.moe_token(layer, x)
        yp, S, w = _py_layer(layer, x)
        assert list(info.ids) == S
        assert np.allclose(y, yp, rtol=1e-11, atol=1e-14)
    H, I, s = 128, 64, 2.0 ** -7
    q = lambda N, K: QMat(np.full((N, K // 4), 0xFF, np.uint8), np.full((N, K // 64), 0x2000, np.uint16),
                          np.full((N, K // 64), 0xA400, np.uint16), 2, N, K)
    ex = Expert(q(I, H), q(I, H), q(H, I))
    lay = Layer(LayerSpec(hidden=H, inter=I, n_experts=4, top_k=2, act="f32", expert_bits=2),
                Router("f32", w=np.zeros((4, H), np.float32)), [ex] * 4, ex)
    x = si.gen_tokens(18, 0, 1, LayerSpec(hidden=H, inter=I, n_experts=4, act="f32"))[0]
    g = s * float(np.sum(x.astype(np.float64)))
    h = g / (1 + math.exp(-g)) * g
    y, _ = oracle.moe_token(lay, x)
    assert np.allclose(y, 2.0 * I * s * h, rtol=1e-12, atol=0)


def pin_dequant_q8_table():
    for case in _read_cases(os.path.join(GOLDEN, "q8g64_dequant.txt")):
        K = 128
        codes = np.zeros((1, K), np.uint8)
        for i, v in case["bytes"].items():
            codes[0, i] = v
        sc = np.zeros((1, K // 64), np.uint16)
        bi = np.zeros((1, K // 64), np.uint16)
        for g, (s, b) in case["groups"].items():
            sc[0, g], bi[0, g] = s, b
        W = oracle.dequant_q8g64(codes, sc, bi)
        for k, v in case["expect"].items():
            assert Fraction(float(W[0, k])) == v, (case["name"], k, float(W[0, k]), float(v))


def pin_format_sizes():
    """Canonical expert sizes against the sizes the pages print."""
    z = read_sizes()
    gemma = si.CONFIGS["gemma_decode"]
    e = si.gen_expert(0, 0, 0, gemma)
    assert e.nbytes == gemma.expert_bytes() == 3 * 2816 * 704 * 9 // 16
    assert abs(e.nbytes / z["gemma_expert_bytes_page"] - 1) < z["gemma_expert_bytes_rel_tol"]
    glm = si.CONFIGS["glm_decode"]
    nib = 3 * glm.hidden * glm.inter // 2
    assert abs(nib / z["glm_expert_nibble_bytes_page"] - 1) < z["glm_expert_nibble_bytes_rel_tol"]
    cold = z["glm_moe_layers"] * glm.top_k * nib
    assert abs(cold / z["glm_cold_token_bytes_page"] - 1) < 0.02


def pin_zero_input_routing():
    """x = 0 and no bias: all logits tie at 0, so ids = 0..k-1 (lower index wins), w = 1/k."""
    layer = tiny_layer(E=12, k=8)
    y, info = oracle.moe_token(layer, np.zeros(layer.spec.hidden, np.float32))
    assert list(info.ids) == list(range(8))
    assert np.all(info.weights == 1.0 / 8)
    assert np.all(y == 0.0)


def pin_topk_is_full_sort():
    """Selection equals the first k of a full sort by (-l, e) done with Python's sorted()."""
    layer = tiny_layer(E=32, k=8, H=128)
    Wr = oracle.router_weights_f64(layer.router)
    for t in range(20):
        x = si.gen_tokens(11, t, 1, layer.spec)[0]
        l = oracle.router_logits(Wr, x.astype(np.float64))
        ids, _ = oracle.select_topk(l, 8)
        want = sorted(range(32), key=lambda e: (-float(l[e]), e))[:8]
        assert list(ids) == want
    # planted ties: identical router rows 3 and 17 and 9 and 30
    l = np.zeros(32)
    l[[3, 17]] = 2.0
    l[[9, 30]] = 1.0
    l[[5, 6, 7, 8]] = 0.5
    ids, gap = oracle.select_topk(l, 5)
    assert list(ids) == [3, 17, 9, 30, 5] and gap == 0.0


def pin_routing_weights():
    """Weights sum to 1; with k = E they are the dense softmax (pure Python)."""
    layer = tiny_layer(E=8, k=8, H=64)
    x = si.gen_tokens(2, 0, 1, layer.spec)[0]
    _, info = oracle.moe_token(layer, x)
    assert abs(info.weights.sum() - 1.0) < 1e-12
    Wr = oracle.router_weights_f64(layer.router)
    l = [sum(float(Wr[e, i]) * float(x[i]) for i in range(64)) for e in range(8)]
    m = max(l)
    z = sum(math.exp(v - m) for v in l)
    for j, e in enumerate(info.ids):
        assert abs(info.weights[j] - math.exp(l[int(e)] - m) / z) < 1e-14
    # softmax over selected == full softmax renormalised over the selection
    layer2 = tiny_layer(E=16, k=4, H=64)
    Wr2 = oracle.router_weights_f64(layer2.router)
    x2 = si.gen_tokens(2, 1, 1, layer2.spec)[0].astype(np.float64)
    l2 = Wr2 @ x2
    ids, _ = oracle.select_topk(l2, 4)
    p = np.exp(l2 - l2.max()) / np.exp(l2 - l2.max()).sum()
    ren = p[ids] / p[ids].sum()
    assert np.allclose(oracle.routing_weights(l2[ids]), ren, rtol=0, atol=1e-15)


def pin_silu():
    """silu(0) = 0; silu(z) - silu(-z) = z; silu(z) ~ z for large z; sigmoid form by hand."""
    z = np.array([-50.0, -3.0, -0.5, 0.0, 0.5, 3.0, 50.0])
    s = oracle.silu(z)
    assert s[3] == 0.0
    assert np.allclose(s - oracle.silu(-z), z, rtol=0, atol=1e-13)
    assert abs(s[-1] - 50.0) < 1e-15 * 50 + 1e-19
    for v, got in zip(z, s):
        assert abs(got - v / (1 + math.exp(-v))) <= 1e-15 * max(1.0, abs(v))


def pin_ffn_closed_form():
    """All codes 9, scale 2^-7, bias -8 * 2^-7: every weight is 2^-7.

    Then g = u = s * sum(x), h = silu(g) * u and each output is I * s * h.
    With every expert identical the layer output is (1 + sum_j w_j) times
    one expert's output = 2 * I * s * h.
    """
    H, I = 128, 64
    layer = const_layer(H, I, E=8, k=4)
    x = si.gen_tokens(7, 0, 1, LayerSpec(hidden=H, inter=I, n_experts=8, act="f32"))[0]
    s = 2.0 ** -7
    g = s * float(np.sum(x.astype(np.float64)))
    h = g / (1 + math.exp(-g)) * g
    want = 2.0 * I * s * h
    y, info = oracle.moe_token(layer, x)
    assert np.allclose(y, want, rtol=1e-12, atol=0)
    f = oracle.expert_ffn(layer.shared, x)
    assert np.allclose(f, I * s * h, rtol=1e-12, atol=0)
    # a zero input gives exactly zero
    y0, _ = oracle.moe_token(layer, np.zeros(H, np.float32))
    assert np.all(y0 == 0.0)


def pin_dense_brute_force():
    """Sparse dispatch equals every expert evaluated densely and masked to S."""
    for zipf in (None, 1.1):
        layer = tiny_layer(E=12, k=3, H=128, I=64, zipf=zipf)
        for t in range(3):
            x = si.gen_tokens(4, t, 1, layer.spec)[0]
            y, _ = oracle.moe_token(layer, x)
            yd = oracle.layer_dense_f64(layer, x)
            assert np.allclose(y, yd, rtol=1e-12, atol=1e-15)


def _py_layer(layer, x):
    """Independent restatement in pure Python (no numpy arithmetic), from raw bytes."""
    H, I, E, k = layer.spec.hidden, layer.spec.inter, layer.spec.n_experts, layer.spec.top_k

    def f16(bits):
        bits = int(bits)
        e, m = (bits >> 10) & 31, bits & 1023
        v = m * 2.0 ** -24 if e == 0 else (1024 + m) * 2.0 ** (e - 25)
        return -v if bits & 0x8000 else v

    def w4(q, n, kk):
        if getattr(q, "bits", 4) == 2:
            c = (int(q.codes[n, kk // 4]) >> (2 * (kk % 4))) & 3
        else:
            byte = int(q.codes[n, kk // 2])
            c = (byte >> 4) if kk % 2 else (byte & 15)
        return c * f16(q.scale[n, kk // 64]) + f16(q.bias[n, kk // 64])

    def matvec(q, v):
        return [sum(w4(q, n, kk) * v[kk] for kk in range(q.K)) for n in range(q.N)]

    def ffn(ex, v):
        g = matvec(ex.gate, v)
        u = matvec(ex.up, v)
        h = [gi / (1.0 + math.exp(-gi)) * ui for gi, ui in zip(g, u)]
        return matvec(ex.down, h)

    xv = [float(v) for v in x]
    if layer.router.fmt == "f32":
        R = [[float(layer.router.w[e, i]) for i in range(H)] for e in range(E)]
    else:
        q = layer.router.q
        R = [[int(q.codes[e, i]) * f16(q.scale[e, i // 64]) + f16(q.bias[e, i // 64])
              for i in range(H)] for e in range(E)]
    l = [sum(R[e][i] * xv[i] for i in range(H)) for e in range(E)]
    bias = [0.0] * E if layer.router_bias is None else [float(b) for b in layer.router_bias]
    if getattr(layer.spec, "router_score", "softmax") == "sigmoid":
        sc = [1.0 / (1.0 + math.exp(-v)) for v in l]
        S = sorted(range(E), key=lambda e: (-(sc[e] + bias[e]), e))[:k]
        z = sum(sc[e] for e in S)
        w = [layer.spec.routed_scaling * sc[e] / z for e in S]
    else:
        l = [l[e] + bias[e] for e in range(E)]
        S = sorted(range(E), key=lambda e: (-l[e], e))[:k]
        m = max(l[e] for e in S)
        z = sum(math.exp(l[e] - m) for e in S)
        w = [math.exp(l[e] - m) / z for e in S]
    y = ffn(layer.shared, xv)
    for j, e in enumerate(S):
        fe = ffn(layer.experts[e], xv)
        y = [a + w[j] * b for a, b in zip(y, fe)]
    return y, S, w


def pin_pure_python():
    """The oracle equals a pure-Python restatement on tiny layers (f32 and 8-bit routers, with and without bias)."""
    for zipf, rf in ((None, "f32"), (1.1, "f32"), (None, "q8g64")):
        layer = tiny_layer(seed=9, E=6, k=2, H=64, I=64, zipf=zipf, router_fmt=rf)
        x = si.gen_tokens(9, 0, 1, layer.spec)[0]
        y, info = oracle.moe_token(layer, x)
        yp, S, w = _py_layer(layer, x)
        assert list(info.ids) == S
        assert np.allclose(info.weights, w, rtol=0, atol=1e-14)
        assert np.allclose(y, yp, rtol=1e-11, atol=1e-14)
    # non-square FFN (H != I) so a transposed operand cannot pass silently
    layer = tiny_layer(seed=10, E=4, k=2, H=128, I=64)
    x = si.gen_tokens(10, 0, 1, layer.spec)[0]
    y, _ = oracle.moe_token(layer, x)
    yp, _, _ = _py_layer(layer, x)
    assert np.allclose(y, yp, rtol=1e-11, atol=1e-14)


def pin_chunk_rows():
    """The chunk evaluation (each expert dequantised once for all its rows) gives,
    row by row, the pure-Python restatement of the layer; with a forced
    selection it gives the single-token oracle on that selection."""
    for zipf, H, I in ((None, 64, 64), (1.1, 128, 64)):
        layer = tiny_layer(seed=14, E=6, k=2, H=H, I=I, zipf=zipf)
        X = si.gen_tokens(14, 0, 7, layer.spec)
        Y, infos = oracle.moe_tokens(layer, X)
        for t in range(len(X)):
            yp, S, w = _py_layer(layer, X[t])
            assert list(infos[t].ids) == S
            assert np.allclose(infos[t].weights, w, rtol=0, atol=1e-14)
            assert np.allclose(Y[t], yp, rtol=1e-11, atol=1e-14)
        forced = np.array([[5, 0]] * len(X))
        Yf, _ = oracle.moe_tokens(layer, X, ids=forced)
        for t in range(len(X)):
            yt, _ = oracle.moe_token(layer, X[t], ids=forced[t])
            assert np.allclose(Yf[t], yt, rtol=1e-12, atol=1e-15)


def pin_permutation_equivariance():
    """Relabelling the experts (router rows moved with them) leaves y unchanged."""
    layer = tiny_layer(seed=12, E=10, k=3, H=64, I=64)
    perm = np.random.default_rng(1).permutation(10)
    inv = np.argsort(perm)
    r2 = Router("f32", w=layer.router.w[perm].copy())
    l2 = Layer(layer.spec, r2, [layer.experts[int(p)] for p in perm], layer.shared)
    for t in range(3):
        x = si.gen_tokens(12, t, 1, layer.spec)[0]
        y1, i1 = oracle.moe_token(layer, x)
        y2, i2 = oracle.moe_token(l2, x)
        assert sorted(int(perm[i]) for i in i2.ids) == sorted(int(i) for i in i1.ids)
        assert np.allclose(y1, y2, rtol=1e-12, atol=1e-15)
        assert set(int(inv[i]) for i in i1.ids) == set(int(i) for i in i2.ids)


def pin_bf16_input():
    """bf16 activations are read exactly: the oracle on bf16 bits equals it on the f32 values."""
    spec_b = LayerSpec(hidden=64, inter=64, n_experts=6, top_k=2, act="bf16")
    layer_b = si.gen_layer(13, 0, spec_b)
    xb = si.gen_tokens(13, 0, 1, spec_b)[0]
    xf = si.bf16_bits_to_f32(xb)
    layer_f = Layer(LayerSpec(hidden=64, inter=64, n_experts=6, top_k=2, act="f32"),
                    layer_b.router, layer_b.experts, layer_b.shared)
    yb, _ = oracle.moe_token(layer_b, xb)
    yf, _ = oracle.moe_token(layer_f, xf)
    assert np.array_equal(yb, yf)
    # a value pinned by hand: bf16 0x3FC0 = 1.5, 0xC0A0 = -5.0
    assert list(oracle.bf16_bits_to_f64(np.array([0x3FC0, 0xC0A0], np.uint16))) == [1.5, -5.0]


def pin_lfu_prefetch_trace():
    slots, rows = read_lfu_prefetch()
    c = oracle.LFUCache(slots)
    for op, ids, want, fills in rows:
        got, f = (c.access if op == "token" else c.prefetch)(ids)
        assert got == want, (op, ids, got, want)
        assert [tuple(v) for v in f] == fills, (op, ids, f, fills)


def pin_lfu_pinned_trace():
    slots, rows = read_lfu_pinned()
    c = oracle.LFUCache(slots)
    for row in rows:
        if row[0] == "pin":
            c.pin(row[1])
        elif row[0] == "hottest":
            assert c.hottest(row[1]) == row[2], (row, c.hottest(row[1]))
        else:
            h, f = c.access(row[1])
            assert h == row[2], (row, h)
            assert [tuple(v) for v in f] == row[3], (row, f)


def pin_lfu_trace():
    slots, rows = read_lfu()
    c = oracle.LFUCache(slots)
    for ids, hits, fills in rows:
        h, f = c.access(ids)
        assert h == hits, (ids, h, hits)
        assert [tuple(v) for v in f] == fills, (ids, f, fills)


def read_sigmoid_cases():
    """Hand-worked sigmoid router cases (tests/golden/sigmoid_router.txt)."""
    cases, cur = [], None
    for raw in open(os.path.join(GOLDEN, "sigmoid_router.txt")):
        line = raw.strip()
        if not line or line.startswith("#"):
            continue
        tok = line.split()
        if tok[0] == "case":
            cur = {"name": tok[1], "bias": {}}
            cases.append(cur)
        elif tok[0] == "k":
            cur["k"] = int(tok[1])
        elif tok[0] == "scale":
            cur["scale"] = Fraction(tok[1])
        elif tok[0] == "logit":
            lg = {}
            for t in tok[1:]:
                e, v = t.split("=")
                if v == "0":
                    lg[int(e)] = 0.0
                else:
                    sign = -1.0 if v.startswith("-") else 1.0
                    lg[int(e)] = sign * math.log(float(Fraction(v.lstrip("-").split(":")[1])))
            cur["logits"] = np.array([lg[e] for e in range(len(lg))])
        elif tok[0] == "bias":
            for t in tok[1:]:
                e, v = t.split("=")
                cur["bias"][int(e)] = float(v)
        elif tok[0] == "ids":
            cur["ids"] = [int(v) for v in tok[1:]]
        elif tok[0] == "w":
            cur["w"] = [Fraction(v) for v in tok[1:]]
    for c in cases:
        E = len(c["logits"])
        c["bias"] = np.array([c["bias"].get(e, 0.0) for e in range(E)], np.float32)
    return cases


def _sigmoid_layer(seed=14, E=10, k=3, H=64, I=64, scale=2.5, bias_sd=0.05):
    spec = LayerSpec(hidden=H, inter=I, n_experts=E, top_k=k, act="f32", router_score="sigmoid",
                     routed_scaling=scale, score_bias_sd=bias_sd)
    return si.gen_layer(seed, 0, spec)


def pin_sigmoid_router_golden():
    """The sigmoid scoring steps against the hand-worked cases."""
    for c in read_sigmoid_cases():
        layer = Layer(LayerSpec(hidden=64, inter=64, n_experts=len(c["logits"]), top_k=c["k"],
                                router_score="sigmoid", routed_scaling=float(c["scale"])),
                      None, [], None, router_bias=c["bias"])
        key, sc = oracle.moe.route_keys(layer, c["logits"])
        ids, _ = oracle.select_topk(key, c["k"])
        assert list(ids) == c["ids"], (c["name"], list(ids))
        w = oracle.moe._weights(layer, key, sc, ids)
        assert np.allclose(w, [float(v) for v in c["w"]], rtol=0, atol=1e-14), (c["name"], w)


def pin_sigmoid_layer_pure_python():
    """A tiny sigmoid-scored layer equals the pure-Python restatement; the weights
    sum to the scaling factor; without a bias the selection is the softmax one."""
    for seed, scale in ((14, 2.5), (15, 1.0)):
        layer = _sigmoid_layer(seed=seed, scale=scale)
        for t in range(3):
            x = si.gen_tokens(seed, t, 1, layer.spec)[0]
            y, info = oracle.moe_token(layer, x)
            yp, S, w = _py_layer(layer, x)
            assert list(info.ids) == S
            assert np.allclose(info.weights, w, rtol=0, atol=1e-14)
            assert abs(info.weights.sum() - scale) < 1e-12
            assert np.allclose(y, yp, rtol=1e-11, atol=1e-14)
    layer = _sigmoid_layer(seed=16, bias_sd=None)
    soft = Layer(LayerSpec(hidden=64, inter=64, n_experts=10, top_k=3, act="f32"), layer.router,
                 layer.experts, layer.shared)
    for t in range(5):
        x = si.gen_tokens(16, t, 1, layer.spec)[0]
        _, a = oracle.moe_token(layer, x)
        _, b = oracle.moe_token(soft, x)
        assert list(a.ids) == list(b.ids)


ALL_PINS = [pin_dequant_q4_table, pin_dequant_q2_table, pin_q2_layer, pin_dequant_q8_table, pin_format_sizes,
            pin_zero_input_routing, pin_topk_is_full_sort, pin_routing_weights,
            pin_silu, pin_ffn_closed_form, pin_dense_brute_force, pin_pure_python, pin_chunk_rows,
            pin_permutation_equivariance, pin_bf16_input, pin_lfu_trace, pin_lfu_prefetch_trace,
            pin_lfu_pinned_trace,
            pin_sigmoid_router_golden,
            pin_sigmoid_layer_pure_python]
