"""Parity helpers: compare the CUDA library's outputs with the fp64 oracle.

Tolerances:
  * expert IDs are compared exactly, except where the oracle's fp64 logits put
    the k-th and (k+1)-th experts (or two selected experts) within TAU * sigma
    of each other, sigma = max_e sum_i |W_r[e][i] x_i| + |bias_e|; there the fp32
    router may resolve the tie either way, so the GPU's selection is checked
    for validity and the output is compared with the oracle run on the GPU's
    selection. TAU = 2^-16 bounds the fp32 summation error of the router
    (< 200 sequential fp32 additions per partial sum, each within 2^-24).
    With sigmoid scoring the keys are s + bias: a key moves by at most a
    quarter of its logit's error plus SIGMOID_EPS = 2^-20 for the fp32
    exponential, division and addition.
  * routing weights: absolute 1e-5 (fp32 softmax of fp32 logits, or fp32
    sigmoid scores renormalised and scaled).
  * layer output: max_i |y_i - yhat_i| / max_i |yhat_i| <= 2e-3 per token on
    the fp32 output, and the bf16 output equals the fp32 output rounded to
    nearest even.
"""
from __future__ import annotations

import numpy as np

import oracle

TAU = 2.0 ** -16
SIGMOID_EPS = 2.0 ** -20
REL_TOL = 2e-3
W_TOL = 1e-5


def f32_to_bf16_rne(a: np.ndarray) -> np.ndarray:
    u = np.asarray(a, np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    return r


def check_selection(layer, x, ids_gpu, Wr=None):
    """Returns (ids_to_use, flagged). Raises AssertionError if the GPU selection is invalid."""
    if Wr is None:
        Wr = oracle.router_weights_f64(layer.router)
    x64 = oracle.moe._x_f64(layer, x)
    sigmoid = getattr(layer.spec, "router_score", "softmax") == "sigmoid"
    # selection keys: biased logits, or sigmoid scores plus the bias
    l, _ = oracle.route_keys(layer, oracle.moe._logits(layer, Wr, x64))
    k = layer.spec.top_k
    ids_o, _ = oracle.select_topk(l, k)
    sigma = float(np.max(np.abs(Wr * x64[None, :]).sum(axis=1)))
    if layer.router_bias is not None and not sigmoid:
        sigma += float(np.max(np.abs(layer.router_bias)))
    # a sigmoid key moves by at most 1/4 of its logit's error, plus the fp32
    # rounding of the exponential, the division and the bias addition
    tau = TAU * sigma * 0.25 + SIGMOID_EPS if sigmoid else TAU * sigma
    ids_g = [int(v) for v in ids_gpu]
    if ids_g == [int(v) for v in ids_o]:
        return ids_o, False
    # validity: distinct, in range, and every unselected expert's logit is not
    # above any selected one by more than tau; the order within the selection
    # descends up to tau
    E = len(l)
    assert len(set(ids_g)) == k and all(0 <= e < E for e in ids_g), ids_g
    sel = set(ids_g)
    lmin_sel = min(l[e] for e in ids_g)
    lmax_unsel = max((l[e] for e in range(E) if e not in sel), default=-np.inf)
    assert lmax_unsel <= lmin_sel + tau, (ids_g, list(ids_o), lmax_unsel - lmin_sel, tau)
    for a, b in zip(ids_g, ids_g[1:]):
        assert l[a] >= l[b] - tau, (ids_g, l[a] - l[b])
    return np.array(ids_g, np.int64), True


def compare_token(layer, x, y32, ids_gpu, w_gpu, y_out=None, Wr=None, y_bf16=None):
    """Check one token; returns (normwise error, flagged)."""
    ids_use, flagged = check_selection(layer, x, ids_gpu, Wr)
    y_ref, info = oracle.moe_token(layer, x, ids=ids_use if flagged else None, Wr=Wr)
    assert np.allclose(np.asarray(w_gpu, np.float64), info.weights, rtol=0, atol=W_TOL), (w_gpu, info.weights)
    y32 = np.asarray(y32, np.float64)
    err = float(np.max(np.abs(y32 - y_ref)) / max(np.max(np.abs(y_ref)), 1e-30))
    assert err <= REL_TOL, err
    if y_bf16 is not None:
        assert np.array_equal(np.asarray(y_bf16, np.uint16), f32_to_bf16_rne(np.asarray(y32, np.float32)))
    return err, flagged


def compare_chunk(layer, X, y32, ids_gpu, w_gpu, y_bf16=None, Wr=None):
    """Check every row of a chunk (T tokens) at once; returns (max normwise
    error, near-tie rows). Each row's GPU selection is checked as in
    compare_token, then the oracle evaluates all rows on those (validated)
    selections with each expert dequantised once (oracle.moe_tokens)."""
    if Wr is None:
        Wr = oracle.router_weights_f64(layer.router)
    T = len(X)
    use, flagged = [], 0
    for t in range(T):
        u, fl = check_selection(layer, X[t], ids_gpu[t], Wr)
        use.append(np.asarray(u, np.int64))
        flagged += fl
    Y, infos = oracle.moe_tokens(layer, X, ids=np.stack(use))
    worst = 0.0
    for t in range(T):
        assert np.allclose(np.asarray(w_gpu[t], np.float64), infos[t].weights, rtol=0, atol=W_TOL), \
            (t, w_gpu[t], infos[t].weights)
        err = float(np.max(np.abs(np.asarray(y32[t], np.float64) - Y[t])) / max(np.max(np.abs(Y[t])), 1e-300))
        assert err <= REL_TOL, (t, err)
        if y_bf16 is not None:
            assert np.array_equal(np.asarray(y_bf16[t], np.uint16), f32_to_bf16_rne(np.asarray(y32[t], np.float32))), t
        worst = max(worst, err)
    return worst, flagged
