"""The fp64 oracle against facts fixed outside itself (CPU only).

Every pin runs on the oracle as it stands; then a list of plausible mistakes
is planted in the oracle (monkeypatched, on the CPU) and each must make at
least one pin fail.
"""
import numpy as np
import pytest

import oracle
import oracle.moe as om
import _pins

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


@pytest.mark.parametrize("pin", _pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


# --- planted mistakes --------------------------------------------------------

_real = {name: getattr(om, name) for name in
         ("dequant_q4g64", "dequant_q2g64", "dequant_q8g64", "routing_weights", "select_topk",
          "silu", "expert_ffn", "router_logits", "moe_token", "sigmoid_keys",
          "routing_weights_sigmoid", "route_keys", "sigmoid_scores")}


def _deq_swapped_nibbles(codes, scale, bias):
    codes = np.asarray(codes, np.uint8)
    swapped = ((codes & 0x0F) << 4) | (codes >> 4)
    return _real["dequant_q4g64"](swapped.astype(np.uint8), scale, bias)


def _deq_bias_sign(codes, scale, bias):
    return _real["dequant_q4g64"](codes, scale, np.asarray(bias, np.uint16) ^ np.uint16(0x8000))


def _deq_group_32(codes, scale, bias):
    codes = np.asarray(codes, np.uint8)
    N, hk = codes.shape
    K = 2 * hk
    q = np.empty((N, K))
    q[:, 0::2] = codes & 15
    q[:, 1::2] = codes >> 4
    s = om.f16_bits_to_f64(scale).reshape(N, -1)
    b = om.f16_bits_to_f64(bias).reshape(N, -1)
    idx = np.minimum(np.arange(K) // 32, s.shape[1] - 1)
    return q * s[:, idx] + b[:, idx]


def _q8_no_bias(codes, scale, bias):
    return _real["dequant_q8g64"](codes, scale, np.zeros_like(np.asarray(bias)))


def _weights_unnormalised(l_sel):
    l_sel = np.asarray(l_sel, np.float64)
    return np.exp(l_sel - l_sel.max())


def _topk_ties_high(l, k):
    l = np.asarray(l, np.float64)
    order = np.lexsort((-np.arange(len(l)), -l))
    gap = float(l[order[k - 1]] - l[order[k]]) if k < len(l) else float("inf")
    return order[:k].astype(np.int64), gap


def _silu_is_sigmoid(z):
    z = np.asarray(z, np.float64)
    return 1.0 / (1.0 + np.exp(-z))


def _ffn_gate_up_swapped(expert, x):
    x = np.asarray(x, np.float64)
    g = om._deq(expert.gate) @ x
    u = om._deq(expert.up) @ x
    return om._deq(expert.down) @ (om.silu(u) * g)


def _ffn_no_down(expert, x):
    x = np.asarray(x, np.float64)
    g = om._deq(expert.gate) @ x
    u = om._deq(expert.up) @ x
    h = om.silu(g) * u
    H = expert.down.N
    return np.resize(h, H)


def _logits_no_bias(Wr, x, bias=None):
    return _real["router_logits"](Wr, x, None)


def _token_weighted_shared(layer, x, ids=None, Wr=None):
    y, info = _real["moe_token"](layer, x, ids, Wr)
    if layer.shared is not None:
        x64 = om._x_f64(layer, x)
        y = y + (info.weights[0] - 1.0) * om.expert_ffn(layer.shared, x64)
    return y, info


def _token_no_shared(layer, x, ids=None, Wr=None):
    y, info = _real["moe_token"](layer, x, ids, Wr)
    if layer.shared is not None:
        y = y - om.expert_ffn(layer.shared, om._x_f64(layer, x))
    return y, info


def _deq2_fields_reversed(codes, scale, bias):
    codes = np.asarray(codes, np.uint8)
    rev = ((codes & 0x03) << 6) | ((codes & 0x0C) << 2) | ((codes & 0x30) >> 2) | ((codes & 0xC0) >> 6)
    return _real["dequant_q2g64"](rev.astype(np.uint8), scale, bias)


def _deq2_row_reversed(codes, scale, bias):
    return _real["dequant_q2g64"](codes, scale, bias)[:, ::-1]


def _sig_bias_dropped(s, bias):
    return _real["sigmoid_keys"](s, None)


def _sig_not_scaled(s_sel, routed_scaling):
    return _real["routing_weights_sigmoid"](s_sel, 1.0)


def _sig_weights_from_keys(layer, l):
    key, sc = _real["route_keys"](layer, l)
    return key, (None if sc is None else key)


class _LfuPrefetchCountsUse(om.LFUCache):
    def prefetch(self, ids):
        r, f = super().prefetch(ids)
        for e, _, _ in f:
            self.count[e] = 1
        return r, f


class _LfuPrefetchRefreshes(om.LFUCache):
    def prefetch(self, ids):
        r, f = super().prefetch(ids)
        for e in r:
            self.last[e] = self.clock
        return r, f


class _LfuPinnedCountsUse(om.LFUCache):
    """a pinned expert also enters an LFU slot when used"""
    def access(self, ids):
        pinned, self.pinned = self.pinned, frozenset()
        try:
            return super().access(ids)
        finally:
            self.pinned = pinned


class _LfuPinKeepsSlot(om.LFUCache):
    """pinning leaves the expert's slot taken"""
    def pin(self, experts):
        self.pinned = frozenset(int(e) for e in experts)


class _LfuUnpinKeepsResident(om.LFUCache):
    """an unpinned expert stays resident (a new pin only adds experts)"""
    def pin(self, experts):
        super().pin(set(int(e) for e in experts) | set(self.pinned))


class _LfuHottestTiesHigh(om.LFUCache):
    def hottest(self, n):
        return sorted(self.usage, key=lambda e: (-self.usage[e], -e))[:n]


def _sig_is_tanh(l):
    return np.tanh(np.asarray(l, np.float64))


MISTAKES = {
    "nibble order swapped": ("dequant_q4g64", _deq_swapped_nibbles),
    "bias sign flipped": ("dequant_q4g64", _deq_bias_sign),
    "group size 32": ("dequant_q4g64", _deq_group_32),
    "8-bit bias dropped": ("dequant_q8g64", _q8_no_bias),
    "weights not renormalised": ("routing_weights", _weights_unnormalised),
    "ties to the higher index": ("select_topk", _topk_ties_high),
    "silu replaced by sigmoid": ("silu", _silu_is_sigmoid),
    "gate and up swapped": ("expert_ffn", _ffn_gate_up_swapped),
    "down projection dropped": ("expert_ffn", _ffn_no_down),
    "router bias dropped": ("router_logits", _logits_no_bias),
    "shared expert weighted": ("moe_token", _token_weighted_shared),
    "shared expert dropped": ("moe_token", _token_no_shared),
    "2-bit fields read high bits first": ("dequant_q2g64", _deq2_fields_reversed),
    "2-bit row reversed": ("dequant_q2g64", _deq2_row_reversed),
    "sigmoid selection bias dropped": ("sigmoid_keys", _sig_bias_dropped),
    "sigmoid weights not scaled": ("routing_weights_sigmoid", _sig_not_scaled),
    "sigmoid bias in the weights": ("route_keys", _sig_weights_from_keys),
    "sigmoid replaced by tanh": ("sigmoid_scores", _sig_is_tanh),
    "prediction admitted as a use": ("LFUCache", _LfuPrefetchCountsUse),
    "prediction refreshes residents": ("LFUCache", _LfuPrefetchRefreshes),
    "pinned expert enters the LFU": ("LFUCache", _LfuPinnedCountsUse),
    "pinning keeps the slot": ("LFUCache", _LfuPinKeepsSlot),
    "unpinned expert stays resident": ("LFUCache", _LfuUnpinKeepsResident),
    "hottest ties to the higher id": ("LFUCache", _LfuHottestTiesHigh),
}


@pytest.mark.parametrize("name", list(MISTAKES))
def test_planted_mistake_is_caught(name, monkeypatch):
    attr, fake = MISTAKES[name]
    monkeypatch.setattr(om, attr, fake)
    if hasattr(oracle, attr):
        monkeypatch.setattr(oracle, attr, fake)
    failed = []
    for pin in _pins.ALL_PINS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake: {name}"
