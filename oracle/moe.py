"""fp64 oracle of the routed Mixture-of-Experts FFN step (test infrastructure).

Every function states the passage of the pages it follows. The pages are:
  * "Inferno" README (GLM-5.2 Q2 on Apple Silicon) -- sections "Current
    Scope", "Model", "Memory Strategy";
  * GeekNews article on TurboFieldfare (Gemma 4 26B-A4B) -- sections
    "execution architecture" (weight format) and "token generation" (router,
    LFU cache, shared expert, combine, prefill chunk);
  * "Colibri" analysis report -- section 2 "Exact Architecture and Data-Flow
    Reconstruction" (Route / Union / Place / Overlap) and section 3 (exact
    routing);
  * Colibri README -- "What's implemented" (batch-union MoE, dequant-on-use,
    the DeepSeek-V3-style sigmoid router).

What the pages leave open is filled with the plainest reading, recorded where
it is used (nibble order, softmax renormalised over the selected experts,
ties to the lower index, LFU details, the sigmoid router's bias and scaling).

Everything here is computed in float64 with numpy; no blocking, fusion or
reordering beyond the definitions. Parity status: every function below is
pinned by tests in ``tests/test_oracle_pins.py`` (hand-computed values,
closed forms, brute force and an independent pure-Python restatement).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------

def f16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """IEEE binary16 bit patterns -> float64 (exact)."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns -> float64 (exact): the upper half of a binary32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def _affine_g64(q: np.ndarray, scale: np.ndarray, bias: np.ndarray) -> np.ndarray:
    """W[n][k] = q[n][k] * s[n][k // 64] + b[n][k // 64] for integer codes q
    [N][K], with the binary16 scale and bias of each group of 64 along k
    (exact in float64: a code times a binary16 plus a binary16)."""
    N, K = q.shape
    s = f16_bits_to_f64(scale).reshape(N, K // 64, 1)
    b = f16_bits_to_f64(bias).reshape(N, K // 64, 1)
    return (q.reshape(N, K // 64, 64) * s + b).reshape(N, K)


def dequant_q4g64(codes: np.ndarray, scale: np.ndarray, bias: np.ndarray) -> np.ndarray:
    """Affine group-64 4-bit dequantisation, W[n][k] = code(n,k) * s[n][k//64] + b[n][k//64].

    Follows TurboFieldfare "execution architecture" (MLX affine 4-bit, group
    64; the shared and routed experts are 4-bit) and Colibri README
    "dequant-on-use". Storage reading (the pages are silent): codes are
    row-major [N][K/2] bytes, element k in byte k//2, low nibble for even k;
    scale and bias are binary16 [N][K/64]. The fp64 result is exact.
    """
    codes = np.asarray(codes, dtype=np.uint8)
    N, half_k = codes.shape
    K = 2 * half_k
    q = np.empty((N, half_k, 2), dtype=np.uint8)   # q[n][k // 2][k % 2]
    q[:, :, 0] = codes & 0x0F
    q[:, :, 1] = codes >> 4
    return _affine_g64(q.reshape(N, K), scale, bias)


def dequant_q2g64(codes: np.ndarray, scale: np.ndarray, bias: np.ndarray) -> np.ndarray:
    """Affine group-64 2-bit dequantisation, W[n][k] = code(n,k) * s[n][k//64] + b[n][k//64].

    Inferno README ("Model"): the routed experts of the GLM-5.2 file it runs are
    2-bit (Q2); Colibri README ("What's implemented"): packed int2 kernels with
    dequant-on-use. Neither prints the layout; the reading here is the 2-bit
    sibling of the 4-bit format: codes row-major [N][K/4] bytes, element k at
    bits 2*(k % 4) of byte k//4 (low bits first); scale and bias binary16
    [N][K/64]. The fp64 result is exact.
    """
    codes = np.asarray(codes, dtype=np.uint8)
    N, quarter_k = codes.shape
    K = 4 * quarter_k
    q = np.empty((N, quarter_k, 4), dtype=np.uint8)   # q[n][k // 4][k % 4]
    for j in range(4):
        q[:, :, j] = (codes >> (2 * j)) & 0x03
    return _affine_g64(q.reshape(N, K), scale, bias)


def dequant_q8g64(codes: np.ndarray, scale: np.ndarray, bias: np.ndarray) -> np.ndarray:
    """Affine group-64 8-bit dequantisation, W[n][k] = code(n,k) * s[n][k//64] + b[n][k//64].

    TurboFieldfare "execution architecture": the router is stored at 8 bits in
    the same affine group-64 scheme. codes are row-major [N][K] bytes.
    """
    return _affine_g64(np.asarray(codes, dtype=np.uint8), scale, bias)


def router_weights_f64(router) -> np.ndarray:
    """Router matrix [E][H] in float64: fp32 values, or the dequantised 8-bit codes."""
    if router.fmt == "f32":
        return np.asarray(router.w, dtype=np.float32).astype(np.float64)
    q = router.q
    return dequant_q8g64(q.codes, q.scale, q.bias)


# ---------------------------------------------------------------------------
# routing
# ---------------------------------------------------------------------------

def router_logits(Wr: np.ndarray, x: np.ndarray, bias: np.ndarray | None = None) -> np.ndarray:
    """l_e = sum_k Wr[e][k] x[k] (+ bias_e).

    TurboFieldfare "token generation": the router runs on the GPU with weights
    that always stay in memory; Colibri report section 2 "Route": the resident
    routing matrix scores the token's hidden state. The optional per-expert
    bias (skewed popularity workload) is added to the logits before selection
    and before the softmax.
    """
    l = Wr @ np.asarray(x, dtype=np.float64)
    if bias is not None:
        l = l + np.asarray(bias, dtype=np.float32).astype(np.float64)
    return l


@dataclass
class RouteInfo:
    ids: np.ndarray        # int64 [k], selection order
    weights: np.ndarray    # float64 [k]
    gap: float             # l_(k) - l_(k+1) (inf when k == E)
    scale: float           # sum_i |Wr[e][i] x[i]| max over e (fp32 rounding scale)


def select_topk(l: np.ndarray, k: int) -> tuple[np.ndarray, float]:
    """Exact top-k: the first k of the experts stably sorted by (-l_e, e).

    Inferno "Current Scope" and Colibri report section 3: exact top-8 routing,
    no approximation. Ties go to the lower expert index (stable sort on the
    negated logits). Also returns the gap between the k-th and (k+1)-th
    largest logits.
    """
    order = np.argsort(-np.asarray(l, dtype=np.float64), kind="stable")
    ids = order[:k]
    gap = float(l[order[k - 1]] - l[order[k]]) if k < len(l) else float("inf")
    return ids.astype(np.int64), gap


def routing_weights(l_sel: np.ndarray) -> np.ndarray:
    """Softmax over the selected logits: w_j = exp(l_j - max) / sum_j' exp(l_j' - max).

    A full softmax over all experts renormalised over the selected ones is the
    same quantity; the pages name softmax top-8 with renormalised weights only
    through the benchmark spec, so this is the plainest reading.
    """
    l_sel = np.asarray(l_sel, dtype=np.float64)
    e = np.exp(l_sel - l_sel.max())
    return e / e.sum()


def sigmoid_scores(l: np.ndarray) -> np.ndarray:
    """s_e = 1 / (1 + exp(-l_e)), in float64.

    Colibri README, "What's implemented": the model's router is a
    DeepSeek-V3-style sigmoid router (noaux_tc, routed_scaling_factor). The
    pages name it only; the reading used here: each expert's score is the
    logistic function of its logit.
    """
    return 1.0 / (1.0 + np.exp(-np.asarray(l, dtype=np.float64)))


def sigmoid_keys(s: np.ndarray, bias: np.ndarray | None) -> np.ndarray:
    """Selection keys of the sigmoid router: key_e = s_e + bias_e.

    Reading of "noaux_tc" (Colibri README, "What's implemented"): the
    per-expert bias steers which experts are selected and takes no part in the
    routing weights; all experts form one group.
    """
    key = np.asarray(s, dtype=np.float64).copy()
    if bias is not None:
        key = key + np.asarray(bias, dtype=np.float32).astype(np.float64)
    return key


def routing_weights_sigmoid(s_sel: np.ndarray, routed_scaling: float) -> np.ndarray:
    """w_j = routed_scaling * s_j / sum_j' s_j' over the selected experts.

    Colibri README, "What's implemented" (routed_scaling_factor). Reading: the
    selected sigmoid scores (without the bias) are renormalised to sum to one
    and then multiplied by the scaling factor.
    """
    s_sel = np.asarray(s_sel, dtype=np.float64)
    return float(routed_scaling) * s_sel / s_sel.sum()


def route_keys(layer, l: np.ndarray) -> tuple[np.ndarray, np.ndarray | None]:
    """(selection keys, sigmoid scores or None) for the layer's router scoring.

    softmax scoring: the keys are the logits with the bias already added by
    ``router_logits``. sigmoid scoring: ``l`` must be the unbiased logits.
    """
    if getattr(layer.spec, "router_score", "softmax") == "sigmoid":
        sc = sigmoid_scores(l)
        return sigmoid_keys(sc, layer.router_bias), sc
    return np.asarray(l, dtype=np.float64), None


def _weights(layer, key: np.ndarray, sc: np.ndarray | None, ids: np.ndarray) -> np.ndarray:
    if sc is None:
        return routing_weights(key[ids])
    return routing_weights_sigmoid(sc[ids], layer.spec.routed_scaling)


def _logits(layer, Wr: np.ndarray, x64: np.ndarray) -> np.ndarray:
    """The router logits: biased for softmax scoring, unbiased for sigmoid."""
    sigmoid = getattr(layer.spec, "router_score", "softmax") == "sigmoid"
    return router_logits(Wr, x64, None if sigmoid else layer.router_bias)


# ---------------------------------------------------------------------------
# expert FFN and the layer
# ---------------------------------------------------------------------------

def silu(z: np.ndarray) -> np.ndarray:
    """silu(z) = z / (1 + exp(-z)), written to avoid overflow for very negative z."""
    z = np.asarray(z, dtype=np.float64)
    out = np.empty_like(z)
    pos = z >= 0
    out[pos] = z[pos] / (1.0 + np.exp(-z[pos]))
    ez = np.exp(z[~pos])
    out[~pos] = z[~pos] * ez / (1.0 + ez)
    return out


def _deq(m) -> np.ndarray:
    if getattr(m, "bits", 4) == 2:
        return dequant_q2g64(m.codes, m.scale, m.bias)
    return dequant_q4g64(m.codes, m.scale, m.bias)


def expert_ffn(expert, x: np.ndarray) -> np.ndarray:
    """f(x) = W_down (silu(W_gate x) * (W_up x)), each matrix dequantised on use.

    Inferno "Model": each routed expert is a gate, an up and a down matrix;
    the gated (SwiGLU) form is the plainest reading of gate/up/down.
    """
    x = np.asarray(x, dtype=np.float64)
    g = _deq(expert.gate) @ x
    u = _deq(expert.up) @ x
    h = silu(g) * u
    return _deq(expert.down) @ h


def _x_f64(layer, x) -> np.ndarray:
    if layer.spec.act == "bf16":
        return bf16_bits_to_f64(x)
    return np.asarray(x, dtype=np.float32).astype(np.float64)


def route_token(layer, x64: np.ndarray, Wr: np.ndarray | None = None) -> RouteInfo:
    """Selection and weights of one token under the layer's router scoring
    (gap: between the k-th and (k+1)-th selection keys)."""
    if Wr is None:
        Wr = router_weights_f64(layer.router)
    key, sc = route_keys(layer, _logits(layer, Wr, x64))
    ids, gap = select_topk(key, layer.spec.top_k)
    w = _weights(layer, key, sc, ids)
    scale = float(np.max(np.abs(Wr * x64[None, :]).sum(axis=1)))
    return RouteInfo(ids, w, gap, scale)


def moe_token(layer, x, ids: np.ndarray | None = None, Wr: np.ndarray | None = None):
    """One decode token: y = f_shared(x) + sum_j w_j f_{S_j}(x).

    TurboFieldfare "token generation": the router picks the top-8 experts; the
    always-resident shared expert runs on every token; after the routed
    experts run, the shared and routed outputs are combined. Colibri report
    section 2: Route, then the experts. The shared expert is unweighted.

    ``ids`` overrides the selection (used when the GPU's fp32 logits resolve a
    near-tie the other way; the weights are then those of the layer's scoring
    over those ids).
    Returns (y float64 [H], RouteInfo).
    """
    x64 = _x_f64(layer, x)
    if Wr is None:
        Wr = router_weights_f64(layer.router)
    info = route_token(layer, x64, Wr)
    if ids is not None:
        key, sc = route_keys(layer, _logits(layer, Wr, x64))
        ids = np.asarray(ids, dtype=np.int64)
        info = RouteInfo(ids, _weights(layer, key, sc, ids), info.gap, info.scale)
    y = np.zeros(layer.spec.hidden, dtype=np.float64)
    if layer.shared is not None:
        y += expert_ffn(layer.shared, x64)
    for j, e in enumerate(info.ids):
        y += info.weights[j] * expert_ffn(layer.experts[int(e)], x64)
    return y, info


def moe_tokens(layer, X, ids: np.ndarray | None = None):
    """A chunk of tokens (prefill): row t is exactly the decode of token t.

    TurboFieldfare "token generation" (prefill in chunks of up to 128 tokens
    so a fetched expert serves several rows) and Colibri "Union" / batch-union
    MoE (each distinct expert of the batch read once, applied to every row
    routed to it): both are execution strategies; the rows are independent.

    Every row is ``moe_token`` of that token (same selection, weights and
    order of the sum: shared first, then the slots in selection order); the
    only difference is that each expert is dequantised once for all the rows
    that selected it, and its gate/up/down products for those rows are one
    matrix product each. Returns (Y float64 [T][H], [RouteInfo] * T).
    """
    Wr = router_weights_f64(layer.router)
    T = len(X)
    X64 = np.stack([_x_f64(layer, X[t]) for t in range(T)])
    infos = []
    for t in range(T):
        info = route_token(layer, X64[t], Wr)
        if ids is not None:
            key, sc = route_keys(layer, _logits(layer, Wr, X64[t]))
            sel = np.asarray(ids[t], dtype=np.int64)
            info = RouteInfo(sel, _weights(layer, key, sc, sel), info.gap, info.scale)
        infos.append(info)

    def ffn_rows(expert, rows):   # f(x_t) for the given rows, one dequantisation
        Xs = X64[rows]
        g = Xs @ _deq(expert.gate).T
        u = Xs @ _deq(expert.up).T
        return (silu(g) * u) @ _deq(expert.down).T

    k = layer.spec.top_k
    F = np.zeros((T, k, layer.spec.hidden))          # F[t][j] = f_{S_j}(x_t)
    users = {}
    for t in range(T):
        for j, e in enumerate(infos[t].ids):
            users.setdefault(int(e), []).append((t, j))
    for e, tj in users.items():
        out = ffn_rows(layer.experts[e], [t for t, _ in tj])
        for (t, j), row in zip(tj, out):
            F[t, j] = row
    Y = ffn_rows(layer.shared, list(range(T))) if layer.shared is not None else np.zeros((T, layer.spec.hidden))
    for t in range(T):
        for j in range(k):
            Y[t] += infos[t].weights[j] * F[t, j]
    return Y, infos


def layer_dense_f64(layer, x) -> np.ndarray:
    """Brute force: evaluate every expert densely, then mask to the selected set.

    Used only to pin ``moe_token``: the same output obtained without the
    sparse dispatch, weights taken from the full softmax renormalised over S.
    """
    x64 = _x_f64(layer, x)
    Wr = router_weights_f64(layer.router)
    l = router_logits(Wr, x64, layer.router_bias)
    E, k = layer.spec.n_experts, layer.spec.top_k
    p = np.exp(l - l.max())
    p /= p.sum()
    S = set(int(i) for i in np.argsort(-l, kind="stable")[:k])
    mask = np.array([1.0 if e in S else 0.0 for e in range(E)])
    pm = p * mask
    pm /= pm.sum()
    outs = np.stack([expert_ffn(layer.experts[e], x64) for e in range(E)])
    y = pm @ outs
    if layer.shared is not None:
        y = y + expert_ffn(layer.shared, x64)
    return y


# ---------------------------------------------------------------------------
# per-layer LFU expert cache (residency trace)
# ---------------------------------------------------------------------------

class LFUCache:
    """Per-layer expert cache with a fixed number of slots, least-frequently-used eviction.

    TurboFieldfare "token generation": the CPU matches the router's 8 expert
    IDs against a 16-slot LFU cache per layer and fills the misses. Readings
    (the pages are silent on the details):
      * an expert's count starts at 1 when it is admitted and grows by 1 on
        every use while it stays resident; the count is dropped on eviction;
      * the victim is the resident expert with the smallest count that the
        current token does not need; ties go to the least recently used, then
        to the lower expert index;
      * the IDs of one token are processed in selection order; hits are
        counted before any miss of the same token is admitted.
    """

    def __init__(self, slots: int):
        self.slots = slots
        self.count: dict[int, int] = {}
        self.last: dict[int, int] = {}
        self.slot_of: dict[int, int] = {}
        self.clock = 0
        self.pinned: frozenset = frozenset()
        self.usage: dict[int, int] = {}

    def pin(self, experts) -> None:
        """Replace the set of pinned experts (the learning cache).

        Colibri README, "Self-learning cache" / "The learning cache": the
        engine records which experts the usage routes to and pins the hottest
        ones in spare memory. Readings (the page gives the idea, not the
        bookkeeping): a pinned expert is always resident outside the LFU
        slots, so its lookups are hits that leave the LFU state alone; pinning
        an expert that holds a slot frees that slot (its count and recency are
        dropped); an expert that stops being pinned is not resident until a
        token stages it again. Pinning is not a token: the clock stays.
        """
        new = frozenset(int(e) for e in experts)
        for e in new:
            if e in self.count:
                del self.slot_of[e]
                del self.count[e]
                del self.last[e]
        self.pinned = new

    def hottest(self, n: int) -> list[int]:
        """The n experts used most often so far (ties: the lower id first)."""
        order = sorted(self.usage, key=lambda e: (-self.usage[e], e))
        return order[:n]

    def access(self, ids) -> tuple[list[int], list[tuple[int, int, int]]]:
        """Process one token's expert IDs.

        Returns (hits, fills) where fills lists (expert, slot, evicted expert
        or -1) in the order the misses are admitted.
        """
        ids = [int(e) for e in ids]
        assert len(set(ids)) == len(ids)
        assert len([e for e in ids if e not in self.pinned]) <= self.slots
        self.clock += 1
        need = set(ids)
        hits, fills = [], []
        for e in ids:
            self.usage[e] = self.usage.get(e, 0) + 1
            if e in self.pinned:
                hits.append(e)
            elif e in self.count:
                hits.append(e)
                self.count[e] += 1
                self.last[e] = self.clock
        for e in ids:
            if e in self.count or e in self.pinned:
                continue
            if len(self.count) < self.slots:
                used = set(self.slot_of.values())
                slot = min(s for s in range(self.slots) if s not in used)
                victim = -1
            else:
                cands = [r for r in self.count if r not in need]
                victim = min(cands, key=lambda r: (self.count[r], self.last[r], r))
                slot = self.slot_of.pop(victim)
                del self.count[victim]
                del self.last[victim]
            self.count[e] = 1
            self.last[e] = self.clock
            self.slot_of[e] = slot
            fills.append((e, slot, victim))
        return hits, fills


    def prefetch(self, ids) -> tuple[list[int], list[tuple[int, int, int]]]:
        """Admit a prediction (router lookahead).

        Colibri analysis report, caching and prefetch: passing the state that
        enters layer L through the router of layer L + 1 predicts that
        layer's experts one layer ahead, and the predicted weights are loaded
        while layer L computes. Readings (the page describes the prediction,
        not its bookkeeping): a predicted expert that is not resident is
        admitted with count 0, since it has not been used; residents keep
        their counts and recency; victims follow the same rule as ``access``,
        taken outside the prediction. Returns (predicted experts already
        resident, fills).
        """
        ids = [int(e) for e in ids]
        assert len(set(ids)) == len(ids)
        assert len([e for e in ids if e not in self.pinned]) <= self.slots
        self.clock += 1
        pred = set(ids)
        resident = [e for e in ids if e in self.count or e in self.pinned]
        fills = []
        for e in ids:
            if e in self.count or e in self.pinned:
                continue
            if len(self.count) < self.slots:
                used = set(self.slot_of.values())
                slot = min(s for s in range(self.slots) if s not in used)
                victim = -1
            else:
                cands = [r for r in self.count if r not in pred]
                victim = min(cands, key=lambda r: (self.count[r], self.last[r], r))
                slot = self.slot_of.pop(victim)
                del self.count[victim]
                del self.last[victim]
            self.count[e] = 0
            self.last[e] = self.clock
            self.slot_of[e] = slot
            fills.append((e, slot, victim))
        return resident, fills


def lfu_trace(id_rows, slots: int):
    """Hit/miss trace of a sequence of tokens through one LFU cache."""
    c = LFUCache(slots)
    out = []
    for ids in id_rows:
        out.append(c.access(ids))
    return out
