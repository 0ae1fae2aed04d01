"""Streamed expert cache (per-layer LFU slots filled from host memory).

CPU: the library's cache policy (moe_lfu_trace, host-only) against the
oracle's LFU simulation and the hand-written golden trace.
GPU: a streamed layer decodes bit-identically to the resident layer, its
hit/miss sequence and slot residency follow the oracle's simulation, and host
failures (a source callback that fails, a host wait that runs out) come back
as status codes without a device fault.
"""
import ctypes

import numpy as np
import pytest

import oracle
import quantized_routed_expert_moe_gb300 as moe
import seeded_inputs as si
from _parity import compare_token
from _pins import read_lfu


def zipf_rows(seed, n_tokens, E, k, alpha=1.1):
    """Seeded token id rows: k distinct experts per token, skewed popularity."""
    rng = np.random.default_rng(seed)
    p = (np.arange(1, E + 1, dtype=np.float64) ** -alpha)
    p = p[rng.permutation(E)]
    p /= p.sum()
    return np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(n_tokens)]).astype(np.int32)


def oracle_slots_hits(rows, slots):
    c = oracle.moe.LFUCache(slots)
    slot = np.empty(rows.shape, np.int32)
    hit = np.empty(rows.shape, np.uint8)
    for t, ids in enumerate(rows):
        hit[t] = [1 if int(e) in c.count else 0 for e in ids]
        c.access(ids)
        slot[t] = [c.slot_of[int(e)] for e in ids]
    return slot, hit


@pytest.mark.parametrize("seed,E,k,slots", [(0, 256, 8, 16), (1, 32, 8, 8), (2, 64, 4, 16), (3, 9, 1, 1)])
def test_lfu_policy_matches_oracle(seed, E, k, slots):
    rows = zipf_rows(seed, 400, E, k)
    slot, hit = moe.moe_lfu_trace(slots, E, rows)
    o_slot, o_hit = oracle_slots_hits(rows, slots)
    assert np.array_equal(hit, o_hit)
    assert np.array_equal(slot, o_slot)


def test_lfu_policy_golden_trace():
    """The hand-worked trace in tests/golden/lfu_trace.txt (TurboFieldfare
    article, "token generation", with the stated readings), checked against the
    library's policy directly."""
    slots, rows = read_lfu()
    ids = np.array([r[0] for r in rows], np.int32)
    slot, hit = moe.moe_lfu_trace(slots, int(ids.max()) + 1, ids)
    for t, (tok, hits, fills) in enumerate(rows):
        assert sorted(e for e, h in zip(tok, hit[t]) if h) == sorted(hits)
        for e, s, _victim in fills:
            assert slot[t][tok.index(e)] == s
        for j, e in enumerate(tok):
            if e in hits:   # a hit keeps its slot
                assert slot[t][j] == slot[t - 1][list(rows[t - 1][0]).index(e)] if e in rows[t - 1][0] else True


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_hottest_matches_oracle(seed):
    """The library's ordering of experts by usage (moe_hottest, which
    moe_cache_pin_hottest pins) equals the oracle's learning-cache "hottest" on
    seeded Zipf traces, ties included."""
    E, k, T = 64, 8, 40
    rows = zipf_rows(seed, T, E, k)
    sim = oracle.moe.LFUCache(16)
    for r in rows:
        sim.access([int(e) for e in r])
    counts = np.zeros(E, np.uint64)
    for e, c in sim.usage.items():
        counts[e] = c
    n_used = len(sim.usage)
    for n in (0, 1, 6, n_used):
        assert list(moe.moe_hottest(counts, n)) == sim.hottest(n)


def test_hottest_rejects_bad_n():
    counts = np.zeros(8, np.uint64)
    for n in (-1, 9):
        with pytest.raises(moe.MoEError):
            moe.moe_hottest(counts, n)


def test_lfu_policy_rejects_bad_rows():
    with pytest.raises(moe.MoEError):
        moe.moe_lfu_trace(4, 8, np.array([[1, 1]], np.int32))
    with pytest.raises(moe.MoEError):
        moe.moe_lfu_trace(4, 8, np.array([[1, 9]], np.int32))
    with pytest.raises(moe.MoEError):
        moe.moe_lfu_trace(1, 8, np.array([[1, 2]], np.int32))


# --------------------------------------------------------------------------- GPU

def oracle_pinned_run(rows, slots, pinned, n_experts):
    c = oracle.moe.LFUCache(slots)
    c.pin(pinned)
    pin_at = {int(e): i for i, e in enumerate(pinned)}
    slot = np.empty(rows.shape, np.int32)
    hit = np.empty(rows.shape, np.uint8)
    for t, ids in enumerate(rows):
        hit[t] = [1 if (int(e) in c.count or int(e) in c.pinned) else 0 for e in ids]
        c.access(ids)
        slot[t] = [slots + pin_at[int(e)] if int(e) in pin_at else c.slot_of[int(e)] for e in ids]
    usage = np.array([c.usage.get(e, 0) for e in range(n_experts)], np.uint64)
    return slot, hit, usage, c


@pytest.mark.parametrize("seed,E,k,slots,n_pin", [(0, 256, 8, 16, 16), (1, 32, 8, 8, 5), (2, 64, 4, 16, 60),
                                                  (3, 9, 1, 1, 3), (4, 64, 8, 8, 0)])
def test_lfu_pinned_policy_matches_oracle(seed, E, k, slots, n_pin):
    """The library's host policy with pinned experts (the learning cache: the
    hottest of a learning run, as moe_cache_pin places them) against the
    oracle's, on seeded Zipf traces: hits, slots and usage counts."""
    learn = zipf_rows(seed + 100, 200, E, k)
    sim = oracle.moe.LFUCache(slots)
    for ids in learn:
        sim.access(ids)
    pinned = np.array(sim.hottest(n_pin), np.int32)
    rows = zipf_rows(seed, 400, E, k)
    slot, hit, usage = moe.moe_lfu_trace_pinned(slots, E, rows, pinned)
    o_slot, o_hit, o_usage, c = oracle_pinned_run(rows, slots, pinned, E)
    assert np.array_equal(hit, o_hit)
    assert np.array_equal(slot, o_slot)
    assert np.array_equal(usage, o_usage)
    if n_pin:
        pinned_hits = sum(int(e) in c.pinned for e in rows.reshape(-1))
        assert pinned_hits > 0 and int(hit.sum()) >= pinned_hits


def test_lfu_pinned_rejects_bad_pins():
    rows = np.array([[1, 2]], np.int32)
    for bad in ([3, 3], [8], [-1]):
        with pytest.raises(moe.MoEError) as ei:
            moe.moe_lfu_trace_pinned(4, 8, rows, bad)
        assert ei.value.status == 1


def packed_records(layer, ml_desc):
    """Host records in the library's layout (moe_pack_expert_record)."""
    recs = []
    n = moe.moe_expert_record_bytes(ml_desc)
    for ex in layer.experts:
        buf = np.zeros(n, np.uint8)
        moe.moe_pack_expert_record(ml_desc, ex, buf)
        recs.append(buf)
    return recs


def _streamed_vs_resident(layer, T, source=False, seed=31):
    import torch
    spec = layer.spec
    X = si.gen_tokens(seed, 0, T, spec)
    xs = torch.from_numpy(np.ascontiguousarray(X).view(np.int16)).cuda()
    y_res = torch.empty((T, spec.hidden), dtype=torch.float32, device="cuda")
    y_str = torch.empty((T, spec.hidden), dtype=torch.float32, device="cuda")
    ids = torch.empty((T, spec.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, spec.top_k), dtype=torch.float32, device="cuda")
    ids_s = torch.empty((T, spec.top_k), dtype=torch.int32, device="cuda")
    w_s = torch.empty((T, spec.top_k), dtype=torch.float32, device="cuda")
    with moe.MoELayer(layer) as res:
        for t in range(T):
            res.decode(xs[t], None, y_res[t])
            res.selection(1, ids[t], w[t])
        torch.cuda.synchronize()
        recs = packed_records(layer, res.desc)
    hm = []
    if source:
        calls = []

        def src(user, e, dst, nbytes):
            calls.append(e)
            ctypes.memmove(dst, recs[e].ctypes.data, nbytes)
            return 0
        kw = dict(source=moe.SOURCE_FN(src))
    else:
        kw = dict(records=recs)
    with moe.MoELayer(layer, cache_slots=16, **kw) as st:
        for t in range(T):
            st.decode(xs[t], None, y_str[t])
            st.selection(1, ids_s[t], w_s[t])
            torch.cuda.synchronize()
            hm.append(st.residency())
        stats = st.cache_stats()
    # the streamed layer's own selection equals the resident one's, and its
    # outputs are checked against the oracle directly
    assert torch.equal(ids_s, ids) and torch.equal(w_s, w)
    Wr = oracle.router_weights_f64(layer.router)
    ys = y_str.cpu().numpy()
    for t in range(T):
        compare_token(layer, X[t], ys[t], ids_s[t].cpu().numpy(), w_s[t].cpu().numpy(), Wr=Wr)
    return (y_res.cpu().numpy(), ys, ids.cpu().numpy(), hm, stats)


@pytest.mark.gpu
@pytest.mark.parametrize("source", [False, True])
def test_streamed_decode_bit_identical_and_lfu(source):
    spec = si.LayerSpec(hidden=512, inter=256, n_experts=64, zipf_alpha=1.1)
    layer = si.gen_layer(30, 0, spec)
    T = 40
    y_res, y_str, ids, residency, stats = _streamed_vs_resident(layer, T, source=source)
    assert np.array_equal(y_res, y_str)
    o_slot, o_hit = oracle_slots_hits(ids, 16)
    for t in range(T):
        # the oracle's slot map after token t, seen through the library's residency
        for j, e in enumerate(ids[t]):
            assert residency[t][o_slot[t][j]] == e
    assert stats["tokens"] == T
    assert stats["hits"] == int(o_hit.sum())
    assert stats["misses"] == T * spec.top_k - int(o_hit.sum())
    assert stats["bytes_h2d"] == stats["misses"] * moe.moe_expert_record_bytes(moe.desc_from_spec(spec))


@pytest.mark.gpu
def test_explicit_stage_counts():
    import torch
    spec = si.LayerSpec(hidden=256, inter=128, n_experts=32)
    layer = si.gen_layer(32, 0, spec)
    desc = moe.desc_from_spec(spec)
    recs = packed_records(layer, desc)
    with moe.MoELayer(layer, cache_slots=8, records=recs) as st:
        a = np.array([3, 5, 7, 9], np.int32)
        assert st.cache_stage(a, 4) == (0, 4)
        assert st.cache_stage(a, 4) == (4, 0)
        b = np.array([3, 11, 12, 13, 14, 15, 16, 17], np.int32)
        assert st.cache_stage(b, 8) == (1, 7)
        torch.cuda.synchronize()
        res = st.residency()
        assert sorted(e for e in res if e >= 0) == sorted(set(b.tolist()))
        with pytest.raises(moe.MoEError) as ei:
            st.cache_stage(np.array([1, 1], np.int32), 2)
        assert ei.value.status == 1


@pytest.mark.gpu
def test_source_failure_reported_and_recovered():
    """Host-side failure injection: the expert source fails for one expert; the
    decode that needs it returns MOE_E_SOURCE and leaves it out of the cache;
    once the source works again the same token decodes normally."""
    import torch
    spec = si.LayerSpec(hidden=256, inter=128, n_experts=16)
    layer = si.gen_layer(33, 0, spec)
    desc = moe.desc_from_spec(spec)
    recs = packed_records(layer, desc)
    X = si.gen_tokens(33, 0, 1, spec)
    x = torch.from_numpy(np.ascontiguousarray(X[0]).view(np.int16)).cuda()
    y = torch.empty(spec.hidden, dtype=torch.float32, device="cuda")
    y_ref = torch.empty(spec.hidden, dtype=torch.float32, device="cuda")
    ids = torch.empty(spec.top_k, dtype=torch.int32, device="cuda")
    w = torch.empty(spec.top_k, dtype=torch.float32, device="cuda")
    with moe.MoELayer(layer) as res:
        res.decode(x, None, y_ref)
        res.selection(1, ids, w)
        torch.cuda.synchronize()
    bad = int(ids[3].item())
    broken = {"on": True}

    def src(user, e, dst, nbytes):
        if broken["on"] and e == bad:
            return 1
        ctypes.memmove(dst, recs[e].ctypes.data, nbytes)
        return 0
    fn = moe.SOURCE_FN(src)
    with moe.MoELayer(layer, cache_slots=8, source=fn) as st:
        with pytest.raises(moe.MoEError) as ei:
            st.decode(x, None, y)
        assert ei.value.status == 7   # MOE_E_SOURCE
        torch.cuda.synchronize()
        assert bad not in st.residency()
        broken["on"] = False
        st.decode(x, None, y)
        torch.cuda.synchronize()
        assert torch.equal(y, y_ref)


@pytest.mark.gpu
def test_host_wait_deadline():
    """The copy stream is held on the host (a callback that sleeps); a short
    host deadline then runs out with MOE_E_TIMEOUT, and the layer works again
    once the stall is lifted."""
    import torch
    spec = si.LayerSpec(hidden=256, inter=128, n_experts=16)
    layer = si.gen_layer(34, 0, spec)
    desc = moe.desc_from_spec(spec)
    recs = packed_records(layer, desc)
    with moe.MoELayer(layer, cache_slots=8, records=recs) as st:
        st.set_option(moe.MOE_OPT_TEST_STALL_COPIES_MS, 400)
        st.set_option(moe.MOE_OPT_HOST_TIMEOUT_MS, 20)
        st.cache_stage(np.array([0, 1], np.int32), 2)
        st.cache_stage(np.array([2, 3], np.int32), 2)
        with pytest.raises(moe.MoEError) as ei:   # the first table buffer is still queued behind the stall
            st.cache_stage(np.array([4, 5], np.int32), 2)
        assert ei.value.status == 5   # MOE_E_TIMEOUT
        torch.cuda.synchronize()
        st.set_option(moe.MOE_OPT_TEST_STALL_COPIES_MS, 0)
        st.set_option(moe.MOE_OPT_HOST_TIMEOUT_MS, 30000)
        st.cache_stage(np.array([6, 7], np.int32), 2)
        torch.cuda.synchronize()


# --------------------------------------------------------------------------- streamed prefill (batch union)

def _prefill(ml, spec, xd, T):
    y = torch_empty(T * spec.hidden)
    y32 = torch_empty(T * spec.hidden)
    ml.prefill_chunk(xd, T, y, y32)
    import torch
    torch.cuda.synchronize()
    st, bits = ml.check()
    assert st == 0, hex(bits)
    return y32.cpu().numpy().reshape(T, spec.hidden)


def torch_empty(n):
    import torch
    return torch.empty(n, dtype=torch.float32, device="cuda")


def _waves(resident_before, distinct, slots):
    """The library's wave order: resident experts first, then the rest in
    ascending id, at most `slots` per wave."""
    res = [e for e in distinct if e in resident_before]
    rest = [e for e in distinct if e not in resident_before]
    waves = [res] if res else []
    for i in range(0, len(rest), slots):
        waves.append(rest[i:i + slots])
    return waves


@pytest.mark.gpu
@pytest.mark.parametrize("slots,T,E", [(16, 64, 64), (8, 24, 32), (8, 3, 16)])
def test_streamed_prefill_bit_identical_and_lfu(slots, T, E):
    """A prefill chunk on a streamed layer (batch union through the cache in
    waves) equals the resident layer's chunk bit for bit, over two chunks (the
    second finds experts resident); slot residency follows the oracle's LFU run
    over the same waves."""
    import torch
    spec = si.LayerSpec(hidden=256, inter=128, n_experts=E, zipf_alpha=1.1, act="f32")
    layer = si.gen_layer(35, 0, spec)
    chunks = [si.gen_tokens(35 + c, 0, T, spec) for c in range(2)]
    xs = [torch.from_numpy(np.ascontiguousarray(X, np.float32)).cuda() for X in chunks]
    ids = torch.empty((T, spec.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, spec.top_k), dtype=torch.float32, device="cuda")
    with moe.MoELayer(layer, max_tokens=T) as res:
        want = [_prefill(res, spec, xd, T) for xd in xs]
        sel = []
        for xd in xs:
            res.route(xd, T, ids, w)
            torch.cuda.synchronize()
            sel.append(ids.cpu().numpy().copy())
        recs = packed_records(layer, res.desc)
    sim = oracle.moe.LFUCache(slots)
    with moe.MoELayer(layer, max_tokens=T, cache_slots=slots, records=recs) as st:
        for c, xd in enumerate(xs):
            got = _prefill(st, spec, xd, T)
            assert np.array_equal(got, want[c])
            distinct = sorted(set(int(e) for e in sel[c].reshape(-1)))
            before = set(sim.count)
            for wv in _waves(before, distinct, slots):
                sim.access(np.array(wv, np.int64))
            residency = st.residency()
            for e, s in sim.slot_of.items():
                assert residency[s] == e
            assert sum(1 for e in residency if e >= 0) == len(sim.slot_of)


@pytest.mark.gpu
def test_streamed_prefill_source_failure():
    """A source that fails during a chunk's waves returns MOE_E_SOURCE; once
    it works again the chunk is computed as on the resident layer."""
    import torch
    spec = si.LayerSpec(hidden=256, inter=128, n_experts=16, act="f32")
    layer = si.gen_layer(36, 0, spec)
    T = 8
    X = si.gen_tokens(36, 0, T, spec)
    xd = torch.from_numpy(np.ascontiguousarray(X, np.float32)).cuda()
    with moe.MoELayer(layer, max_tokens=T) as res:
        want = _prefill(res, spec, xd, T)
        recs = packed_records(layer, res.desc)
    broken = {"on": True}

    def src(user, e, dst, nbytes):
        if broken["on"] and e % 3 == 1:
            return 1
        ctypes.memmove(dst, recs[e].ctypes.data, nbytes)
        return 0
    fn = moe.SOURCE_FN(src)
    with moe.MoELayer(layer, max_tokens=T, cache_slots=8, source=fn) as st:
        y = torch_empty(T * spec.hidden)
        with pytest.raises(moe.MoEError) as ei:
            st.prefill_chunk(xd, T, y, y)
        assert ei.value.status == 7   # MOE_E_SOURCE
        torch.cuda.synchronize()
        broken["on"] = False
        got = _prefill(st, spec, xd, T)
        assert np.array_equal(got, want)


# --------------------------------------------------------------------------- router lookahead

@pytest.mark.gpu
@pytest.mark.parametrize("exact", [True, False])
def test_lookahead_prefetch(exact):
    """moe_cache_prefetch stages a prediction; the decode that follows finds the
    predicted experts resident. With the token's own input as the prediction
    every routed expert is a hit; with the previous token's input some are.
    Outputs equal the resident layer's bit for bit, and the slots follow the
    oracle's LFU run of the same predictions and tokens."""
    import torch
    spec = si.LayerSpec(hidden=512, inter=256, n_experts=64, zipf_alpha=1.1)
    layer = si.gen_layer(37, 0, spec)
    T, k = 24, spec.top_k
    y_res, _, ids, _, _ = _streamed_vs_resident(layer, T, seed=37)
    X = si.gen_tokens(37, 0, T, spec)
    xs = torch.from_numpy(np.ascontiguousarray(X).view(np.int16)).cuda()
    with moe.MoELayer(layer, max_tokens=T) as res:
        recs = packed_records(layer, res.desc)
        # the selection each prediction input gives (the router of this layer)
        pid = torch.empty((T, k), dtype=torch.int32, device="cuda")
        pw = torch.empty((T, k), dtype=torch.float32, device="cuda")
        res.route(xs, T, pid, pw)
        torch.cuda.synchronize()
        pred_ids = pid.cpu().numpy()
    y = torch.empty((T, spec.hidden), dtype=torch.float32, device="cuda")
    sim = oracle.moe.LFUCache(16)
    with moe.MoELayer(layer, cache_slots=16, records=recs) as st:
        with moe.MoELayer(layer) as plain:
            with pytest.raises(moe.MoEError) as ei:
                plain.cache_prefetch(xs[0])
            assert ei.value.status == 2   # MOE_E_UNSUPPORTED on a resident layer
        for t in range(T):
            src = t if exact else max(t - 1, 0)
            s0 = st.cache_stats()
            r, f = st.cache_prefetch(xs[src])
            want_r, want_f = sim.prefetch(pred_ids[src])
            assert (r, f) == (len(want_r), len(want_f))
            st.decode(xs[t], None, y[t])
            torch.cuda.synchronize()
            h, _ = sim.access(ids[t])
            s1 = st.cache_stats()
            assert s1["hits"] - s0["hits"] == len(h)
            if exact:
                assert len(h) == k
            residency = st.residency()
            for e, s in sim.slot_of.items():
                assert residency[s] == e
        ps = st.prefetch_stats()
        assert ps["calls"] == T
    assert np.array_equal(y.cpu().numpy(), y_res)


@pytest.mark.gpu
def test_set_next_changes_no_result():
    """moe_layer_set_next (the next layer's router warmed into L2) is a hint:
    two chained layers, resident and streamed, give the same bits with it."""
    import torch
    spec = si.LayerSpec(hidden=512, inter=256, n_experts=32)
    lays = [si.gen_layer(38, l, spec) for l in range(2)]
    X = si.gen_tokens(38, 0, 6, spec)
    xs = torch.from_numpy(np.ascontiguousarray(X).view(np.int16)).cuda()

    def run(mls, link):
        if link:
            mls[0].set_next(mls[1])
            mls[1].set_next(mls[0])
        y = torch.empty((len(X), spec.hidden), dtype=torch.float32, device="cuda")
        yb = torch.empty(spec.hidden, dtype=torch.bfloat16, device="cuda")
        for t in range(len(X)):
            mls[0].decode(xs[t], yb, None)
            mls[1].decode(yb.view(torch.int16), None, y[t])
        torch.cuda.synchronize()
        return y.cpu().numpy()

    with moe.MoELayer(lays[0]) as a, moe.MoELayer(lays[1]) as b:
        plain = run([a, b], False)
    with moe.MoELayer(lays[0]) as a, moe.MoELayer(lays[1]) as b:
        linked = run([a, b], True)
        with pytest.raises(moe.MoEError):
            moe.moe_layer_set_next(None, b.handle)
    assert np.array_equal(plain, linked)
    recs = []
    for lay in lays:
        d = moe.desc_from_spec(spec, cache_slots=16)
        r = []
        for ex in lay.experts:
            buf = np.zeros(moe.moe_expert_record_bytes(d), np.uint8)
            moe.moe_pack_expert_record(d, ex, buf)
            r.append(buf)
        recs.append(r)
    with moe.MoELayer(lays[0], cache_slots=16, records=recs[0]) as a, \
            moe.MoELayer(lays[1], cache_slots=16, records=recs[1]) as b:
        streamed = run([a, b], True)
    assert np.array_equal(plain, streamed)


# ---- device-managed cache (MOE_OPT_CACHE_DEVICE) ------------------------------------

def pinned_records(recs):
    """The records copied into page-locked host memory: a device-managed cache
    reads them through their device mapping."""
    import torch
    out = []
    for r in recs:
        t = torch.empty(len(r), dtype=torch.uint8).pin_memory()
        t.numpy()[:] = r
        out.append(t)
    return out


def _resident(layer, xs):
    import torch
    T, spec = xs.shape[0], layer.spec
    y = torch.empty((T, spec.hidden), dtype=torch.float32, device="cuda")
    ids = torch.empty((T, spec.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, spec.top_k), dtype=torch.float32, device="cuda")
    with moe.MoELayer(layer) as res:
        for t in range(T):
            res.decode(xs[t], None, y[t])
            res.route(xs[t], 1, ids[t], w[t])
        torch.cuda.synchronize()
        recs = packed_records(layer, res.desc)
    return y.cpu().numpy(), ids.cpu().numpy(), recs


def _tokens(spec, seed, T):
    import torch
    X = si.gen_tokens(seed, 0, T, spec)
    return torch.from_numpy(np.ascontiguousarray(X).view(np.int16)).cuda()


@pytest.mark.gpu
def test_device_cache_bit_identical_and_lfu():
    """Each token's LFU step and fills run on the device; the outputs equal the
    resident layer's bit for bit and the slot map after every token is the
    oracle's."""
    import torch
    spec = si.LayerSpec(hidden=512, inter=256, n_experts=64, zipf_alpha=1.1)
    layer = si.gen_layer(30, 0, spec)
    T = 40
    xs = _tokens(spec, 31, T)
    y_res, ids, recs = _resident(layer, xs)
    y = torch.empty((T, spec.hidden), dtype=torch.float32, device="cuda")
    residency = []
    with moe.MoELayer(layer, cache_slots=16, records=pinned_records(recs)) as st:
        st.set_option(moe.MOE_OPT_CACHE_DEVICE, 1)
        for t in range(T):
            st.decode(xs[t], None, y[t])
            residency.append(st.residency())   # synchronises
        stats = st.cache_stats()
        assert st.check() == (0, 0)
    assert np.array_equal(y_res, y.cpu().numpy())
    o_slot, o_hit = oracle_slots_hits(ids, 16)
    for t in range(T):
        for j, e in enumerate(ids[t]):
            assert residency[t][o_slot[t][j]] == e
    assert stats["tokens"] == T
    assert stats["hits"] == int(o_hit.sum())
    assert stats["misses"] == T * spec.top_k - int(o_hit.sum())
    assert stats["bytes_h2d"] == stats["misses"] * moe.moe_expert_record_bytes(moe.desc_from_spec(spec))


@pytest.mark.gpu
def test_device_cache_switch_queue_and_graph():
    """Host staging, then device-managed tokens queued with no host wait, host
    staging again, then device-managed decodes replayed from a CUDA graph: one
    LFU run throughout (the oracle's), outputs bit-identical to resident."""
    import torch
    spec = si.LayerSpec(hidden=256, inter=128, n_experts=32, top_k=4, zipf_alpha=1.1)
    layer = si.gen_layer(32, 0, spec)
    T = 40
    xs = _tokens(spec, 33, T)
    y_res, ids, recs = _resident(layer, xs)
    slots = 8
    y = torch.empty((T, spec.hidden), dtype=torch.float32, device="cuda")
    with moe.MoELayer(layer, cache_slots=slots, records=pinned_records(recs)) as st:
        for t in range(0, 10):                      # host staging
            st.decode(xs[t], None, y[t])
        st.set_option(moe.MOE_OPT_CACHE_DEVICE, 1)
        for t in range(10, 22):                     # queued, no synchronisation
            st.decode(xs[t], None, y[t])
        st.set_option(moe.MOE_OPT_CACHE_DEVICE, 0)
        mid = st.residency()
        for t in range(22, 28):                     # host staging again
            st.decode(xs[t], None, y[t])
        st.set_option(moe.MOE_OPT_CACHE_DEVICE, 1)
        x_in = torch.empty_like(xs[0])
        y_out = torch.empty(spec.hidden, dtype=torch.float32, device="cuda")
        x_in.copy_(xs[28])
        gs = torch.cuda.Stream()
        gs.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(gs):
            st.decode(x_in, None, y_out, stream=gs.cuda_stream)   # token 28, outside the graph
            gs.synchronize()
            y[28].copy_(y_out)
            gs.synchronize()
            with torch.cuda.graph(g, stream=gs):
                st.decode(x_in, None, y_out, stream=gs.cuda_stream)
        torch.cuda.current_stream().wait_stream(gs)
        for t in range(29, T):                      # graph replays
            x_in.copy_(xs[t])
            g.replay()
            y[t].copy_(y_out)
        torch.cuda.synchronize()
        final = st.residency()
        stats = st.cache_stats()
        assert st.check() == (0, 0)
        del g
    assert np.array_equal(y_res, y.cpu().numpy())
    o_slot, o_hit = oracle_slots_hits(ids, slots)
    for j, e in enumerate(ids[21]):
        assert mid[o_slot[21][j]] == e
    for j, e in enumerate(ids[T - 1]):
        assert final[o_slot[T - 1][j]] == e
    assert stats["tokens"] == T
    assert stats["hits"] == int(o_hit.sum())
    assert stats["misses"] == T * spec.top_k - int(o_hit.sum())


@pytest.mark.gpu
def test_device_cache_refusals():
    """A source callback cannot run on the device; while the cache is
    device-managed, host staging and lookahead refuse with MOE_E_STATE; a
    resident layer has no cache to manage."""
    import torch
    spec = si.LayerSpec(hidden=256, inter=128, n_experts=16, top_k=4)
    layer = si.gen_layer(34, 0, spec)
    xs = _tokens(spec, 35, 4)
    _, _, recs = _resident(layer, xs)

    def src(user, e, dst, nbytes):
        ctypes.memmove(dst, recs[e].ctypes.data, nbytes)
        return 0
    with moe.MoELayer(layer, cache_slots=8, source=moe.SOURCE_FN(src)) as st:
        with pytest.raises(moe.MoEError) as ei:
            st.set_option(moe.MOE_OPT_CACHE_DEVICE, 1)
        assert ei.value.status == 2
    with moe.MoELayer(layer, cache_slots=8, records=pinned_records(recs), max_tokens=4) as st:
        st.set_option(moe.MOE_OPT_CACHE_DEVICE, 1)
        ids = np.array([0, 1, 2, 3], np.int32)
        with pytest.raises(moe.MoEError) as ei:
            st.cache_stage(ids, 4)
        assert ei.value.status == 6
        with pytest.raises(moe.MoEError) as ei:
            st.cache_prefetch(xs[0])
        assert ei.value.status == 6
        with pytest.raises(moe.MoEError) as ei:
            st.set_option(moe.MOE_OPT_CACHE_DEVICE, 2)
        assert ei.value.status == 1
    with moe.MoELayer(layer) as res:
        with pytest.raises(moe.MoEError) as ei:
            res.set_option(moe.MOE_OPT_CACHE_DEVICE, 1)
        assert ei.value.status == 6


# ---- the learning cache (usage counts, pinned experts) -------------------------------

@pytest.mark.gpu
@pytest.mark.parametrize("device", [False, True])
def test_learning_cache_pin_hottest(device):
    """Usage counts equal the oracle's; pinning the hottest experts (the
    oracle's choice, ties to the lower id) keeps the outputs bit-identical to
    the resident layer's; pinned lookups hit and leave the LFU alone, so the
    slot map follows the oracle's run with the same pins, through a re-pin and
    an unpin; host-managed and device-managed alike."""
    import torch
    spec = si.LayerSpec(hidden=512, inter=256, n_experts=64, zipf_alpha=1.1)
    layer = si.gen_layer(36, 0, spec)
    T = 48
    xs = _tokens(spec, 37, T)
    y_res, ids, recs = _resident(layer, xs)
    slots = 8
    sim = oracle.moe.LFUCache(slots)
    hits = misses = 0
    y = torch.empty((T, spec.hidden), dtype=torch.float32, device="cuda")
    with moe.MoELayer(layer, cache_slots=slots, records=pinned_records(recs)) as st:
        if device:
            st.set_option(moe.MOE_OPT_CACHE_DEVICE, 1)
        for t in range(T):
            if t == 16:
                use = st.cache_usage()
                want = np.zeros(spec.n_experts, np.uint64)
                for e, n in sim.usage.items():
                    want[e] = n
                assert np.array_equal(use, want)
                hot = sim.hottest(6)
                st.pin_hottest(6)
                sim.pin(hot)
            if t == 30:   # a new set: some stay, some leave, some come
                new = sim.hottest(10)[4:]
                st.cache_pin(np.array(new, np.int32))
                sim.pin(new)
            if t == 40:
                st.cache_pin([])
                sim.pin([])
            st.decode(xs[t], None, y[t])
            h, f = sim.access(ids[t])
            hits += len(h)
            misses += len(f)
            res = st.residency()
            for e, s in sim.slot_of.items():
                assert res[s] == e, (t, e, s, res)
            assert sum(1 for e in res if e >= 0) == len(sim.slot_of)
        stats = st.cache_stats()
        assert st.check() == (0, 0)
    assert np.array_equal(y_res, y.cpu().numpy())
    assert stats["tokens"] == T
    assert stats["hits"] == hits
    assert stats["misses"] == misses


@pytest.mark.gpu
def test_learning_cache_streamed_prefill():
    """A prefill chunk on a streamed layer with pinned experts: the pinned ones
    join the first (resident) wave, the output equals the resident layer's bit
    for bit, and the LFU follows the oracle's run over the same waves."""
    import torch
    T, E, slots = 24, 32, 8
    spec = si.LayerSpec(hidden=256, inter=128, n_experts=E, zipf_alpha=1.1, act="f32")
    layer = si.gen_layer(38, 0, spec)
    chunks = [si.gen_tokens(38 + c, 0, T, spec) for c in range(2)]
    xs = [torch.from_numpy(np.ascontiguousarray(X, np.float32)).cuda() for X in chunks]
    ids = torch.empty((T, spec.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, spec.top_k), dtype=torch.float32, device="cuda")
    with moe.MoELayer(layer, max_tokens=T) as res:
        want = [_prefill(res, spec, xd, T) for xd in xs]
        sel = []
        for xd in xs:
            res.route(xd, T, ids, w)
            torch.cuda.synchronize()
            sel.append(ids.cpu().numpy().copy())
        recs = packed_records(layer, res.desc)
    sim = oracle.moe.LFUCache(slots)
    with moe.MoELayer(layer, max_tokens=T, cache_slots=slots, records=recs) as st:
        for c, xd in enumerate(xs):
            if c == 1:   # pin the hottest after the first chunk
                hot = sim.hottest(5)
                st.pin_hottest(5)
                sim.pin(hot)
            got = _prefill(st, spec, xd, T)
            assert np.array_equal(got, want[c])
            distinct = sorted(set(int(e) for e in sel[c].reshape(-1)))
            for wv in _waves(set(sim.count) | set(sim.pinned), distinct, slots):
                sim.access(np.array(wv, np.int64))
            residency = st.residency()
            for e, s in sim.slot_of.items():
                assert residency[s] == e
            assert sum(1 for e in residency if e >= 0) == len(sim.slot_of)
        use = st.cache_usage()
    assert [int(use[e]) for e in range(E)] == [sim.usage.get(e, 0) for e in range(E)]


@pytest.mark.gpu
def test_learning_cache_refusals():
    spec = si.LayerSpec(hidden=256, inter=128, n_experts=16, top_k=4)
    layer = si.gen_layer(39, 0, spec)
    xs = _tokens(spec, 40, 2)
    _, _, recs = _resident(layer, xs)
    with moe.MoELayer(layer, cache_slots=8, records=recs) as st:
        for bad in ([1, 1], [16], [-1]):
            with pytest.raises(moe.MoEError) as ei:
                st.cache_pin(bad)
            assert ei.value.status == 1
    with moe.MoELayer(layer) as res:
        with pytest.raises(moe.MoEError) as ei:
            res.cache_pin([0])
        assert ei.value.status == 6
        with pytest.raises(moe.MoEError) as ei:
            moe.moe_cache_usage(res.handle, spec.n_experts)
        assert ei.value.status == 6


@pytest.mark.gpu
def test_device_cache_with_streamed_prefill():
    """Device-managed decodes, a streamed prefill chunk (its waves staged on the
    host, the state handed over and back), then device-managed decodes again:
    one LFU run (the oracle's), outputs bit-identical to the resident layer."""
    import torch
    T, E, slots = 24, 32, 8
    spec = si.LayerSpec(hidden=256, inter=128, n_experts=E, zipf_alpha=1.1, act="f32")
    layer = si.gen_layer(41, 0, spec)
    Xd = si.gen_tokens(41, 0, 12, spec)
    Xp = si.gen_tokens(42, 0, T, spec)
    xd = torch.from_numpy(np.ascontiguousarray(Xd, np.float32)).cuda()
    xp = torch.from_numpy(np.ascontiguousarray(Xp, np.float32)).cuda()
    ids = torch.empty((T, spec.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, spec.top_k), dtype=torch.float32, device="cuda")
    y_dec = torch.empty((12, spec.hidden), dtype=torch.float32, device="cuda")
    with moe.MoELayer(layer, max_tokens=T) as res:
        want_p = _prefill(res, spec, xp, T)
        for t in range(12):
            res.decode(xd[t], None, y_dec[t])
        res.route(xp, T, ids, w)
        torch.cuda.synchronize()
        sel_p = ids.cpu().numpy().copy()
        res.route(xd, 12, ids[:12], w[:12])
        torch.cuda.synchronize()
        sel_d = ids[:12].cpu().numpy().copy()
        want_d = y_dec.cpu().numpy()
        recs = packed_records(layer, res.desc)
    sim = oracle.moe.LFUCache(slots)
    got_d = torch.empty((12, spec.hidden), dtype=torch.float32, device="cuda")
    with moe.MoELayer(layer, max_tokens=T, cache_slots=slots, records=pinned_records(recs)) as st:
        st.set_option(moe.MOE_OPT_CACHE_DEVICE, 1)
        for t in range(6):
            st.decode(xd[t], None, got_d[t])
            sim.access(sel_d[t])
        got_p = _prefill(st, spec, xp, T)
        distinct = sorted(set(int(e) for e in sel_p.reshape(-1)))
        for wv in _waves(set(sim.count) | set(sim.pinned), distinct, slots):
            sim.access(np.array(wv, np.int64))
        for t in range(6, 12):
            st.decode(xd[t], None, got_d[t])
            sim.access(sel_d[t])
        res_final = st.residency()
        assert st.check() == (0, 0)
    assert np.array_equal(got_p, want_p)
    assert np.array_equal(got_d.cpu().numpy(), want_d)
    for e, s_ in sim.slot_of.items():
        assert res_final[s_] == e
    assert sum(1 for e in res_final if e >= 0) == len(sim.slot_of)
