"""Pins for the CPU oracle: each test checks it against something other than itself
(values printed on the pages, closed forms, brute force, a library routine, or an
independently written simulation).  CPU only."""
import math
import os
import random
from fractions import Fraction

import numpy as np
import pytest

import oracle as O
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [l.split() for l in f if l.strip() and not l.startswith("#")]


# ------------------------------------------------------------------------ q*
def test_qstar_worked_examples_from_pages():
    for m, bp, bh, printed, dec, fills, host in _rows("qstar_worked_examples.txt"):
        m, fills, host = int(m), int(fills), int(host)
        # the page's continuous value m*B_P/B_H, to the printed precision
        assert round(m * float(bp) / float(bh), int(dec)) == pytest.approx(float(printed))
        q = O.split_misses(m, O.mbps(float(bp)), O.mbps(float(bh)), evictable=10 ** 6)
        assert q == fills and m - q == host


def _balance_root(m, bp, bh):
    """Solve q/B_P = (m-q)/(B_H-B_P) by bisection (the equal-branch-time condition)."""
    lo, hi = Fraction(0), Fraction(m)
    f = lambda q: q / Fraction(bp) - (m - q) / Fraction(bh - bp)
    for _ in range(200):
        mid = (lo + hi) / 2
        if f(mid) > 0:
            hi = mid
        else:
            lo = mid
    return (lo + hi) / 2


def test_qstar_solves_branch_balance_and_rounds_half_up():
    rng = random.Random(7)
    for _ in range(300):
        m = rng.randint(1, 64)
        bp = rng.randint(1000, 200000)
        bh = bp + rng.randint(1, 300000)
        root = _balance_root(m, bp, bh)
        expect = max(1, math.floor(root + Fraction(1, 2)))
        # bisection is accurate to ~m/2^200; the rounding boundary is a multiple of 1/(2bh)
        assert O.split_misses(m, bp, bh, 10 ** 6) == min(expect, m)


def test_qstar_rounding_ties_go_up():
    # 25:50 with odd m lands exactly on .5
    assert O.split_misses(1, 25000, 50000, 99) == 1     # 0.5 -> 1 (also the >=1 rule)
    assert O.split_misses(3, 25000, 50000, 99) == 2     # 1.5 -> 2
    assert O.split_misses(5, 25000, 50000, 99) == 3     # 2.5 -> 3


def test_qstar_limits_and_clamps():
    for m in range(1, 40):
        # B_H approaching B_P from above: every miss is filled
        assert O.split_misses(m, 100000, 100001, 10 ** 6) == m
        # residual bandwidth max(B_H-B_P, 0) = 0 -> all misses go to the link
        assert O.split_misses(m, 80000, 50000, 10 ** 6) == m
        assert O.split_misses(m, 50000, 50000, 10 ** 6) == m
        # at least one fill whenever there is a miss
        assert O.split_misses(m, 1, 10 ** 9, 10 ** 6) == 1
        # never more fills than evictable slots
        assert O.split_misses(m, 80000, 50000, 2) == min(m, 2)
        assert O.split_misses(m, 80000, 50000, 0) == 0
    assert O.split_misses(0, 1, 2, 5) == 0


def test_mbps_rounding():
    assert O.mbps(52.7) == 52700 and O.mbps(77.3) == 77300 and O.mbps(11.8) == 11800
    assert O.mbps(0.0005) == 1 and O.mbps(0.0004) == 0


# --------------------------------------------------------------------- router
def test_router_matches_torch_topk_softmax():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(3)
    for B, E, k in [(1, 16, 2), (8, 256, 8), (64, 256, 8), (3, 40, 7)]:
        z = rng.standard_normal((B, E)).astype(np.float32)
        sel, gates = O.route(z, k)
        tz = torch.from_numpy(z).double()
        v, i = torch.topk(tz, k, dim=1)
        i_sorted, perm = torch.sort(i, dim=1)
        g = torch.softmax(torch.gather(tz, 1, i_sorted), dim=1)
        assert np.array_equal(sel, i_sorted.numpy())
        np.testing.assert_allclose(gates, g.float().numpy(), rtol=1e-6, atol=0)


def test_router_ties_pick_lower_id_brute_force():
    rng = random.Random(11)
    for _ in range(200):
        E = rng.randint(2, 24)
        k = rng.randint(1, E)
        z = np.array([rng.choice([0.0, 1.0, -1.0, 0.5]) for _ in range(E)], dtype=np.float32)
        ranked = sorted(range(E), key=lambda e: (-float(z[e]), e))
        sel, gates = O.route(z[None, :], k)
        assert list(sel[0]) == sorted(ranked[:k])
        w = [math.exp(float(z[e]) - max(float(z[j]) for j in ranked[:k])) for e in sorted(ranked[:k])]
        assert np.allclose(gates[0], np.array(w) / sum(w), rtol=1e-6)


def test_router_nan_ranks_as_minus_inf_and_signed_zeros_tie():
    """Brute force over small rows with NaN, -inf, -0 and +0: NaN takes the place of -inf,
    -0 equals +0, and equal keys go to the lower id.  Gates of the softmax over the chosen:
    a -inf logit among them gets exactly 0."""
    rng = random.Random(17)
    vals = [0.0, -0.0, 1.0, -1.0, float("-inf"), float("nan"), 2.5]
    for _ in range(300):
        E = rng.randint(2, 20)
        k = rng.randint(1, E)
        z = np.array([rng.choice(vals) for _ in range(E)], dtype=np.float32)
        z[rng.randrange(E)] = 3.0                      # at least one finite logit on top
        key = [float("-inf") if math.isnan(float(v)) else float(v) for v in z]
        ranked = sorted(range(E), key=lambda e: (-key[e], e))
        chosen = sorted(ranked[:k])
        sel, gates = O.route(z[None, :], k)
        assert list(sel[0]) == chosen
        top = max(key[e] for e in chosen)
        ex = [0.0 if key[e] == float("-inf") else math.exp(key[e] - top) for e in chosen]
        np.testing.assert_allclose(gates[0], np.array(ex) / sum(ex), rtol=1e-6, atol=0)
        assert all(g == 0.0 for g, e in zip(gates[0], chosen) if key[e] == float("-inf"))


def test_rel_err_rows_hand_computed():
    """The output metric, per row max|y - ref| / max|ref|, then the largest row.  The case
    is built so that each plausible slip gives another value: |y| as the denominator gives
    0.142857, one global max over all rows 0.1, an element-wise ratio 1.0, a mean over the
    rows 0.1125."""
    y = np.array([[1.0, -2.0, 3.5], [90.0, 0.0, 0.0]])
    ref = np.array([[0.5, -2.0, 4.0], [100.0, 0.0, 0.0]])
    assert O.rel_err_rows(y, ref) == pytest.approx(0.125, abs=1e-15)
    assert O.rel_err_rows(ref, y) == pytest.approx(max(0.5 / 3.5, 10.0 / 90.0), abs=1e-15)
    assert O.rel_err_rows(np.array([1.0, 2.0]), np.array([2.0, 2.0])) == pytest.approx(0.5)  # one row
    assert O.rel_err_rows(np.zeros((2, 3)), np.zeros((2, 3))) == 0.0
    assert O.rel_err_rows(ref, ref) == 0.0


def test_router_gate_functions_match_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    for B, E, k in [(1, 16, 2), (8, 256, 8), (5, 40, 7)]:
        z = (rng.standard_normal((B, E)) * 3).astype(np.float32)
        tz = torch.from_numpy(z).double()
        sel0, _ = O.route(z, k)
        idx = torch.from_numpy(sel0)
        sel1, g1 = O.route(z, k, O.GATE_SOFTMAX_ALL)
        sel2, g2 = O.route(z, k, O.GATE_SIGMOID_TOPK)
        assert np.array_equal(sel1, sel0) and np.array_equal(sel2, sel0)
        ref1 = torch.gather(torch.softmax(tz, dim=1), 1, idx)
        s = torch.gather(torch.sigmoid(tz), 1, idx)
        ref2 = s / s.sum(dim=1, keepdim=True)
        np.testing.assert_allclose(g1, ref1.float().numpy(), rtol=1e-6, atol=0)
        np.testing.assert_allclose(g2, ref2.float().numpy(), rtol=1e-6, atol=0)


def test_router_gate_functions_brute_force_and_closed_forms():
    rng = random.Random(13)
    for _ in range(100):
        E = rng.randint(2, 20)
        k = rng.randint(1, E)
        z = np.array([rng.uniform(-6, 6) for _ in range(E)], dtype=np.float32)
        ranked = sorted(range(E), key=lambda e: (-float(z[e]), e))
        chosen = sorted(ranked[:k])
        ex = [math.exp(float(v)) for v in z]
        sg = [1.0 / (1.0 + math.exp(-float(v))) for v in z]
        _, g1 = O.route(z[None, :], k, O.GATE_SOFTMAX_ALL)
        _, g2 = O.route(z[None, :], k, O.GATE_SIGMOID_TOPK)
        assert np.allclose(g1[0], [ex[e] / sum(ex) for e in chosen], rtol=1e-6)
        assert np.allclose(g2[0], [sg[e] / sum(sg[j] for j in chosen) for e in chosen], rtol=1e-6)
        # softmax over all E is the top-k softmax scaled by the chosen experts' share of the mass
        _, g0 = O.route(z[None, :], k)
        share = sum(ex[e] for e in chosen) / sum(ex)
        assert np.allclose(g1[0], g0[0] * share, rtol=1e-6)
    # two experts with opposite logits: s(a) + s(-a) = 1, so the normalised sigmoid gate is s(a)
    for a in (0.25, 1.0, 3.0):
        _, g = O.route(np.array([[a, -a]], dtype=np.float32), 2, O.GATE_SIGMOID_TOPK)
        assert abs(float(g[0, 0]) - 1.0 / (1.0 + math.exp(-a))) < 1e-7
    # k = E: softmax over all E and over the k chosen coincide
    z = np.array([[0.5, -1.0, 2.0, 0.0]], dtype=np.float32)
    assert np.array_equal(O.route(z, 4, O.GATE_SOFTMAX_ALL)[1], O.route(z, 4)[1])


def _bf16_bits(v: np.ndarray) -> np.ndarray:
    """float32 values that are exact in BF16 -> their BF16 bit patterns"""
    b = np.asarray(v, dtype=np.float32).view(np.uint32)
    assert np.all((b & 0xFFFF) == 0)
    return (b >> 16).astype(np.uint16)


def test_router_logits_brute_force_and_closed_forms():
    rng = np.random.default_rng(17)
    B, E, H = 3, 5, 24
    # small integers and halves are exact in BF16
    x = rng.integers(-8, 9, size=(B, H)).astype(np.float32) / 2
    w = rng.integers(-8, 9, size=(E, H)).astype(np.float32) / 4
    z = O.router_logits(_bf16_bits(x), _bf16_bits(w))
    assert z.shape == (B, E)
    for t in range(B):
        for e in range(E):
            assert z[t, e] == sum(float(x[t, h]) * float(w[e, h]) for h in range(H))
    # one-hot router rows pick single hidden coordinates
    eye = np.zeros((E, H), dtype=np.float32)
    for e in range(E):
        eye[e, 3 * e + 1] = 1.0
    ze = O.router_logits(_bf16_bits(x), _bf16_bits(eye))
    assert np.array_equal(ze, x[:, [3 * e + 1 for e in range(E)]].astype(np.float64))
    # a router row equal to the token gives its squared norm
    zs = O.router_logits(_bf16_bits(x[:1]), _bf16_bits(x))
    assert zs[0, 0] == float(np.dot(x[0].astype(np.float64), x[0].astype(np.float64)))


def _naive_on_demand(slots, layer, E, active, clock):
    """Independent model of an on-demand prefill layer: `slots` is a list of
    [stamp, owner] per slot; returns the new clock.  Hits are refreshed; the misses
    go, W at a time in ascending id, into the W least recently used slots that hold
    no hit, ordered by (stamp, slot index)."""
    clock += 1
    want = sorted({layer * E + e for e in active})
    where = {o: i for i, (st, o) in enumerate(slots) if o >= 0}
    hit_slots = {where[u] for u in want if u in where}
    for i in hit_slots:
        slots[i][0] = clock
    missing = [u for u in want if u not in where]
    free = sorted((st, i) for i, (st, o) in enumerate(slots) if i not in hit_slots)
    if missing:
        assert free, "capacity"
    width = len(free)
    for start in range(0, len(missing), max(1, width)):
        for (st, i), u in zip(free, missing[start:start + width]):
            slots[i] = [clock, u]
    return clock


def test_on_demand_prefill_matches_naive_model_and_invariants():
    rng = random.Random(23)
    for _ in range(300):
        E = rng.randint(2, 12)
        L = rng.randint(1, 3)
        S = rng.randint(1, 2 * E - 1)
        cache = O.SlotCache(S, L * E)
        slots = [[0, -1] for _ in range(S)]
        clock = 0
        for _step in range(rng.randint(1, 6)):
            layer = rng.randrange(L)
            active = rng.sample(range(E), rng.randint(1, E))
            hits_before = sum(1 for e in set(active) if cache.res[layer * E + e] >= 0)
            if hits_before == S and len(set(active)) > S:
                continue  # no slot outside the hits: the capacity error case
            waves = cache.prefill_layer_on_demand(layer, E, active)
            clock = _naive_on_demand(slots, layer, E, active, clock)
            assert cache.clock == clock
            assert [int(v) for v in cache.stamp] == [st for st, _ in slots]
            assert [int(v) for v in cache.owner] == [o for _, o in slots]
            # residency is a bijection on occupied slots
            for v in range(S):
                if cache.owner[v] >= 0:
                    assert cache.res[cache.owner[v]] == v
            assert int(np.count_nonzero(cache.res >= 0)) == int(np.count_nonzero(cache.owner >= 0))
            # the last wave and every hit of the layer are resident and stamped now
            for u in (waves[-1] if waves else []):
                assert cache.res[u] >= 0 and cache.stamp[cache.res[u]] == cache.clock
            assert sum(len(w) for w in waves) == len(set(active)) - hits_before
    # no slot outside the hits and a miss left: the reading has no answer
    cache = O.SlotCache(1, 4)
    cache.prefill_layer_on_demand(0, 4, [0])
    before = (cache.clock, cache.res.copy(), cache.owner.copy(), cache.stamp.copy())
    with pytest.raises(ValueError):
        cache.prefill_layer_on_demand(0, 4, [0, 1])
    assert cache.clock == before[0] and np.array_equal(cache.res, before[1])
    assert np.array_equal(cache.owner, before[2]) and np.array_equal(cache.stamp, before[3])


def test_e2m1_values_from_float32_bit_patterns():
    """Every FP4 (E2M1) code against the float32 with the same sign, exponent and
    mantissa fields (exponent rebiased from 1 to 127; exponent 0 is subnormal)."""
    import struct

    for code in range(16):
        sign, exp, man = code >> 3, (code >> 1) & 3, code & 1
        if exp == 0:
            ref = (-1.0 if sign else 1.0) * man * 0.5
        else:
            bits = (sign << 31) | ((exp - 1 + 127) << 23) | (man << 22)
            ref = struct.unpack("<f", struct.pack("<I", bits))[0]
        assert O.E2M1_TABLE[code] == ref, code
    # byte 0x21: element 0 is the low nibble (code 1 = 0.5), element 1 the high one (code 2 = 1)
    assert O.e2m1_unpack_to_f64(np.array([[0x21, 0xF7]], dtype=np.uint8)).tolist() == [[0.5, 1.0, 6.0, -6.0]]


def test_nvfp4_matvec_post_scaled_equals_dequantise_first_and_brute_force():
    rng = np.random.default_rng(29)
    R, K = 5, 64
    packed = rng.integers(0, 256, size=(R, K // 2), dtype=np.uint8)
    bscale = rng.integers(0x28, 0x48, size=(R, K // O.NVFP4_BLOCK), dtype=np.uint8)
    ts = 0.0073
    x = rng.standard_normal(K)
    y = O.matvec_nvfp4(packed, bscale, ts, x)
    w = O.e2m1_unpack_to_f64(packed) * np.repeat(O.e4m3_to_f64(bscale), O.NVFP4_BLOCK, axis=1) * ts
    np.testing.assert_allclose(y, w @ x, rtol=1e-12, atol=1e-15)
    for r in range(R):  # scalar loop: nibbles, blocks, scales written out
        tot = 0.0
        for b in range(K // 16):
            part = 0.0
            for j in range(16):
                k = 16 * b + j
                code = (int(packed[r, k // 2]) >> (4 * (k % 2))) & 0xF
                part += O.E2M1_TABLE[code] * x[k]
            tot += part * O.e4m3_to_f64(np.array([bscale[r, b]]))[0]
        assert abs(ts * tot - y[r]) <= 1e-12 * max(1.0, abs(y[r]))


def test_e8m0_and_mxfp4_matvec():
    """E8M0 codes against ldexp; the MXFP4 post-scaled product against dequantise-first and
    a scalar loop over nibbles and 32-element blocks."""
    codes = np.arange(255)
    assert all(O.e8m0_to_f64(codes)[c] == math.ldexp(1.0, int(c) - 127) for c in codes)
    assert np.isnan(O.e8m0_to_f64(np.array([255]))[0])
    rng = np.random.default_rng(31)
    R, K = 4, 96
    packed = rng.integers(0, 256, size=(R, K // 2), dtype=np.uint8)
    sc = rng.integers(118, 124, size=(R, K // O.MXFP4_BLOCK), dtype=np.uint8)
    x = rng.standard_normal(K)
    y = O.matvec_mxfp4(packed, sc, x)
    w = O.e2m1_unpack_to_f64(packed) * np.repeat(O.e8m0_to_f64(sc), O.MXFP4_BLOCK, axis=1)
    np.testing.assert_allclose(y, w @ x, rtol=1e-12, atol=1e-15)
    for r in range(R):
        tot = 0.0
        for b in range(K // 32):
            part = sum(O.E2M1_TABLE[(int(packed[r, k // 2]) >> (4 * (k % 2))) & 0xF] * x[k]
                       for k in range(32 * b, 32 * b + 32))
            tot += part * 2.0 ** (int(sc[r, b]) - 127)
        assert abs(tot - y[r]) <= 1e-12 * max(1.0, abs(y[r]))


def test_dedupe_is_sorted_union():
    sel = np.array([[3, 5], [1, 5], [3, 9]])
    assert O.dedupe(sel, 2, 16) == [33, 35, 37, 41]


# ----------------------------------------------------------------------- LRU
class NaiveListLRU:
    """Move-to-back list model of the same policy, written independently: `order` runs
    from least to most recently used; all slots touched in one step (hits and fills)
    become equally recent and are appended in ascending slot order."""

    def __init__(self, S, n_logical):
        self.order = list(range(S))       # all empty, equally old: slot order
        self.table = {}                   # u -> slot
        self.slot_u = {}

    def step(self, A, bp, bh):
        hits = [u for u in A if u in self.table]
        miss = [u for u in A if u not in self.table]
        hit_slots = [self.table[u] for u in hits]
        for s in hit_slots:
            self.order.remove(s)
        m = len(miss)
        if m == 0:
            q = 0
        elif bh <= bp:
            q = m
        else:
            q = max(1, math.floor(Fraction(m * bp, bh) + Fraction(1, 2)))
        q = min(q, m, len(self.order))
        victims = self.order[:q]
        del self.order[:q]
        for s, u in zip(victims, miss[:q]):
            if s in self.slot_u:
                del self.table[self.slot_u[s]]
            self.slot_u[s] = u
            self.table[u] = s
        self.order.extend(sorted(hit_slots + victims))
        return hits, miss, q, victims


def _check_state_bijection(c: O.SlotCache):
    occ = {int(s): int(c.owner[s]) for s in range(c.S) if c.owner[s] >= 0}
    res = {int(u): int(s) for u, s in enumerate(c.res) if s >= 0}
    assert {u: s for s, u in occ.items()} == res


@pytest.mark.parametrize("seed", range(12))
def test_lru_matches_naive_list_simulation(seed):
    rng = np.random.default_rng(seed)
    L, E = 3, 8
    S = int(rng.integers(1, 17))
    B, k = int(rng.integers(1, 4)), int(rng.integers(1, 4))
    bp, bh = [(11800, 47500), (25000, 50000), (52700, 77300), (80000, 50000)][seed % 4]
    c = O.SlotCache(S, L * E)
    n = NaiveListLRU(S, L * E)
    for step in range(60):
        layer = step % L
        sel, _ = O.route(rng.standard_normal((B, E)).astype(np.float32), k)
        rec = c.decode_step(layer, E, sel, bp, bh)
        hits, miss, q, victims = n.step(O.dedupe(sel, layer, E), bp, bh)
        assert (rec.H, rec.M, rec.q) == (hits, miss, q)
        assert rec.victims[:rec.q] == victims
        assert len(rec.victims) == (min(B * k, E, S - len(rec.H)) if rec.q else 0)
        assert {int(u): int(s) for u, s in enumerate(c.res) if s >= 0} == n.table
        _check_state_bijection(c)
        # full LRU order of the cache equals the list model's order
        by_recency = sorted(range(S), key=lambda s: (int(c.stamp[s]), s))
        assert by_recency == n.order


def test_lru_invariants_on_trace():
    w = synth.decode_bf16().with_(n_layers=4, n_experts=64, cache_slots=40, steps=80)
    tr = synth.routing_trace(w)
    c = O.SlotCache(w.cache_slots, w.n_logical)
    bp, bh = O.mbps(w.bp_gbps), O.mbps(w.bh_gbps)
    total_A = 0
    for s in range(w.steps):
        for l in range(w.n_layers):
            sel, _ = O.route(synth.decode_logits(w, s, l, tr), w.top_k)
            before = c.cnt.fills
            rec = c.decode_step(l, w.n_experts, sel, bp, bh)
            total_A += len(rec.A)
            assert set(rec.F) | set(rec.C) == set(rec.M) and not set(rec.F) & set(rec.C)
            assert c.cnt.fills - before == rec.q
            for u in rec.C:      # C set: residency unchanged (still absent)
                assert c.res[u] < 0
            for u in rec.H + rec.F:
                assert c.stamp[c.res[u]] == c.clock
            _check_state_bijection(c)
    assert c.cnt.hits + c.cnt.misses == total_A
    assert c.cnt.fills <= c.cnt.misses
    assert c.cnt.fills + c.cnt.cpu_execs == c.cnt.misses


def test_full_capacity_misses_are_first_touches():
    w = synth.decode_bf16().with_(n_layers=3, n_experts=32, steps=40)
    w = w.with_(cache_slots=w.n_logical)
    tr = synth.routing_trace(w)
    c = O.SlotCache(w.cache_slots, w.n_logical)
    seen = set()
    first = 0
    for s in range(w.steps):
        for l in range(w.n_layers):
            sel, _ = O.route(synth.decode_logits(w, s, l, tr), w.top_k)
            A = O.dedupe(sel, l, w.n_experts)
            first += len(set(A) - seen)
            seen |= set(A)
            c.decode_step(l, w.n_experts, sel, 80000, 50000)      # B_H < B_P: q = m
    assert c.cnt.misses == first and c.cnt.evictions == 0


# --------------------------------------------------------------- expert maths
def test_e4m3_decoder_points_and_exhaustive_vs_torch():
    torch = pytest.importorskip("torch")
    for code, val in _rows("e4m3_points.txt"):
        v = O.e4m3_to_f64(np.array([int(code, 16)], dtype=np.uint8))[0]
        assert v == float(val) and math.copysign(1, v) == math.copysign(1, float(val))
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).double().numpy()
    mine = O.e4m3_to_f64(codes)
    ok = ~np.isnan(ref)
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    assert np.array_equal(mine[ok], ref[ok])


def test_e4m3_normals_match_exponent_rebias_bit_trick():
    # "OSDI'26 | 双路 CPU…", §4.2: an E4M3 normal becomes a valid BF16 by adding 120
    # to the exponent and zero-filling the mantissa (integer shifts only).
    for code in range(256):
        e = (code >> 3) & 0xF
        if e == 0 or (code & 0x7F) == 0x7F:
            continue
        bf = ((code & 0x80) << 8) | ((e + 120) << 7) | ((code & 0x7) << 4)
        v = np.array([bf << 16], dtype=np.uint32).view(np.float32)[0]
        assert O.e4m3_to_f64(np.array([code], dtype=np.uint8))[0] == float(v)


def test_bf16_decode_matches_torch():
    torch = pytest.importorskip("torch")
    bits = np.random.default_rng(0).integers(0, 1 << 16, 5000).astype(np.uint16)
    bits = bits[((bits >> 7) & 0xFF) != 0xFF]      # drop inf/nan patterns
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    assert np.array_equal(O.bf16_to_f64(bits), ref)


def _loop_swiglu(Wg, Wu, Wd, x):
    I, H = len(Wg), len(Wg[0])
    a = [sum(Wg[i][j] * x[j] for j in range(H)) for i in range(I)]
    b = [sum(Wu[i][j] * x[j] for j in range(H)) for i in range(I)]
    h = [a[i] / (1.0 + math.exp(-a[i])) * b[i] for i in range(I)]
    return [sum(Wd[o][i] * h[i] for i in range(I)) for o in range(H)]


def test_swiglu_bf16_brute_force_loops():
    rng = np.random.default_rng(5)
    H, I = 12, 5                      # non-square: a transposed operand cannot pass
    ex = {"gate": synth.f32_to_bf16_bits(rng.standard_normal((I, H)).astype(np.float32)),
          "up": synth.f32_to_bf16_bits(rng.standard_normal((I, H)).astype(np.float32)),
          "down": synth.f32_to_bf16_bits(rng.standard_normal((H, I)).astype(np.float32))}
    xb = synth.f32_to_bf16_bits(rng.standard_normal(H).astype(np.float32))
    f = lambda a: O.bf16_to_f64(a).tolist()
    ref = _loop_swiglu(f(ex["gate"]), f(ex["up"]), f(ex["down"]), f(xb))
    np.testing.assert_allclose(O.swiglu_expert(ex, O.bf16_to_f64(xb), fp8=False), ref, rtol=1e-12, atol=1e-12)


def test_swiglu_fp8_post_scaling_vs_dequant_first_and_loops():
    w = synth.decode_fp8().with_(hidden=256, inter=128)
    pool = synth.ExpertPool(w)
    ex = pool.expert(17)
    x = O.bf16_to_f64(synth.decode_x(w, 0, 0)[0])
    y = O.swiglu_expert(ex, x, fp8=True)
    # dequantise first (scale*w elementwise), then plain dot products
    deq = lambda c, s: O.e4m3_to_f64(c) * np.repeat(s.astype(np.float64), 128, axis=1)
    Wg, Wu, Wd = deq(ex["gate"], ex["gate_scale"]), deq(ex["up"], ex["up_scale"]), deq(ex["down"], ex["down_scale"])
    np.testing.assert_allclose(y, Wd @ (O.silu(Wg @ x) * (Wu @ x)), rtol=1e-10, atol=1e-13)
    ref = _loop_swiglu(Wg.tolist(), Wu.tolist(), Wd.tolist(), x.tolist())
    np.testing.assert_allclose(y, ref, rtol=1e-9, atol=1e-12)


def test_silu_closed_form():
    for a in [-30.0, -2.0, -0.5, 0.0, 0.5, 3.0, 30.0]:
        assert O.silu(np.array([a]))[0] == pytest.approx(a * (1 / (1 + math.exp(-a))), rel=1e-15)
    assert O.silu(np.array([0.0]))[0] == 0.0


# ------------------------------------------------ layer output & identities
def _dense_moe(pool, w, layer, z, xbits, shared=None):
    """All-expert formulation: sum over every expert e of [e in top-k] * gate_e * SwiGLU_e(x)."""
    E, k = w.n_experts, w.top_k
    x = O.bf16_to_f64(xbits)
    zz = [float(v) for v in z]
    rank = [sum(1 for j in range(E) if zz[j] > zz[e] or (zz[j] == zz[e] and j < e)) for e in range(E)]
    members = [e for e in range(E) if rank[e] < k]
    zmax = max(zz[e] for e in members)
    den = sum(math.exp(zz[e] - zmax) for e in members)
    out = np.zeros(w.hidden) if shared is None else O.swiglu_expert(shared, x, False)
    for e in range(E):
        if rank[e] < k:
            g = np.float32(math.exp(zz[e] - zmax) / den)
            out = out + float(g) * O.swiglu_expert(pool.expert(layer * E + e), x, False)
    return out


def test_routed_layer_equals_dense_all_expert_sum():
    w = synth.tiny()
    pool = synth.ExpertPool(w)
    c = O.SlotCache(w.n_logical, w.n_logical)
    for s in range(3):
        for l in range(w.n_layers):
            z = synth.decode_logits(w, s, l)
            xb = synth.decode_x(w, s, l)
            sel, gates = O.route(z, w.top_k)
            rec = c.decode_step(l, w.n_experts, sel, 80000, 50000)
            out = O.decode_layer_outputs(rec, sel, gates, xb, None, pool.expert, n_experts=w.n_experts)
            np.testing.assert_allclose(out[0], _dense_moe(pool, w, l, z[0], xb[0]), rtol=1e-12, atol=1e-14)


def test_output_independent_of_capacity_and_split():
    w = synth.decode_bf16().with_(n_layers=2, n_experts=32, hidden=128, inter=64, batch=3, steps=6)
    pool = synth.ExpertPool(w)
    shared = pool.shared(0)
    tr = synth.routing_trace(w)
    outs = {}
    for S, (bp, bh) in [(64, (80000, 50000)), (5, (11800, 47500)), (9, (52700, 77300)), (3, (25000, 50000))]:
        c = O.SlotCache(S, w.n_logical)
        res = []
        for s in range(w.steps):
            for l in range(w.n_layers):
                z = synth.decode_logits(w, s, l, tr)
                xb = synth.decode_x(w, s, l)
                sel, gates = O.route(z, w.top_k)
                rec = c.decode_step(l, w.n_experts, sel, bp, bh)
                cp = O.all_pair_rows(l, sel, gates, xb, pool.expert, w.n_experts)
                res.append(O.decode_layer_outputs(rec, sel, gates, xb, cp, pool.expert,
                                                  shared=pool.shared(l), n_experts=w.n_experts))
        outs[S] = np.stack(res)
    base = outs[64]
    for S, o in outs.items():
        np.testing.assert_array_equal(o, base)


def test_c_rows_are_used_for_host_pairs():
    # a planted C row must appear in the output exactly where the pair is in C
    w = synth.tiny()
    pool = synth.ExpertPool(w)
    c = O.SlotCache(1, w.n_logical)
    z = synth.decode_logits(w, 0, 0)
    xb = synth.decode_x(w, 0, 0)
    sel, gates = O.route(z, w.top_k)
    rec = c.decode_step(0, w.n_experts, sel, 11800, 47500)     # m=2, q=1 -> one C pair
    assert rec.q == 1 and len(rec.C) == 1
    cp = np.zeros((1, w.top_k, w.hidden))
    r_c = [r for r in range(w.top_k) if rec.slot_of_pair[0, r] == O.FT_CPU][0]
    cp[0, r_c, :] = 1000.0
    out = O.decode_layer_outputs(rec, sel, gates, xb, cp, pool.expert, n_experts=w.n_experts)
    r_g = 1 - r_c
    g_row = O.pair_row(pool.expert(int(sel[0, r_g])), O.bf16_to_f64(xb[0]), gates[0, r_g], False)
    np.testing.assert_allclose(out[0], g_row + 1000.0, rtol=1e-15)


# ------------------------------------------------------------------ prefill
def test_prefill_double_buffer_state_and_output():
    w = synth.prefill().with_(n_layers=5, n_experts=8, hidden=64, inter=32, cache_slots=20, prefill_tokens=24)
    pool = synth.ExpertPool(w)
    c = O.SlotCache(w.cache_slots, w.n_logical)
    # some decode history first so that prefill must evict and invalidate
    for s in range(4):
        for l in range(w.n_layers):
            sel, _ = O.route(synth.decode_logits(w.with_(logits="normal"), s, l), w.top_k)
            c.decode_step(l, w.n_experts, sel, 80000, 50000)
    bufs = []
    for l in range(w.n_layers):
        clock_before = c.clock
        buf = c.prefill_layer(l, w.n_experts, w.n_layers)
        bufs.append(buf)
        assert len(set(buf)) == w.n_experts
        for e in range(w.n_experts):
            assert c.res[l * w.n_experts + e] == buf[e]
            assert c.stamp[buf[e]] == clock_before + 1
        if l >= 2:
            assert bufs[l] == bufs[l - 2]
            assert all(c.res[(l - 2) * w.n_experts + e] < 0 for e in range(w.n_experts))
        _check_state_bijection(c)
    assert not set(bufs[0]) & set(bufs[1])
    # prefill output of a few tokens equals the decode-path evaluation with every pair resident
    l = w.n_layers - 1
    T = w.prefill_tokens
    z = synth.prefill_logits(w, 0, l, T)
    xb = synth.prefill_x(w, 0, l, T)
    sel, gates = O.route(z, w.top_k)
    out = O.prefill_outputs(l, sel, gates, xb, pool.expert, w.n_experts, tokens=[0, 5, 23])
    for i, t in enumerate([0, 5, 23]):
        np.testing.assert_allclose(out[i], _dense_moe(pool, w, l, z[t], xb[t]), rtol=1e-12, atol=1e-14)


def test_prefill_chunk_restart_takes_least_recent_slots():
    c = O.SlotCache(10, 3 * 4)
    c.stamp[:] = [5, 1, 9, 0, 3, 7, 2, 8, 4, 6]
    c.clock = 9
    buf = c.prefill_layer(0, 4, 3)
    assert buf == [3, 1, 6, 4]             # stamps 0,1,2,3
    buf1 = c.prefill_layer(1, 4, 3)
    assert buf1 == [8, 0, 9, 5]            # stamps 4,5,6,7


# -------------------------------------------------------------------- resize
def test_resize_keeps_most_recent_and_output_unchanged():
    w = synth.decode_bf16().with_(n_layers=3, n_experts=16, hidden=64, inter=32, steps=8, batch=2)
    pool = synth.ExpertPool(w)
    tr = synth.routing_trace(w)
    c = O.SlotCache(24, w.n_logical)
    for s in range(6):
        for l in range(w.n_layers):
            sel, _ = O.route(synth.decode_logits(w, s, l, tr), w.top_k)
            c.decode_step(l, w.n_experts, sel, 80000, 50000)
    occ = [s for s in range(c.S) if c.owner[s] >= 0]
    newest = sorted(occ, key=lambda s: (-int(c.stamp[s]), s))[:10]
    kept_u = {int(c.owner[s]) for s in newest}
    kept_stamp = {int(c.owner[s]): int(c.stamp[s]) for s in newest}
    moves = c.resize(10)
    assert c.S == 10
    assert {int(u) for u in c.owner if u >= 0} == kept_u
    assert {int(c.owner[s]): int(c.stamp[s]) for s in range(10) if c.owner[s] >= 0} == kept_stamp
    assert all(src >= 10 and dst < 10 for src, dst in moves)
    _check_state_bijection(c)
    c.resize(30)
    assert c.S == 30 and all(c.owner[10:] == -1) and all(c.stamp[10:] == 0)


def test_resize_pairs_movers_and_free_slots_in_ascending_order():
    """Hand-worked shrink: keep the new_slots most recent (stamp desc, slot asc), then move
    the kept entries at slots >= new_slots into the free slots below, both ascending."""
    c = O.SlotCache(8, 20)
    c.owner[:] = [10, 11, -1, 13, 14, 15, 16, 17]
    c.stamp[:] = [1, 9, 0, 3, 8, 7, 2, 6]
    for s, u in enumerate(c.owner):
        if u >= 0:
            c.res[u] = s
    c.clock = 9
    moves = c.resize(4)
    assert moves == [(4, 0), (5, 2), (7, 3)]
    assert list(c.owner) == [14, 11, 15, 17] and list(c.stamp) == [8, 9, 7, 6]
    assert [int(c.res[u]) for u in (10, 11, 13, 14, 15, 16, 17)] == [-1, 1, -1, 0, 2, -1, 3]
    # equal stamps at the cut: the lower slot is kept
    c = O.SlotCache(6, 6)
    c.owner[:] = [0, 1, 2, 3, 4, 5]
    c.res[:] = [0, 1, 2, 3, 4, 5]
    c.stamp[:] = [1, 5, 2, 5, 5, 5]
    c.clock = 5
    moves = c.resize(3)
    assert moves == [(3, 0), (4, 2)]
    assert list(c.owner) == [3, 1, 4] and list(c.stamp) == [5, 5, 5]
    assert [int(v) for v in c.res] == [-1, 1, -1, 0, 2, -1]
