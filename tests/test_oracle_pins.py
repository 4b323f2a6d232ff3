"""Pins of the CPU oracle against what the pages and mathematics fix.

Each test checks the oracle against something other than itself: a value the
pages print for a worked example (fixtures under tests/golden/, each with its
citation), a closed form, an exact special case, a brute-force search, or a
float64 computation with an error bound.
"""
import itertools
import math
import os
from collections import OrderedDict
from fractions import Fraction

import numpy as np
import pytest

from moe_expert_offload_gb300 import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    out = []
    for line in open(os.path.join(GOLD, name)):
        line = line.split("#")[0].strip()
        if line:
            out.append(line.split())
    return out


def _bf(v):
    return int(synth.bf16_bits(np.float32(v)).reshape(-1)[0])


# ------------------------------------------------------------------ layout
def test_blob_size_matches_edge0_sizes(oracle):
    g = {k: float(v) for k, v in _rows("edge0_sizes.txt")}
    L, E, H, I = int(g["layers"]), int(g["experts"]), int(g["hidden"]), int(g["inter"])
    se = oracle.expert_bytes(H, I)
    assert se == 1_769_472
    assert round(se / 1e6, 2) == g["per_expert_MB"]
    assert round(se * E / 1e6) == g["per_layer_MB"]
    assert round(se * E * L / 1e9) == g["total_GB"]
    assert round(se * E * L / 2**30, 1) == g["total_GiB"]


def test_blob_offsets_agree_with_packer(oracle):
    for H, I in ((256, 128), (2048, 512), (7168, 2048)):
        off = oracle.blob_offsets(H, I)
        soff, _, total = synth.blob_sections(H, I)
        assert off["total"] == total == oracle.expert_bytes(H, I)
        for k in soff:
            assert off[k] == soff[k]
        assert total % 256 == 0
    assert oracle.expert_bytes(7168, 2048) == 24_772_608
    assert oracle.expert_bytes(256, 128) == 55_296


# ----------------------------------------------------------------- dequant
def test_dequant_hand_worked(oracle):
    # s = 2^-6, b = -2^-3  =>  w = (q - 8) / 64
    s, b = _bf(2.0**-6), _bf(-(2.0**-3))
    assert s == 0x3C80 and b == 0xBE00
    q = np.arange(16, dtype=np.uint8).repeat(4).reshape(1, 64)
    codes = synth.pack_codes(q)
    w = oracle.dequant(codes, np.array([s], np.uint16), np.array([b], np.uint16), 1, 64)
    assert w[0, 0] == -0.125  # q = 0
    assert w[0, 8 * 4] == 0.0  # q = 8
    assert w[0, 63] == 0.109375  # q = 15
    # codes 0..15 each four times, dotted with ones: 4 * sum(q - 8) / 64 = -0.5
    q2 = np.tile(np.arange(16, dtype=np.uint8), 4).reshape(1, 64)
    w2 = oracle.dequant(synth.pack_codes(q2), np.array([s], np.uint16), np.array([b], np.uint16),
                        1, 64)
    assert float(np.sum(w2.astype(np.float64))) == -0.5


def test_nibble_order(oracle):
    # byte 0x1F holds column 0 in its low nibble (15) and column 1 in its high nibble (1)
    codes = np.zeros((1, 32), np.uint8)
    codes[0, 0] = 0x1F
    one, zero = _bf(1.0), _bf(0.0)
    w = oracle.dequant(codes, np.array([one], np.uint16), np.array([zero], np.uint16), 1, 64)
    assert w[0, 0] == 15.0 and w[0, 1] == 1.0 and np.all(w[0, 2:] == 0.0)


def test_group_boundaries(oracle):
    # two rows x 128 columns: every group gets its own scale; the bias picks the group
    rows, cols = 2, 128
    q = np.full((rows, cols), 1, np.uint8)
    s = np.array([_bf(1.0)] * 4, np.uint16)
    b = np.array([_bf(v) for v in (0.0, 10.0, 20.0, 30.0)], np.uint16)
    w = oracle.dequant(synth.pack_codes(q), s, b, rows, cols)
    assert np.all(w[0, :64] == 1.0) and np.all(w[0, 64:] == 11.0)
    assert np.all(w[1, :64] == 21.0) and np.all(w[1, 64:] == 31.0)


# --------------------------------------------------------------------- exp
def _ulp32(v):
    v = abs(v)
    if v == 0:
        return 2.0**-149
    e = math.floor(math.log2(v))
    return 2.0 ** (max(e, -126) - 23)


def test_exp_within_2ulp_of_float64(oracle):
    xs = np.concatenate([np.linspace(-87, 88, 40001), np.linspace(-1, 1, 20001),
                         np.float32(np.random.default_rng(1).uniform(-87, 88, 20000))])
    worst = 0.0
    for x in np.float32(xs):
        got = oracle.exp(float(x))
        ref = math.exp(float(x))
        worst = max(worst, abs(got - ref) / _ulp32(ref))
    assert worst <= 2.0, worst


def test_exp_special_values(oracle):
    assert oracle.exp(0.0) == 1.0
    assert oracle.exp(-100.0) == oracle.exp(-87.0)
    assert oracle.exp(100.0) == oracle.exp(88.0)
    assert math.isfinite(oracle.exp(88.0)) and oracle.exp(-87.0) >= 2.0**-126
    assert abs(oracle.exp(1.0) - math.e) <= 2 * _ulp32(math.e)
    assert oracle.exp(float(np.float32(math.log(2.0)))) == pytest.approx(2.0, rel=2**-22)


def test_sigmoid(oracle):
    assert oracle.sigmoid(0.0) == 0.5
    for z in np.float32(np.linspace(-20, 20, 4001)):
        ref = 1.0 / (1.0 + math.exp(-float(z)))
        got = oracle.sigmoid(float(z))
        assert abs(got - ref) <= 4 * _ulp32(ref)


# ------------------------------------------------------------ router logits
def test_logits_exact_on_integers(oracle):
    rng = np.random.default_rng(3)
    T, E, H = 3, 5, 512
    x = rng.integers(-4, 5, size=(T, H)).astype(np.float32)
    w = rng.integers(-4, 5, size=(E, H)).astype(np.float32)
    l = oracle.router_logits(synth.bf16_bits(x), synth.bf16_bits(w))
    assert np.array_equal(l, (x.astype(np.int64) @ w.astype(np.int64).T).astype(np.float32))


def test_logits_canonical_order_hand_cases():
    import oracle as o
    H = 256
    one = np.zeros((1, H), np.float32)
    w = np.zeros((1, H), np.float32)
    # elements 0, 8, 24 live in chunks 0, 1, 3 -> lanes 0, 1, 3.  Butterfly: step 2 makes
    # lane1 = 1 + 1 = 2, step 1 makes lane0 = 2^24 + 2 (exact).
    one[0, [0, 8, 24]] = 1.0
    w[0, 0], w[0, 8], w[0, 24] = 2.0**24, 1.0, 1.0
    assert o.router_logits(synth.bf16_bits(one), synth.bf16_bits(w))[0, 0] == 2.0**24 + 2
    # elements 0, 8, 16 -> lanes 0, 1, 2.  Step 2: lane0 = 2^24 + 1 -> 2^24 (ties to even),
    # lane1 = 1; step 1: 2^24 + 1 -> 2^24.  The exact sum 2^24 + 2 is NOT reached.
    one[:] = 0.0
    w[:] = 0.0
    one[0, [0, 8, 16]] = 1.0
    w[0, 0], w[0, 8], w[0, 16] = 2.0**24, 1.0, 1.0
    assert o.router_logits(synth.bf16_bits(one), synth.bf16_bits(w))[0, 0] == 2.0**24


def test_logits_error_bound_vs_float64(oracle):
    rng = np.random.default_rng(4)
    for H in (256, 2048, 7168):
        T, E = 2, 16
        xb = synth.bf16_bits(rng.normal(0, 1, (T, H)))
        wb = synth.bf16_bits(rng.normal(0, 0.02, (E, H)))
        l = oracle.router_logits(xb, wb)
        x = synth.bf16_value(xb).astype(np.float64)
        w = synth.bf16_value(wb).astype(np.float64)
        ref = x @ w.T
        bound = H * 2.0**-24 * (np.abs(x) @ np.abs(w).T)
        assert np.all(np.abs(l - ref) <= bound)


# ------------------------------------------------------------------ routing
def test_softmax_topk_vs_float64_two_step(oracle):
    rng = np.random.default_rng(5)
    T, E, k = 64, 64, 8
    logits = rng.normal(0, 2, (T, E)).astype(np.float32)
    ids, w = oracle.route_softmax_topk(logits, k)
    for t in range(T):
        l = logits[t].astype(np.float64)
        order = sorted(range(E), key=lambda e: (-l[e], e))[:k]
        assert list(ids[t]) == order
        p = np.exp(l - l.max())
        p /= p.sum()  # softmax over all experts
        sel = p[order] / p[order].sum()  # keep top-k, renormalise
        assert np.allclose(w[t], sel, rtol=1e-6, atol=0)
        assert abs(float(np.sum(w[t].astype(np.float64))) - 1.0) <= k * 2.0**-24


def test_softmax_topk_ties_prefer_lower_index(oracle):
    logits = np.array([[1.0, 3.0, 3.0, 2.0, 3.0, 0.0]], np.float32)
    ids, w = oracle.route_softmax_topk(logits, 4)
    assert list(ids[0]) == [1, 2, 4, 3]
    assert w[0, 0] == w[0, 1] == w[0, 2]


def _brute_sigmoid_group(s, sel, n_groups, G, k):
    E = len(s)
    gsz = E // n_groups
    score = []
    for g in range(n_groups):
        v = sorted(sel[g * gsz:(g + 1) * gsz], reverse=True)
        score.append(np.float32(v[0]) + np.float32(v[1]))
    best = None
    for sub in itertools.combinations(range(n_groups), G):  # lexicographic order
        tot = sum(float(score[g]) for g in sub)
        if best is None or tot > best[0]:
            best = (tot, sub)
    cand = [e for g in best[1] for e in range(g * gsz, (g + 1) * gsz)]
    bestk = None
    for sub in itertools.combinations(sorted(cand), k):
        key = sorted(sub, key=lambda e: (-sel[e], e))
        vals = [sel[e] for e in key]
        if bestk is None or vals > bestk[0]:
            bestk = (vals, key)
    return bestk[1]


@pytest.mark.parametrize("E,ng,G,k", [(8, 4, 2, 2), (16, 4, 2, 3), (12, 3, 1, 2)])
def test_sigmoid_group_brute_force(oracle, E, ng, G, k):
    rng = np.random.default_rng(E * 100 + k)
    for trial in range(40):
        logits = rng.normal(0, 1.5, (1, E)).astype(np.float32)
        bias = rng.normal(0, 0.3, E).astype(np.float32)
        ids, w = oracle.route_sigmoid_group(logits, bias, ng, G, k, 2.5)
        s = np.array([oracle.sigmoid(float(v)) for v in logits[0]], np.float32)
        sel = (s + bias).astype(np.float32)
        expect = _brute_sigmoid_group(list(s), list(sel), ng, G, k)
        assert list(ids[0]) == expect
        # weights: raw sigmoid values renormalised over the k, then scaled
        ref = s[expect].astype(np.float64) / np.sum(s[expect].astype(np.float64)) * 2.5
        assert np.allclose(w[0], ref, rtol=1e-6)
        assert abs(float(np.sum(w[0].astype(np.float64))) - 2.5) <= 2.5 * 4 * k * 2.0**-24


def test_sigmoid_group_bias_only_steers_selection(oracle):
    # a large bias forces expert 5 in; its weight is still its raw sigmoid share
    logits = np.zeros((1, 8), np.float32)
    bias = np.zeros(8, np.float32)
    bias[5] = 10.0
    ids, w = oracle.route_sigmoid_group(logits, bias, 4, 2, 2, 1.0)
    assert ids[0, 0] == 5
    assert w[0, 0] == w[0, 1] == 0.5


# ----------------------------------------------------------------------- q*
def test_q_star_worked_examples(oracle):
    for m, bp, bh, q, _src in _rows("q_star_examples.txt"):
        assert oracle.q_star(int(m), int(bp), int(bh)) == int(q), _src


def test_q_star_closed_form_and_bounds(oracle):
    for bp, bh in ((52700, 77300), (11800, 47500), (77300, 77300), (1, 3), (2, 4)):
        for m in range(0, 65):
            q = oracle.q_star(m, bp, bh)
            if bh <= bp:
                assert q == m
            else:
                exact = Fraction(m * bp, bh)
                assert q == math.floor(exact + Fraction(1, 2))
            assert 0 <= q <= m
    assert [oracle.q_star(m, 52700, 77300) for m in range(1, 9)] == [1, 1, 2, 3, 3, 4, 5, 5]
    assert [oracle.q_star(m, 11800, 47500) for m in range(1, 9)] == [0, 0, 1, 1, 1, 1, 2, 2]


def test_q_star_balances_fill_and_cpu_time():
    # reader, "Semantic-Aware Expert Caching": S = 1, B_P = 4, B_H = 8, m = 3, q = 2:
    # T_fill = qS/B_P = 0.5 s and T_cpu = (m-q)S/(B_H-B_P) = 0.25 s; the real-valued balance
    # point qS/B_P = (m-q)S/(B_H-B_P) is q = m*B_P/B_H.
    S, BP, BH, m, q = 1, 4, 8, 3, 2
    assert Fraction(q * S, BP) == Fraction(1, 2)
    assert Fraction((m - q) * S, BH - BP) == Fraction(1, 4)
    qs = Fraction(m * BP, BH)
    assert qs * S / BP == (m - qs) * S / (BH - BP)


# --------------------------------------------------------------- control step
def test_lru_victims_worked_example(oracle):
    rows = _rows("lru_victims.txt")
    K = int([r for r in rows if r[0] == "K"][0][1])
    slots = [(int(a), int(b), int(c)) for a, b, c in (r for r in rows if r[0] != "K")]
    S, E = len(slots), 16
    st = oracle.CacheState(E, S)
    for slot, ts, _ in slots:
        st.id_of_slot[slot] = 10 + slot
        st.slot_of_id[10 + slot] = slot
        st.ts[slot] = ts
    st.clock[0] = 30
    before = st.ts.copy()
    # two misses, pure fill (B_H = B_P) -> both victims consumed
    plan = oracle.cache_step(st, E, 0, np.array([0, 1]), K, 100, 100)
    want = [slot for slot, _, v in sorted(slots, key=lambda r: r[1]) if v]
    assert list(plan["victims"]) == want
    assert sorted(plan["fill_slots"]) == sorted(want)
    for slot, _, v in slots:
        assert st.ts[slot] == (plan["now"] if v else before[slot])
    assert plan["now"] == 31


def test_figure2_split(oracle):
    # reader Figure 2: 12 routed experts, 8 of them hit, m = 4 misses -> 1 fill, 3 direct.
    E, S, K = 64, 16, 8
    st = oracle.CacheState(E, S)
    for j in range(8):  # experts 0..7 resident
        st.id_of_slot[j] = j
        st.slot_of_id[j] = j
        st.ts[j] = 1 + j
    st.clock[0] = 10
    plan = oracle.cache_step(st, E, 0, np.arange(12), K, 11800, 47500)
    assert (plan["n_hit"], plan["n_miss"], plan["n_fill"], plan["n_direct"]) == (8, 4, 1, 3)
    assert list(plan["fill_ids"]) == [8] and list(plan["direct_ids"]) == [9, 10, 11]
    assert plan["fill_slots"][0] == 8  # first empty slot (ts 0)


def test_reader_two_miss_example(oracle):
    # reader "System Architecture": m = 2, B_P/B_H = 12/24 -> q = 1: e3 filled, e4 on the CPU side
    E, S = 8, 4
    st = oracle.CacheState(E, S)
    st.id_of_slot[:2] = [1, 2]
    st.slot_of_id[[1, 2]] = [0, 1]
    st.ts[:2] = [5, 6]
    st.clock[0] = 6
    plan = oracle.cache_step(st, E, 0, np.array([1, 2, 3, 4]), 4, 12, 24)
    assert list(plan["hit_ids"]) == [1, 2]
    assert list(plan["fill_ids"]) == [3] and list(plan["direct_ids"]) == [4]


class BruteLRU:
    """Independent recency simulator: a dict of resident ids plus an ordered log."""

    def __init__(self, S):
        self.S = S
        self.res = {}  # id -> slot
        self.slots = [None] * S  # slot -> id
        self.last = OrderedDict((s, 0) for s in range(S))  # slot -> last use step
        self.step = 0

    def run(self, E, layer, ids, K, bp, bh):
        self.step += 1
        now = self.step
        U = sorted({layer * E + int(i) for i in ids})
        H = [u for u in U if u in self.res]
        for u in H:
            self.last[self.res[u]] = now
        M = [u for u in U if u not in self.res]
        m = len(M)
        if bh <= bp:
            q = m
        else:
            q = math.floor(Fraction(m * bp, bh) + Fraction(1, 2))
        cands = [s for s in range(self.S) if self.last[s] != now]
        # repeated linear scans for the oldest, as a classic LRU would do per eviction
        victims = []
        pool = list(cands)
        while pool and len(victims) < K:
            best = min(pool, key=lambda s: (self.last[s], s))
            victims.append(best)
            pool.remove(best)
        n_fill = min(q, len(victims))
        evicted = []
        for i in range(n_fill):
            v = victims[i]
            old = self.slots[v]
            if old is not None:
                del self.res[old]
            evicted.append(-1 if old is None else old)
            self.slots[v] = M[i]
            self.res[M[i]] = v
            self.last[v] = now
        return dict(uniq=U, hit=H, fill=M[:n_fill], fill_slots=victims[:n_fill],
                    direct=M[n_fill:], victims=victims, evicted=evicted, q=q)


@pytest.mark.parametrize("seed", range(6))
def test_control_step_equals_brute_force_lru(oracle, seed):
    rng = np.random.default_rng(seed)
    E, L = 16, 3
    S = int(rng.integers(1, 12))
    K = int(rng.integers(1, 6))
    bp, bh = [(52700, 77300), (11800, 47500), (77300, 77300), (5, 3)][seed % 4]
    st = oracle.CacheState(L * E, S)
    ref = BruteLRU(S)
    for step in range(120):
        layer = step % L
        T = int(rng.integers(1, 4))
        ids = rng.integers(0, E, size=(T, 2))
        plan = oracle.cache_step(st, E, layer, ids, K, bp, bh)
        r = ref.run(E, layer, ids.reshape(-1), K, bp, bh)
        assert list(plan["uniq"]) == r["uniq"]
        assert list(plan["hit_ids"]) == r["hit"]
        assert list(plan["fill_ids"]) == r["fill"]
        assert list(plan["fill_slots"]) == r["fill_slots"]
        assert list(plan["direct_ids"]) == r["direct"]
        assert list(plan["evicted_ids"]) == r["evicted"]
        assert [v for v in plan["victims"] if v >= 0] == r["victims"]
        assert plan["q"] == r["q"]
        # invariants: the tables are a bijection between resident ids and used slots
        used = st.id_of_slot >= 0
        assert np.all(st.slot_of_id[st.id_of_slot[used]] == np.nonzero(used)[0])
        assert np.sum(st.slot_of_id >= 0) == np.sum(used)
        assert plan["n_hit"] + plan["n_fill"] + plan["n_direct"] == plan["n_uniq"]
        assert set(plan["fill_ids"]) <= set(plan["uniq"]) - set(plan["hit_ids"])


def test_control_step_rejects_bad_ids(oracle):
    st = oracle.CacheState(16, 4)
    with pytest.raises(ValueError):
        oracle.cache_step(st, 16, 0, np.array([3, 16]), 2, 1, 2)


# ------------------------------------------------ replacement policies (1, 2)
@pytest.mark.parametrize("seed", range(6))
def test_layer_lru_equals_independent_lru_per_layer(oracle, seed):
    """Edge0 §3.1 "hot" path: a fixed per-layer resident set.  Policy 1 over an
    interleaved multi-layer trace must act as L separate LRU caches of S_l =
    floor(S / L) slots, each seeing only its own layer's steps, at slot offset
    l * S_l; the slots past L * S_l are never used."""
    rng = np.random.default_rng(100 + seed)
    E, L = 12, 3
    S = int(rng.integers(L, 14))
    Sl = S // L
    K = int(rng.integers(1, 6))
    bp, bh = [(52700, 77300), (11800, 47500), (77300, 77300)][seed % 3]
    st = oracle.CacheState(L * E, S)
    refs = [BruteLRU(Sl) for _ in range(L)]
    for step in range(150):
        layer = int(rng.integers(0, L))  # uneven, random layer order
        ids = rng.integers(0, E, size=(int(rng.integers(1, 4)), 2))
        plan = oracle.cache_step(st, E, layer, ids, K, bp, bh, policy=oracle.LAYER_LRU, L=L)
        r = refs[layer].run(E, layer, ids.reshape(-1), K, bp, bh)
        off = layer * Sl
        assert list(plan["hit_ids"]) == r["hit"]
        assert list(plan["fill_ids"]) == r["fill"]
        assert list(plan["fill_slots"]) == [off + v for v in r["fill_slots"]]
        assert list(plan["direct_ids"]) == r["direct"]
        assert list(plan["evicted_ids"]) == r["evicted"]
        assert [v for v in plan["victims"] if v >= 0] == [off + v for v in r["victims"]]
        assert plan["q"] == r["q"]
        for v in np.nonzero(st.id_of_slot >= 0)[0]:
            assert v < L * Sl and st.id_of_slot[v] // E == v // Sl


def test_layer_lru_closed_forms(oracle):
    """With room for a whole layer (S_l >= E) and pure fill, an LRU misses each
    id exactly once (compulsory misses only); with S_l = 1 and one new expert
    per step it misses on every change of expert and hits on every repeat."""
    E, L, K = 8, 2, 8
    st = oracle.CacheState(L * E, L * E)
    rng = np.random.default_rng(7)
    seen, misses = set(), 0
    for step in range(200):
        layer = step % L
        ids = rng.integers(0, E, size=3)
        plan = oracle.cache_step(st, E, layer, ids, K, 77300, 77300,
                                 policy=oracle.LAYER_LRU, L=L)
        misses += plan["n_miss"]
        seen |= {layer * E + int(i) for i in ids}
    assert misses == len(seen)
    st = oracle.CacheState(L * E, L)
    seq = [3, 3, 5, 5, 5, 2, 3, 3]
    got = [oracle.cache_step(st, E, 1, np.array([e]), 1, 77300, 77300, policy=oracle.LAYER_LRU,
                             L=L)["n_hit"] for e in seq]
    assert got == [0, 1, 0, 1, 1, 0, 0, 1]
    assert st.id_of_slot[0] == -1 and st.id_of_slot[1] == E + 3


@pytest.mark.parametrize("seed", range(3))
def test_static_policy_is_membership(oracle, seed):
    """Policy 2 (the pages' static baselines): the placed set never changes,
    a routed id hits iff it was placed, and every miss goes to C (q = 0)."""
    rng = np.random.default_rng(200 + seed)
    E, L, S = 16, 4, 20
    placed = rng.choice(L * E, size=S - 3, replace=False)
    st = oracle.CacheState(L * E, S)
    oracle.cache_place(st, E, L, placed, policy=oracle.STATIC)
    soi, ios = st.slot_of_id.copy(), st.id_of_slot.copy()
    pset = set(int(u) for u in placed)
    for step in range(100):
        layer = step % L
        ids = rng.integers(0, E, size=(2, 3))
        plan = oracle.cache_step(st, E, layer, ids, 4, 52700, 77300, policy=oracle.STATIC, L=L)
        U = sorted({layer * E + int(i) for i in ids.reshape(-1)})
        assert list(plan["hit_ids"]) == [u for u in U if u in pset]
        assert list(plan["direct_ids"]) == [u for u in U if u not in pset]
        assert plan["q"] == 0 and plan["n_fill"] == 0
        assert np.array_equal(st.slot_of_id, soi) and np.array_equal(st.id_of_slot, ios)


def test_placed_slots_are_first_victims_until_used(oracle):
    """A placed slot has ts 0 (placed, not yet used): under the shared LRU the placed but
    unrouted slots are taken first, in slot order, before any slot routed since; a placed
    id that is routed is a hit and leaves the victim list."""
    E, L, S, K = 8, 2, 6, 6
    st = oracle.CacheState(L * E, S)
    placed = [9, 2, 14, 5]  # slots 0..3; slots 4, 5 empty (ts 0 too)
    oracle.cache_place(st, E, L, placed)
    plan = oracle.cache_step(st, E, 0, np.array([2, 7]), K, 77300, 77300)  # 2 hits, 7 misses
    assert list(plan["hit_ids"]) == [2] and list(plan["hit_slots"]) == [1]
    assert [v for v in plan["victims"] if v >= 0] == [0, 2, 3, 4, 5]
    assert list(plan["fill_slots"]) == [0] and list(plan["evicted_ids"]) == [9]
    plan = oracle.cache_step(st, E, 1, np.array([0, 1, 2]), K, 77300, 77300)  # ids 8, 9, 10
    # slots 2, 3, 4, 5 still have ts 0; slots 0 (id 7) and 1 (id 2) were used at steps 1
    assert [v for v in plan["victims"] if v >= 0] == [2, 3, 4, 5, 0, 1]
    assert list(plan["fill_slots"]) == [2, 3, 4]
    assert list(plan["evicted_ids"]) == [14, 5, -1]


def test_cache_place_layout_and_errors(oracle):
    E, L, S = 10, 3, 10
    st = oracle.CacheState(L * E, S)
    ids = [25, 3, 14, 4, 11]
    for policy in (oracle.SHARED_LRU, oracle.STATIC):
        oracle.cache_place(st, E, L, ids, policy=policy)
        assert list(st.id_of_slot) == ids + [-1] * (S - len(ids))
        assert [st.slot_of_id[u] for u in ids] == list(range(len(ids)))
        assert np.sum(st.slot_of_id >= 0) == len(ids)
        assert not st.ts.any() and st.clock[0] == 0
    # per-layer: S_l = 3; layer 0 -> slots 0.., layer 1 -> 3.., layer 2 -> 6..; slot 9 unused
    oracle.cache_place(st, E, L, ids, policy=oracle.LAYER_LRU)
    assert list(st.id_of_slot) == [3, 4, -1, 14, 11, -1, 25, -1, -1, -1]
    bad = [[3, 3], [30], [-1], list(range(11)), [0, 1, 2, 5]]  # dup, range, range, > S, > S_l
    for b in bad:
        with pytest.raises(ValueError):
            oracle.cache_place(st, E, L, b, policy=oracle.LAYER_LRU if b == [0, 1, 2, 5]
                               else oracle.SHARED_LRU)
    with pytest.raises(ValueError):
        oracle.cache_step(oracle.CacheState(L * E, 2), E, 0, np.array([1]), 1, 1, 2,
                          policy=oracle.LAYER_LRU, L=L)  # S < L
    with pytest.raises(ValueError):
        oracle.cache_step(st, E, 0, np.array([1]), 1, 1, 2, policy=3, L=L)


# ---------------------------------------------------------------------- FFN
def _uniform_expert(H, I, code, s, b):
    qg = np.full((I, H), code, np.uint8)
    qd = np.full((H, I), code, np.uint8)
    sb = lambda shape, v: np.full(shape, _bf(v), np.uint16)
    return synth.pack_blob(H, I, qg, qg, qd, sb((I, H // 64), s), sb((I, H // 64), b),
                           sb((I, H // 64), s), sb((I, H // 64), b), sb((H, I // 64), s),
                           sb((H, I // 64), b))


def test_ffn_closed_form_constant_weights(oracle):
    H, I = 128, 64
    s, b = 2.0**-7, -2.0**-5  # w = s*q + b = (q - 4) / 128; q = 6 -> w0 = 1/64
    blob = _uniform_expert(H, I, 6, s, b)
    x = np.linspace(-1, 1, H).astype(np.float32)
    xb = synth.bf16_bits(x)
    sx = float(np.sum(synth.bf16_value(xb).astype(np.float64)))
    w0 = 1.0 / 64
    g = w0 * sx
    h = g / (1.0 + math.exp(-g)) * g
    y = oracle.expert_forward(blob, H, I, xb)
    assert np.allclose(y[0], w0 * I * h, rtol=1e-12, atol=1e-15)


def test_ffn_one_hot_structure(oracle):
    # gate row i picks x[(2i+1) % H], up row i picks 2*x[(3i+2) % H], down row o picks
    # h[(5o+3) % I]: a transposed or mis-indexed operand changes the answer.
    H, I = 192, 128
    s = 2.0**-4
    qg = np.full((I, H), 8, np.uint8)
    qu = np.full((I, H), 8, np.uint8)
    qd = np.full((H, I), 8, np.uint8)
    for i in range(I):
        qg[i, (2 * i + 1) % H] = 9
        qu[i, (3 * i + 2) % H] = 10
    for o in range(H):
        qd[o, (5 * o + 3) % I] = 9
    sv = lambda shape: np.full(shape, _bf(s), np.uint16)
    bv = lambda shape: np.full(shape, _bf(-8 * s), np.uint16)
    blob = synth.pack_blob(H, I, qg, qu, qd, sv((I, H // 64)), bv((I, H // 64)),
                           sv((I, H // 64)), bv((I, H // 64)), sv((H, I // 64)), bv((H, I // 64)))
    rng = np.random.default_rng(7)
    xb = synth.bf16_bits(rng.normal(0, 4, H))
    x = synth.bf16_value(xb).astype(np.float64)
    y = oracle.expert_forward(blob, H, I, xb)[0]
    for o in range(H):
        i = (5 * o + 3) % I
        g = s * x[(2 * i + 1) % H]
        u = 2 * s * x[(3 * i + 2) % H]
        hval = g / (1.0 + math.exp(-g)) * u
        assert y[o] == pytest.approx(s * hval, rel=1e-12, abs=1e-300)


def test_moe_ffn_is_weighted_sum_plus_shared(oracle):
    H, I, E = 128, 64, 4
    bank = synth.make_bank(E + 1, H, I, seed=11)
    rng = np.random.default_rng(8)
    xb = synth.bf16_bits(rng.normal(0, 1, (3, H)))
    ids = np.array([[2, 0], [1, 3], [3, 3]], np.int32)
    w = np.array([[0.75, 0.25], [0.5, 0.5], [0.25, 0.125]], np.float32)
    y = oracle.moe_ffn(bank[:E], H, I, xb, ids, w, shared_blob=bank[E], shared_I=I)
    for t in range(3):
        ref = oracle.expert_forward(bank[E], H, I, xb[t])[0]
        for j in range(2):
            ref = ref + float(w[t, j]) * oracle.expert_forward(bank[ids[t, j]], H, I, xb[t])[0]
        assert np.allclose(y[t], ref, rtol=1e-12, atol=1e-12)
    # shared expert alone: zero routing weights
    y0 = oracle.moe_ffn(bank[:E], H, I, xb, ids, np.zeros_like(w), shared_blob=bank[E], shared_I=I)
    assert np.allclose(y0, oracle.expert_forward(bank[E], H, I, xb), rtol=1e-12, atol=1e-12)


def test_threaded_row_loops_give_identical_bits(oracle):
    """The timed all-cores baseline runs the oracle's row loops on several host
    threads; every output row is still one thread's sum in the same order, so the
    dequantised matrices and the float64 outputs equal the one-thread results."""
    H, I, E = 256, 128, 6
    bank = synth.make_bank(E + 1, H, I, seed=21)
    rng = np.random.default_rng(9)
    xb = synth.bf16_bits(rng.normal(0, 1, (2, H)))
    ids = np.array([[4, 1, 0], [2, 2, 5]], np.int32)
    w = np.array([[0.5, 0.3, 0.2], [0.6, 0.1, 0.3]], np.float32)
    try:
        oracle.set_threads(1)
        y1 = oracle.moe_ffn(bank[:E], H, I, xb, ids, w, shared_blob=bank[E], shared_I=I)
        d1 = [oracle.blob_matrix(bank[3], H, I, m) for m in range(3)]
        n = oracle.set_threads(4)
        yn = oracle.moe_ffn(bank[:E], H, I, xb, ids, w, shared_blob=bank[E], shared_I=I)
        dn = [oracle.blob_matrix(bank[3], H, I, m) for m in range(3)]
    finally:
        oracle.set_threads(1)
    assert n in (1, 4)
    assert np.array_equal(y1.view(np.uint64), yn.view(np.uint64))
    for a, b in zip(d1, dn):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
