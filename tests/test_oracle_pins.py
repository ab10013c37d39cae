"""Pins of the oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: numbers the
pages print (fixtures under tests/golden/, each citing its page and section),
closed forms, brute force on tiny inputs, and structural invariants.
"""

import math
import random

import numpy as np
import pytest

from conftest import read_golden
from oracle import attention as oatt
from oracle import scheduler as oscheduler
from oracle import speculative as ospec
from oracle.harness import run_bookkeeping
from oracle.hicache import TwoTierRadixCache
from oracle.radix_cache import NoSpace, RadixCache, StateError
from radix_tree_prefix_gb300 import workloads


# ----------------------------------------------------------------- golden
def _toy_fixture():
    lines = read_golden("toy_trie_reuse.txt")
    reqs, exp, total = [], [], None
    mode = None
    for ln in lines:
        if ln == "requests:":
            mode = "r"
        elif ln == "expected:":
            mode = "e"
        elif ln.startswith("total:"):
            total = ln.split()[1]
        elif mode == "r":
            reqs.append(ln.split(" "))
        elif mode == "e":
            exp.append(tuple(int(x) for x in ln.split()))
    return reqs, exp, total


def test_toy_trie_reuse_counts():
    """Per-request reuse printed by the toy prefix tree listing."""
    reqs, expected, total = _toy_fixture()
    vocab = {}
    cache = RadixCache(1000)
    got = []
    for words in reqs:
        toks = [vocab.setdefault(w, len(vocab)) for w in words]
        slots, node = cache.match_prefix(toks)
        new = cache.alloc(len(toks) - len(slots))
        cache.insert(toks, slots + new)
        got.append((len(toks), len(slots)))
    assert got == expected
    cached = sum(h for _, h in got)
    n = sum(t for t, _ in got)
    assert f"{cached}/{n}" == total


def _golden_kv(name):
    out = {}
    for ln in read_golden(name):
        parts = ln.split()
        if parts[0] != "case":
            out[parts[0]] = int(parts[1])
    return out


def test_nested_example_prefill_counts():
    """12,960 / 6,660 / 3,060 prompt tokens prefilled."""
    g = _golden_kv("nested_prefill_counts.txt")
    wl = workloads.nested_share()
    waves = wl.oracle_waves()
    prompts = [p for _, p, _ in waves[0]]
    # no sharing: every prompt prefilled in full
    assert sum(len(p) for p in prompts) == g["no_sharing"]
    # instruction block only: the block is prefilled once, then every request
    # reuses it and nothing else (inserts disabled)
    cache = RadixCache(wl.num_slots)
    instr = prompts[0][:900]
    cache.insert(instr, cache.alloc(900))
    pre = 900
    for p in prompts:
        slots, _ = cache.match_prefix(p[:-1])
        pre += len(p) - len(slots)
    assert pre == g["instruction_only"]
    # the radix tree at all levels, with the in-batch rule
    trace, _ = run_bookkeeping(waves, wl.num_slots, 0)
    assert trace.prefilled == g["radix_tree"]
    assert [[rid for rid, _, _ in b] for b in trace.batches] == \
        [[0], [1, 2, 3, 4], [5, 6, 7]]


def test_agent_step5_reuse():
    """2,800 of 3,000 tokens reused at agent step 5."""
    g = _golden_kv("agent_step_reuse.txt")
    rng = random.Random(5)
    instr = [rng.randrange(32000) for _ in range(g["instructions"])]
    steps = [[rng.randrange(32000) for _ in range(g["per_step"])]
             for _ in range(g["step"])]
    waves = []
    for k in range(1, g["step"] + 1):
        prompt = instr + sum(steps[:k], [])
        waves.append([(k, prompt, [])])
    trace, _ = run_bookkeeping(waves, 10000, 0)
    rid, m, row = trace.batches[g["step"] - 1][0]
    assert len(row) == g["prompt_tokens"]
    assert m == g["reused"]


def _worked_cache(locked):
    g = _golden_kv("worked_eviction.txt")
    cache = RadixCache(g["capacity"] + 1)
    rng = random.Random(7)
    seq = lambda n: [rng.randrange(32000) for _ in range(n)]
    s = seq(g["S"])
    branches = {b: seq(g[b]) for b in "ABC"}
    nodes = {}
    for b in "ABC":      # A used longest ago, then B, then C
        toks = s + branches[b]
        slots, _ = cache.match_prefix(toks)
        new = cache.alloc(len(toks) - len(slots))
        _, nodes[b] = cache.insert(toks, slots + new)
    assert cache.cached_size() == g["S"] + g["A"] + g["B"] + g["C"]
    for b in locked:
        cache.inc_lock_ref(nodes[b])
    d = s + seq(g["D_new"])
    slots, dnode = cache.match_prefix(d[:-1])
    assert len(slots) == g["S"]
    cache.inc_lock_ref(dnode)
    return cache, nodes, d, slots, g


@pytest.mark.parametrize("locked,victim,held", [
    ("C", "A", 3500), ("AC", "B", 3800), ("ABC", None, None)])
def test_worked_eviction_example(locked, victim, held):
    cache, nodes, d, slots, g = _worked_cache(locked)
    if victim is None:
        with pytest.raises(NoSpace):
            cache.alloc(g["D_new"])
        assert cache.eviction_log == []
        return
    new = cache.alloc(g["D_new"])
    assert cache.eviction_log == [(nodes[victim].id, g[victim])]
    cache.insert(d, slots + new)
    assert cache.cached_size() == held


# ------------------------------------------------------------ brute force
def test_match_against_prefix_dictionary():
    """Match length and slots equal a naive dict-of-prefixes trie."""
    rng = random.Random(11)
    for trial in range(300):
        alpha = rng.randint(1, 4)
        cache = RadixCache(2000)
        first_slot = {}          # prefix tuple -> slot of its last token
        for _ in range(rng.randint(1, 8)):
            seq = [rng.randrange(alpha) for _ in range(rng.randint(1, 12))]
            # brute force: longest prefix present in the dictionary
            n = 0
            while n < len(seq) and tuple(seq[:n + 1]) in first_slot:
                n += 1
            want = [first_slot[tuple(seq[:p + 1])] for p in range(n)]
            assert cache.match_length(seq) == n
            slots, node = cache.match_prefix(seq)
            assert slots == want
            new = cache.alloc(len(seq) - n)
            row = slots + new
            already, _ = cache.insert(seq, row)
            assert already == n
            for p in range(len(seq)):
                first_slot.setdefault(tuple(seq[:p + 1]), row[p])
        assert cache.cached_size() == len(first_slot)


def test_split_at_divergence():
    """Second session sharing the system prompt splits the first node."""
    cache = RadixCache(100)
    sys_p = [1, 2, 3, 4]
    a = sys_p + [10, 11]
    b = sys_p + [20, 21, 22]
    cache.insert(a, cache.alloc(len(a)))
    assert cache.num_nodes() == 1
    slots, node = cache.match_prefix(b)
    assert len(slots) == 4 and node.key == sys_p   # split during the match
    assert cache.num_nodes() == 2
    cache.insert(b, slots + cache.alloc(3))
    assert cache.num_nodes() == 3
    keys = sorted(tuple(c.key) for c in node.children.values())
    assert keys == [(10, 11), (20, 21, 22)]


# -------------------------------------------------------------- invariants
def test_lock_and_eviction_invariants():
    """Random operations: accounting, locks and leaf-inward LRU eviction."""
    rng = random.Random(3)
    for trial in range(40):
        n_slots = rng.randint(20, 60)
        cache = RadixCache(n_slots)
        held = {}                  # handle -> (node, slots it owns privately)
        private = 0
        locks = []
        for step in range(80):
            op = rng.random()
            seq = [rng.randrange(3) for _ in range(rng.randint(1, 10))]
            if op < 0.5:
                slots, node = cache.match_prefix(seq[:-1])
                cache.inc_lock_ref(node)
                # snapshot before allocation
                before = {}
                stack = [cache.root]
                while stack:
                    x = stack.pop()
                    before[x.id] = (x.lock_ref, [c.id for c in x.children.values()],
                                    x.last_access_time)
                    stack.extend(x.children.values())
                log0 = len(cache.eviction_log)
                try:
                    new = cache.alloc(len(seq) - len(slots))
                except NoSpace:
                    cache.dec_lock_ref(node)
                    new = None
                evicted = [nid for nid, _ in cache.eviction_log[log0:]]
                for pos, nid in enumerate(evicted):
                    lock, kids, _ = before[nid]
                    assert lock == 0, "locked node evicted"
                    # every child was evicted before its parent
                    for c in kids:
                        assert c in evicted[:pos], "parent evicted before child"
                if evicted:
                    leaves = [(before[i][2], i) for i in before
                              if i != 0 and not before[i][1] and before[i][0] == 0]
                    assert evicted[0] == min(leaves)[1], "not least recent leaf"
                if new is None:
                    continue
                row = slots + new
                already, node2 = cache.insert(seq, row)
                cache.free(row[len(slots):already])
                cache.inc_lock_ref(node2)
                cache.dec_lock_ref(node)
                locks.append(node2)
            elif locks:
                node = locks.pop(rng.randrange(len(locks)))
                cache.dec_lock_ref(node)
            cached = cache.cached_size()
            assert cache.evictable_size_ + cache.protected_size_ == cached
            assert len(cache.free_slots) + cached + private == n_slots - 1
        for node in locks:
            cache.dec_lock_ref(node)
        assert cache.protected_size_ == 0
        with pytest.raises(StateError):
            leaf = next(iter(cache.root.children.values()), None)
            if leaf is None:
                raise StateError("empty")
            cache.dec_lock_ref(leaf)


# --------------------------------------------------------------- attention
def test_single_key_returns_its_value():
    rng = np.random.default_rng(0)
    q = rng.standard_normal((1, 2, 8))
    k = rng.standard_normal((1, 1, 8))
    v = rng.standard_normal((1, 1, 8))
    o, lse = oatt.softmax_attention(q, k, v, [1])
    assert np.array_equal(o[0, 0], v[0, 0]) and np.array_equal(o[0, 1], v[0, 0])
    assert lse[0, 0] == pytest.approx(q[0, 0] @ k[0, 0] / math.sqrt(8), abs=1e-15)


def test_brute_force_in_exact_and_high_precision_arithmetic():
    """Tiny inputs (n <= 8 keys, d = 4) with dyadic entries: q.k is formed
    exactly with fractions, the exponentials and the normalisation at 50
    digits (mpmath), each query seeing a causal prefix; the fp64 oracle must
    agree to 1e-13 in the output and the log-sum-exp."""
    from fractions import Fraction
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    rng = random.Random(7)
    for trial in range(25):
        n = rng.randint(1, 8)
        hq, hkv, d = 2, 1, 4
        dy = lambda: Fraction(rng.randint(-16, 16), 8)   # exact in binary
        q = [[[dy() for _ in range(d)] for _ in range(hq)] for _ in range(n)]
        k = [[[dy() for _ in range(d)] for _ in range(hkv)] for _ in range(n)]
        v = [[[dy() for _ in range(d)] for _ in range(hkv)] for _ in range(n)]
        visible = [i + 1 for i in range(n)]
        o, lse = oatt.softmax_attention(np.array(q, dtype=np.float64),
                                        np.array(k, dtype=np.float64),
                                        np.array(v, dtype=np.float64), visible)
        scale = 1 / mpmath.sqrt(d)            # 1/2 exactly for d = 4
        for i in range(n):
            for h in range(hq):
                dots = [sum(q[i][h][c] * k[j][0][c] for c in range(d)) for j in range(visible[i])]
                s = [mpmath.mpf(x.numerator) / x.denominator * scale for x in dots]
                m = max(s)
                w = [mpmath.exp(x - m) for x in s]
                z = mpmath.fsum(w)
                for c in range(d):
                    want = mpmath.fsum(w[j] * v[j][0][c] for j in range(len(w))) / z
                    assert abs(o[i, h, c] - float(want)) < 1e-13, (trial, i, h, c)
                assert abs(lse[i, h] - float(m + mpmath.log(z))) < 1e-13, (trial, i, h)


def test_two_keys_closed_form():
    """Score gap ln 3 with scale 1/sqrt(d) gives weights 1/4 and 3/4."""
    d = 4
    q = np.zeros((1, 1, d)); q[0, 0, 0] = 1.0
    k = np.zeros((2, 1, d)); k[1, 0, 0] = 2.0 * math.log(3.0)   # sqrt(4) = 2
    v = np.zeros((2, 1, d)); v[0, 0, :] = 1.0; v[1, 0, :] = 5.0
    o, lse = oatt.softmax_attention(q, k, v, [2])
    assert o[0, 0] == pytest.approx(np.full(d, 0.25 * 1 + 0.75 * 5), abs=1e-14)
    assert lse[0, 0] == pytest.approx(math.log(4.0), abs=1e-14)


def test_equal_keys_average_visible_values():
    """Causal boundary: query at position p+i averages values 0..p+i."""
    n, p, d = 9, 4, 3
    k = np.ones((n, 1, d))
    v = np.arange(n, dtype=np.float64)[:, None, None] * np.ones((n, 1, d))
    q = np.ones((n - p, 2, d))
    o, _ = oatt.extend_attention(q, k, v, p)
    for i in range(n - p):
        assert o[i, 0] == pytest.approx(np.full(d, (p + i) / 2.0), abs=1e-13)


def test_gqa_head_mapping():
    """Query head h reads KV head h // G."""
    hq, hkv, d, n = 8, 2, 4, 5
    rng = np.random.default_rng(1)
    q = rng.standard_normal((n, hq, d))
    k = rng.standard_normal((n, hkv, d))
    v = np.zeros((n, hkv, d))
    for j in range(hkv):
        v[:, j, :] = j + 1
    o, _ = oatt.softmax_attention(q, k, v, list(range(1, n + 1)))
    for h in range(hq):
        assert np.allclose(o[:, h, :], h // (hq // hkv) + 1, atol=1e-14)


def test_lse_merge_equals_unsplit():
    rng = np.random.default_rng(2)
    n, hq, hkv, d = 37, 4, 2, 16
    q = rng.standard_normal((1, hq, d))
    k = rng.standard_normal((n, hkv, d))
    v = rng.standard_normal((n, hkv, d))
    full_o, full_l = oatt.softmax_attention(q, k, v, [n])
    parts = []
    for lo, hi in [(0, 5), (5, 6), (6, 30), (30, 37)]:
        o, l = oatt.softmax_attention(q, k[lo:hi], v[lo:hi], [hi - lo])
        parts.append((o, l))
    mo, ml = oatt.lse_merge(parts)
    assert np.allclose(mo, full_o, atol=1e-12)
    assert np.allclose(ml, full_l, atol=1e-12)
    # a single part merges to itself
    so, sl = oatt.lse_merge([(full_o, full_l)])
    assert np.allclose(so, full_o, atol=1e-15) and np.allclose(sl, full_l, atol=1e-15)


def test_cached_prefix_equals_full_recompute():
    """Suffix rows with a cached prefix equal rows of the whole prompt."""
    rng = np.random.default_rng(4)
    n, p, hq, hkv, d = 23, 15, 4, 1, 8
    q = rng.standard_normal((n, hq, d))
    k = rng.standard_normal((n, hkv, d))
    v = rng.standard_normal((n, hkv, d))
    full_o, full_l = oatt.softmax_attention(q, k, v, list(range(1, n + 1)))
    o, l = oatt.extend_attention(q[p:], k, v, p)
    assert np.array_equal(o, full_o[p:]) and np.array_equal(l, full_l[p:])
    do, dl = oatt.decode_attention(q[-1], k, v)
    assert np.array_equal(do, full_o[-1]) and np.array_equal(dl, full_l[-1])


def test_lock_protects_whole_path():
    """inc_lock_ref moves every node from the node up to the root."""
    cache = RadixCache(100)
    a = [1, 2, 3, 4, 10, 11]
    b = [1, 2, 3, 4, 20, 21, 22]
    cache.insert(a, cache.alloc(len(a)))
    slots, _ = cache.match_prefix(b)
    _, leaf_b = cache.insert(b, slots + cache.alloc(3))
    assert (cache.evictable_size_, cache.protected_size_) == (9, 0)
    cache.inc_lock_ref(leaf_b)
    assert (cache.evictable_size_, cache.protected_size_) == (2, 7)
    cache.inc_lock_ref(leaf_b)
    assert (cache.evictable_size_, cache.protected_size_) == (2, 7)
    cache.dec_lock_ref(leaf_b)
    cache.dec_lock_ref(leaf_b)
    assert (cache.evictable_size_, cache.protected_size_) == (9, 0)
    with pytest.raises(StateError):
        cache.dec_lock_ref(leaf_b)


def test_touch_makes_node_recent():
    """A reused branch becomes recent: the least recently used leaf goes.

    "Eviction on a tree" (bibekananda.in): a node touched by requests stays
    warm; the worked example evicts the branch used longest ago.
    """
    cache = RadixCache(100)
    s = [1, 2, 3]
    nodes = {}
    for name, tail in (("A", [10, 11]), ("B", [20, 21]), ("C", [30, 31])):
        toks = s + tail
        slots, _ = cache.match_prefix(toks)
        _, nodes[name] = cache.insert(toks, slots + cache.alloc(len(toks) - len(slots)))
    cache.match_prefix(s + [10, 11])          # user A comes back
    assert cache.evict(1) == 2
    assert cache.eviction_log == [(nodes["B"].id, 2)]
    assert cache.evict(1) == 2
    assert cache.eviction_log[-1] == (nodes["C"].id, 2)


def test_cascade_reaches_parent_after_children():
    """A parent becomes a candidate only once its last child is gone."""
    cache = RadixCache(100)
    a, b = [1, 2, 3, 4], [1, 2, 5, 6]
    cache.insert(a, cache.alloc(4))
    slots, _ = cache.match_prefix(b)
    _, nb = cache.insert(b, slots + cache.alloc(2))
    parent = nb.parent
    assert cache.evict(100) == 6
    ids = [i for i, _ in cache.eviction_log]
    assert ids[-1] == parent.id and len(ids) == 3
    assert cache.cached_size() == 0 and cache.num_nodes() == 0


def test_allocator_fifo_reading():
    """Reading (pages silent): FIFO free list 1..N-1, freed slots at the tail."""
    cache = RadixCache(8)
    assert cache.alloc(3) == [1, 2, 3]
    cache.free([2])
    assert cache.alloc(4) == [4, 5, 6, 7]
    assert cache.alloc(1) == [2]
    with pytest.raises(NoSpace):
        cache.alloc(1)


def test_evicted_slots_return_in_stored_order():
    """Reading (pages silent): an evicted node's slots join the free list tail
    in the order the node stores them."""
    cache = RadixCache(6)
    slots = cache.alloc(5)                     # [1, 2, 3, 4, 5]
    order = [3, 1, 5, 2, 4]
    cache.free([s for s in slots if s not in order])
    cache.insert([7, 8, 9, 10, 11], order)
    assert cache.alloc(5) == order             # forces eviction of the node


def test_pool_store_writes_only_its_slots():
    from oracle import pool as opool
    rng = np.random.default_rng(9)
    base = rng.standard_normal((2, 3, 10, 4))
    kv = rng.standard_normal((3, 3, 4))
    out = opool.store(base, 1, [7, 2, 5], kv)
    for i, s in enumerate([7, 2, 5]):
        assert np.array_equal(out[1, :, s, :], kv[i])
    untouched = [s for s in range(10) if s not in (7, 2, 5)]
    assert np.array_equal(out[1, :, untouched, :], base[1, :, untouched, :])
    assert np.array_equal(out[0], base[0])


# ------------------------------------------------- decode, finish, adoption
def _tree_slots(cache):
    """Every slot the tree holds, node by node."""
    out = []
    stack = [cache.root]
    while stack:
        n = stack.pop()
        out.extend(n.value)
        stack.extend(n.children.values())
    return out


def _assert_slots_conserved(cache):
    """Once every request has finished, each slot outside the pad page is
    either held by exactly one tree position or on the free list (a page is
    free as a whole), never both and never neither (no slot leaked, none
    handed out twice)."""
    held = _tree_slots(cache) + list(cache.free_slots)
    assert sorted(held) == list(range(cache.page_size, cache.num_slots)), \
        "slots leaked or duplicated"
    assert len(set(_tree_slots(cache))) == cache.cached_size()


def _agent_steps_with_actions(actions, seed=5):
    """The agent example run through decode: a 2,000-token preamble and 200
    new tokens per step, of which the first ``actions`` are the previous
    step's decoded action (its outputs) and the rest fresh tool tokens (step
    1's 200 tokens are all fresh).  Step k's prompt has 2,000 + 200 k tokens."""
    g = _golden_kv("agent_step_reuse.txt")
    rng = random.Random(seed)
    fresh = lambda n: [rng.randrange(32000) for _ in range(n)]
    prompt = fresh(g["instructions"]) + fresh(g["per_step"])
    waves = []
    for k in range(1, g["step"] + 1):
        outs = fresh(actions)
        waves.append([(k, list(prompt), outs)])
        prompt = prompt + outs + fresh(g["per_step"] - actions)
    return waves, g


@pytest.mark.parametrize("actions", [0, 8, 32])
def test_agent_steps_through_decode_reuse(actions):
    """"The problem SGLang solves" ("Pause and think"): step 5's prompt of
    3,000 tokens finds 2,800 of them already computed by steps 1-4.  With
    step 4's action decoded before step 5 ("How RadixAttention reuses past
    work", step 4: the output tokens become nodes of the tree at finish),
    step 5 reuses step 4's whole prompt plus that action: 2,800 + D tokens
    for an action of D tokens, and every earlier step k reuses 2,000 +
    200 (k-1) + D.  A finish that drops the outputs reuses only 2,800."""
    waves, g = _agent_steps_with_actions(actions)
    trace, cache = run_bookkeeping(waves, 10000, actions)
    for k in range(2, g["step"] + 1):
        rid, m, row = trace.batches[k - 1][0]
        assert len(row) == g["instructions"] + g["per_step"] * k
        assert m == g["instructions"] + g["per_step"] * (k - 1) + actions
    rid, m, row = trace.batches[g["step"] - 1][0]
    assert len(row) == g["prompt_tokens"] and m == g["reused"] + actions
    # each step's decoded action sits in the tree on the slots its decode
    # steps allocated (one per step, in order)
    last_rid, last_prompt, last_outs = waves[-1][0]
    full = last_prompt + last_outs
    assert cache.match_length(full) == len(full)
    tree_row = cache.lookup_slots(full)
    for k, wave in enumerate(waves):
        _, prompt, outs = wave[0]
        decoded = [trace.decode_steps[k * actions + t][0][1] for t in range(actions)]
        assert tree_row[len(prompt):len(prompt) + actions] == decoded
    # at finish only the prompt (inserted when its extend ended) is cached
    assert [a for _, a in trace.finishes] == [len(w[0][1]) for w in waves]
    _assert_slots_conserved(cache)


def test_identical_samples_share_prompt_and_free_duplicate_outputs():
    """Two samples of one prompt that decode the same tokens ("One tree for
    everybody": matched state is pointed at, not stored twice).  The second
    request waits for the first (the in-batch rule), recomputes only its last
    prompt token and then points at the first one's slots for the whole
    prompt; at finish the second finds the first's outputs cached and frees
    its own copies.  Afterwards every slot is held exactly once."""
    rng = random.Random(17)
    prompt = [rng.randrange(32000) for _ in range(40)]
    outs = [rng.randrange(32000) for _ in range(6)]
    other = prompt[:10] + [rng.randrange(32000) for _ in range(7)]
    waves = [[(0, prompt, outs), (1, list(prompt), list(outs)),
              (2, other, [rng.randrange(32000) for _ in range(6)])]]
    rows_seen = {}

    def on_decode(step, rows):
        rows_seen[step] = rows

    trace, cache = run_bookkeeping(waves, 200, 6, on_decode=on_decode)
    assert [[rid for rid, _, _ in b] for b in trace.batches] == [[0], [1, 2]]
    _, m1, row1 = trace.batches[1][0]
    assert m1 == len(prompt) - 1
    # the second sample's prompt row is the first's, slot for slot
    for step, rows in rows_seen.items():
        assert rows[1][:len(prompt)] == rows[0][:len(prompt)]
        assert rows[1][len(prompt):] != rows[0][len(prompt):]   # own decode slots
    assert trace.finishes == [(0, len(prompt)), (1, len(prompt) + 6), (2, len(other))]
    assert cache.cached_size() == len(prompt) + 6 + (len(other) - 10) + 6
    _assert_slots_conserved(cache)


def test_chat_turn_reuses_whole_history():
    """Multi-turn chat: turn t+1 of a session is its history (system prompt,
    earlier user turns and the replies decoded for them) plus a new user
    turn, and with a pool that never evicts it reuses the whole history; at
    the end every slot is held exactly once."""
    wl = workloads.multi_turn_chat(sessions=5, turns=4, system=60, user=9, decode_steps=4,
                                   layers=1)
    waves = wl.oracle_waves()
    trace, cache = run_bookkeeping(waves, wl.num_slots, wl.decode_steps)
    hist = {}
    batches = [rec for b in trace.batches for rec in b]
    by_rid = {rid: (m, row) for rid, m, row in batches}
    for wave in waves:
        for rid, prompt, outs in wave:
            m, row = by_rid[rid]
            sess = rid % 5
            want = hist.get(sess, 60 if rid else 0)   # the very first request finds nothing
            assert m == want, (rid, m, want)
            hist[sess] = len(prompt) + len(outs)
    _assert_slots_conserved(cache)


@pytest.mark.parametrize("make", [
    lambda: workloads.agent_loop(calls=7, preamble=120, lo=5, hi=40, decode_steps=5),
    lambda: workloads.fork_tree(branching=3, depth=3, level_tokens=12, decode_steps=3),
    lambda: workloads.long_shared(batch=6, prefix=90, unique=11, decode_steps=4),
])
def test_request_flow_conserves_slots(make):
    """Every slot is held exactly once after the flow ends, eviction and slot
    reuse included (fork_tree's pool holds 60% of its distinct tokens)."""
    wl = make()
    trace, cache = run_bookkeeping(wl.oracle_waves(), wl.num_slots, wl.decode_steps)
    _assert_slots_conserved(cache)
    assert trace.stats["protected"] == 0


# ------------------------------------------------------------------- pages
def _toy_run(page_size):
    reqs, _, _ = _toy_fixture()
    vocab = {}
    cache = RadixCache(4096, page_size)
    got = []
    for words in reqs:
        toks = [vocab.setdefault(w, len(vocab)) for w in words]
        slots, node = cache.match_prefix(toks)
        new = cache.alloc(len(toks) - len(slots))
        cache.insert(toks, slots + new)
        got.append(len(slots))
    return reqs, got


@pytest.mark.parametrize("page_size", [2, 4, 8, 16])
def test_toy_trie_reuse_counts_with_pages(page_size):
    """The toy's requests with page-aligned keys: reuse per request as derived
    by hand (fixture), and as brute force over the request strings."""
    want = {}
    for ln in read_golden("toy_trie_reuse_pages.txt"):
        ps, rest = ln.split(":")
        *counts, total = rest.split()
        want[int(ps)] = ([int(c) for c in counts], total)
    reqs, got = _toy_run(page_size)
    counts, total = want[page_size]
    assert got == counts
    assert f"{sum(got)}/{sum(len(r) for r in reqs)}" == total
    # brute force: longest whole-page prefix shared with an earlier request's
    # whole pages
    al = lambda n: n - n % page_size
    brute = []
    for i, r in enumerate(reqs):
        best = 0
        for j in range(i):
            c = 0
            while c < min(len(r), len(reqs[j])) and r[c] == reqs[j][c]:
                c += 1
            best = max(best, min(c, al(len(reqs[j]))))
        brute.append(al(best))
    assert brute == counts


@pytest.mark.parametrize("page_size,want", [(4, 3060), (60, 3060), (16, 3136)])
def test_nested_example_with_pages(page_size, want):
    g = {ln.split()[2]: int(ln.split()[4]) for ln in read_golden("nested_prefill_counts.txt")
         if ln.startswith("case page")}
    assert g[str(page_size)] == want
    wl = workloads.nested_share()
    slots = (wl.num_slots // page_size + 40) * page_size
    trace, cache = run_bookkeeping(wl.oracle_waves(), slots, 0, page_size=page_size)
    assert trace.prefilled == want
    assert [[rid for rid, _, _ in b] for b in trace.batches] == [[0], [1, 2, 3, 4], [5, 6, 7]]
    _assert_slots_conserved(cache)


@pytest.mark.parametrize("locked,victim,held", [
    ("C", "A", 3500), ("AC", "B", 3800), ("ABC", None, None)])
def test_worked_eviction_example_with_pages(locked, victim, held):
    """Every size of the worked example is a multiple of 100: with pages of
    100 slots (one pad page) the same node goes and the same occupancy
    results."""
    g = _golden_kv("worked_eviction.txt")
    ps = 100
    cache = RadixCache(g["capacity"] + ps, ps)
    rng = random.Random(7)
    seq = lambda n: [rng.randrange(32000) for _ in range(n)]
    s = seq(g["S"])
    nodes = {}
    for b in "ABC":
        toks = s + seq(g[b])
        slots, _ = cache.match_prefix(toks)
        _, nodes[b] = cache.insert(toks, slots + cache.alloc(len(toks) - len(slots)))
    for b in locked:
        cache.inc_lock_ref(nodes[b])
    d = s + seq(g["D_new"])
    slots, dnode = cache.match_prefix(d[:-1])
    assert len(slots) == g["S"]
    cache.inc_lock_ref(dnode)
    if victim is None:
        with pytest.raises(NoSpace):
            cache.alloc(g["D_new"])
        assert cache.eviction_log == []
        return
    new = cache.alloc(g["D_new"])
    assert cache.eviction_log == [(nodes[victim].id, g[victim])]
    cache.insert(d, slots + new)
    assert cache.cached_size() == held


@pytest.mark.parametrize("page_size", [2, 3])
def test_match_against_page_prefix_dictionary(page_size):
    """Match length and slots equal a naive dictionary of the whole-page
    prefixes of every inserted sequence (tiny alphabets)."""
    rng = random.Random(13 + page_size)
    al = lambda n: n - n % page_size
    for trial in range(200):
        alpha = rng.randint(1, 3)
        cache = RadixCache(3000 * page_size, page_size)
        slot_at = {}             # whole-page prefix -> slots of its last page
        for _ in range(rng.randint(1, 8)):
            seq = [rng.randrange(alpha) for _ in range(rng.randint(1, 14))]
            n = 0
            while n + page_size <= len(seq) and tuple(seq[:n + page_size]) in slot_at:
                n += page_size
            want = []
            for p in range(page_size, n + 1, page_size):
                want += slot_at[tuple(seq[:p])]
            assert cache.match_length(seq) == n
            slots, node = cache.match_prefix(seq)
            assert slots == want
            new = cache.alloc(len(seq) - n)
            row = slots + new
            already, _ = cache.insert(seq, row)
            assert already == n
            for p in range(page_size, al(len(seq)) + 1, page_size):
                slot_at.setdefault(tuple(seq[:p]), row[p - page_size:p])
        assert cache.cached_size() == len(slot_at) * page_size


def test_page_allocator_reading():
    """Reading (pages silent on the order): a FIFO free list of pages 1 ..
    N/page_size - 1 (page 0 is the pad page); a request's slots fill its
    pages in order; freeing any slot of a page returns the whole page, once."""
    cache = RadixCache(24, 4)
    assert cache.alloc(5) == [4, 5, 6, 7, 8]
    assert cache.alloc(4) == [12, 13, 14, 15]
    cache.free([9, 8, 6])
    assert list(cache.free_pages) == [4, 5, 2, 1]
    assert cache.alloc(12) == [16, 17, 18, 19, 20, 21, 22, 23, 8, 9, 10, 11]
    with pytest.raises(NoSpace):
        cache.alloc(5)


def _assert_rows_page_consistent(rows, ps):
    """Positions [k ps, (k+1) ps) of a request lie in one page, in order."""
    for row in rows.values():
        for p, s in enumerate(row):
            assert s % ps == p % ps and s // ps == row[p - p % ps] // ps


@pytest.mark.parametrize("page_size", [4, 16])
@pytest.mark.parametrize("make", [
    lambda: workloads.agent_loop(calls=7, preamble=120, lo=5, hi=40, decode_steps=9),
    lambda: workloads.fork_tree(branching=3, depth=3, level_tokens=24, decode_steps=5),
    lambda: workloads.multi_turn_chat(sessions=4, turns=3, system=50, user=13, decode_steps=6,
                                      layers=1),
])
def test_request_flow_with_pages_conserves_pages(make, page_size):
    """With pages: every row keeps each page's positions together and in
    order at every decode step, and after the flow every page is held by
    exactly one tree position or the free list (fork_tree evicts)."""
    wl = make()
    seen = {}

    def on_decode(step, rows):
        seen[step] = True
        _assert_rows_page_consistent(rows, page_size)

    slots = -(-int(wl.num_slots * 1.3) // page_size) * page_size
    trace, cache = run_bookkeeping(wl.oracle_waves(), slots, wl.decode_steps,
                                   on_decode=on_decode, page_size=page_size)
    assert seen
    for b in trace.batches:
        for rid, m, row in b:
            assert m % page_size == 0
    _assert_slots_conserved(cache)
    assert trace.stats["protected"] == 0


@pytest.mark.parametrize("actions", [8, 32])
def test_agent_steps_through_decode_reuse_with_pages(actions):
    """The agent example through decode with pages of 8 slots: every length
    of the example is a multiple of 8, so step 5 again reuses 2,800 + D."""
    waves, g = _agent_steps_with_actions(actions)
    trace, cache = run_bookkeeping(waves, 16000, actions, page_size=8)
    rid, m, row = trace.batches[g["step"] - 1][0]
    assert len(row) == g["prompt_tokens"] and m == g["reused"] + actions
    _assert_slots_conserved(cache)


# -------------------------------------------------------------- scheduling
def _lpm_toy(policy):
    """The cache-aware scheduling toy served one request at a time through
    the oracle's scheduler and radix cache (the last token of each request is
    its own, so matching the prompt minus its last token matches what the toy
    matches)."""
    g = {}
    for ln in read_golden("lpm_toy.txt"):
        k, *v = ln.split()
        g[k] = v
    n = int(g["prompt_tokens"][0])
    X = [f"x{i}" for i in range(n)]
    Y = [f"y{i}" for i in range(n)]
    queue = [("X1", X + ["a"]), ("Y1", Y + ["b"]), ("X2", X + ["c"]),
             ("Y2", Y + ["d"]), ("X3", X + ["e"]), ("Y3", Y + ["f"])]
    vocab = {}
    pending = [(name, [vocab.setdefault(w, len(vocab)) for w in words]) for name, words in queue]
    cache = RadixCache(int(g["capacity"][0]) + 1)
    log, prefilled = [], 0
    while pending:
        k = oscheduler.order(cache, [t for _, t in pending], policy)[0]
        name, toks = pending.pop(k)
        slots, node = cache.match_prefix(toks[:-1])
        cache.inc_lock_ref(node)
        new = cache.alloc(len(toks) - len(slots))
        cache.insert(toks, slots + new)
        cache.dec_lock_ref(node)
        prefilled += len(toks) - len(slots)
        log.append(f"{name}:{len(slots)}")
    return log, prefilled, g


@pytest.mark.parametrize("policy", ["fcfs", "lpm"])
def test_lpm_toy_served_order_and_prefill(policy):
    """126 of 126 tokens prefilled in arrival order, 46 of 126 with the
    longest prefix first, in the printed served order."""
    log, prefilled, g = _lpm_toy(policy)
    assert log == g[policy]
    assert [prefilled, 126] == [int(x) for x in g[policy + "_prefilled"]]


def test_lpm_queue_limit_falls_back_to_fcfs():
    """More than 128 waiting requests: arrival order; 128: LPM."""
    cache = RadixCache(5000)
    base = list(range(1, 41))
    cache.insert(base, cache.alloc(40))
    prompts = [[1000 + i, 7] if i % 2 else base[:30] + [2000 + i, 7] for i in range(129)]
    assert oscheduler.order(cache, prompts, "lpm") == list(range(129))
    got = oscheduler.order(cache, prompts[:128], "lpm")
    assert got[:64] == list(range(0, 128, 2))     # 30 tokens matched, first


def test_in_batch_prefix_deprioritises_siblings():
    """A request with a thin tree match (<= 32) that shares >= 32 tokens with
    an earlier queued request goes to the back; 31 shared tokens do not
    count; a request matching more than 32 tokens of the tree is not checked
    against the queue."""
    cache = RadixCache(5000)
    S = list(range(100, 140))                     # 40 tokens, not in the tree
    T31 = S[:31] + [900, 901, 902]                # shares 31 with S
    cache.insert(list(range(500, 540)), cache.alloc(40))
    R = list(range(500, 533)) + [7, 8]            # 33 tokens in the tree
    prompts = [S + [1], S + [2], T31 + [3], S + [4], R, list(range(600, 640)) + [5]]
    # keys: S+[1]: 0 (queued); S+[2]: back; T31: 0 (queued); S+[4]: back;
    # R: -33; the last: 0 (queued)
    assert oscheduler.order(cache, prompts, "lpm") == [4, 0, 2, 5, 1, 3]
    # exactly 32 shared tokens deprioritise, 31 do not
    Z = list(range(700, 710))
    T32 = S[:32] + [903, 904]
    assert oscheduler.order(cache, [S + [1], T32 + [5], Z], "lpm") == [0, 2, 1]
    assert oscheduler.order(cache, [T32 + [5], S + [1], Z], "lpm") == [0, 2, 1]
    assert oscheduler.order(cache, [S + [1], S[:31] + [5], Z], "lpm") == [0, 1, 2]
    # a tree match of exactly 32 tokens is still checked against the queue,
    # one of 33 is not
    W = list(range(300, 360))
    cache.insert(W[:32] + [999], cache.alloc(33))
    assert oscheduler.order(cache, [W + [1], W + [2], Z], "lpm") == [0, 2, 1]
    cache.insert(W[:33] + [998], cache.alloc(34))
    assert oscheduler.order(cache, [W + [1], W + [2], Z], "lpm") == [0, 1, 2]


def _dfs_tree():
    cache = RadixCache(5000)
    P = list(range(10, 20))
    P1, P2 = list(range(20, 25)), list(range(30, 35))
    Q = list(range(40, 50))
    # two leaves below each of P1, P2 and Q make each a node of its own
    for seq in (P + P1 + [0], P + P1 + [1], P + P2 + [0], P + P2 + [1], Q + [0], Q + [1]):
        slots, _ = cache.match_prefix(seq)
        cache.insert(seq, slots + cache.alloc(len(seq) - len(slots)))
    return cache, P, P1, P2, Q


def test_dfs_weight_order_by_hand():
    """Weights: P1 2 (r1, r4), P2 1 (r3), P 1 + 3 = 4 (r5 hangs off P), Q 2
    (r0, r6), root 1 (r2).  Depth first, a node's own requests first, heavier
    children first: r2, then P's subtree (r5; P1: r1, r4; P2: r3), then Q
    (r0, r6)."""
    cache, P, P1, P2, Q = _dfs_tree()
    prompts = [Q + [99, 98], P + P1 + [5, 6], [77, 78], P + P2 + [7, 8], P + P1 + [9, 9],
               P + [50, 51, 52], Q + [66, 67]]
    assert oscheduler.order(cache, prompts, "dfs-weight") == [2, 5, 1, 4, 3, 0, 6]
    # equal weights: the subtree whose earliest waiting request came first
    prompts = [Q + [7, 2], P + P2 + [3, 4], P + P1 + [5, 6], Q + [8, 8]]
    # P (2: r1 via P2, r2 via P1) ties Q (2: r0, r3); Q's earliest is r0
    assert oscheduler.order(cache, prompts, "dfs-weight") == [0, 3, 1, 2]


@pytest.mark.parametrize("policy", ["lpm", "dfs-weight"])
def test_scheduled_flow_conserves_slots_and_serves_everyone(policy):
    """A shuffled fork tree under a small pool: every request is served once,
    every slot is held exactly once after the flow."""
    wl = workloads.fork_tree(branching=3, depth=3, level_tokens=12, decode_steps=3)
    rng = random.Random(3)
    waves = [rng.sample(w, len(w)) for w in wl.oracle_waves()]
    trace, cache = run_bookkeeping(waves, wl.num_slots, wl.decode_steps, policy=policy)
    served = [rid for b in trace.batches for rid, _, _ in b]
    assert sorted(served) == sorted(r[0] for w in waves for r in w)
    assert len(trace.eviction_log) > 0
    _assert_slots_conserved(cache)


# ------------------------------------------------------- draft-tree verify
def _draft_fixture():
    g = {}
    for ln in read_golden("draft_tree.txt"):
        k, *v = ln.split()
        g[k] = [int(x) for x in v]
    return g


def test_draft_positions_example():
    g = _draft_fixture()
    parents = [-1, 0, 0, 1]                      # depths 0, 1, 1, 2
    assert ospec.depths(parents) == g["depths"]
    assert ospec.positions(g["prompt_len"][0], parents) == g["positions"]


def test_tree_mask_by_hand_and_size_formula():
    """The example tree after 2 context tokens, by hand; the entry count of
    materialised masks equals the page's formula, and at the page's sizes
    the formula gives its 128 MiB."""
    m = ospec.tree_mask(2, [-1, 0, 0, 1])
    want = np.array([[1, 1, 1, 0, 0, 0],
                     [1, 1, 1, 1, 0, 0],
                     [1, 1, 1, 0, 1, 0],
                     [1, 1, 1, 1, 0, 1]], dtype=bool)
    assert np.array_equal(m, want)
    rng = random.Random(4)
    for trial in range(20):
        bs, nv = rng.randint(1, 5), rng.randint(1, 9)
        lens = [rng.randint(0, 30) for _ in range(bs)]
        parents = [[rng.randrange(-1, i) for i in range(nv)] for _ in range(bs)]
        total = sum(ospec.tree_mask(p, par).size for p, par in zip(lens, parents))
        assert total == sum(lens) * nv + nv * nv * bs
    g = _draft_fixture()
    bs, ctx, nv = g["mask_requests"][0], g["mask_context"][0], g["mask_verify"][0]
    entries = bs * ctx * nv + nv * nv * bs
    assert round(entries / 2 ** 20) == g["mask_mib"][0]


def _qkv(rng, n, p, hq=4, hkv=2, d=8):
    return (rng.standard_normal((n, hq, d)), rng.standard_normal((p, hkv, d)),
            rng.standard_normal((p, hkv, d)), rng.standard_normal((n, hkv, d)),
            rng.standard_normal((n, hkv, d)))


def test_chain_tree_equals_causal_extend():
    """A chain of drafts (each continues the one before) sees exactly what a
    causal extend of the same tokens after the prefix sees."""
    rng = np.random.default_rng(5)
    n, p = 7, 11
    q, kp, vp, kd, vd = _qkv(rng, n, p)
    o, lse = ospec.verify_attention(q, kp, vp, kd, vd, list(range(-1, n - 1)))
    eo, el = oatt.extend_attention(q, np.concatenate([kp, kd]), np.concatenate([vp, vd]), p)
    assert np.array_equal(o, eo) and np.array_equal(lse, el)


def test_depth_zero_drafts_are_independent_decodes():
    """Drafts that all continue the verified token see the prefix and
    themselves only: each equals a decode of that token alone."""
    rng = np.random.default_rng(6)
    n, p = 5, 9
    q, kp, vp, kd, vd = _qkv(rng, n, p)
    o, lse = ospec.verify_attention(q, kp, vp, kd, vd, [-1] * n)
    for i in range(n):
        do, dl = oatt.decode_attention(q[i], np.concatenate([kp, kd[i:i + 1]]),
                                       np.concatenate([vp, vd[i:i + 1]]))
        assert np.array_equal(o[i], do) and np.array_equal(lse[i], dl)


def test_branch_equals_its_own_chain():
    """Any draft's result equals the chain made of its root path alone."""
    rng = np.random.default_rng(7)
    parents = [-1, 0, 0, 1, 1, 2, 5, -1, 7]
    n, p = len(parents), 6
    q, kp, vp, kd, vd = _qkv(rng, n, p)
    o, _ = ospec.verify_attention(q, kp, vp, kd, vd, parents)
    for i in range(n):
        path = ospec.ancestors_and_self(parents, i)
        co, _ = oatt.extend_attention(q[path], np.concatenate([kp, kd[path]]),
                                      np.concatenate([vp, vd[path]]), p)
        assert np.allclose(o[i], co[-1], atol=1e-14)


def test_move_kv_reads_before_writes():
    rng = np.random.default_rng(8)
    pool = rng.standard_normal((2, 3, 12, 4))
    out = ospec.move_kv(pool, [3, 5, 9], [5, 3, 1])      # 3 <-> 5 swap, 1 -> 9
    assert np.array_equal(out[:, :, 3], pool[:, :, 5])
    assert np.array_equal(out[:, :, 5], pool[:, :, 3])
    assert np.array_equal(out[:, :, 9], pool[:, :, 1])
    keep = [s for s in range(12) if s not in (3, 5, 9)]
    assert np.array_equal(out[:, :, keep], pool[:, :, keep])


def test_chunked_extend_equals_unchunked():
    """An extend split into chunks (each chunk's queries after the prefix
    plus the earlier chunks) gives the unchunked rows exactly."""
    rng = np.random.default_rng(9)
    n, p = 37, 14
    q = rng.standard_normal((n - p, 4, 8))
    k = rng.standard_normal((n, 2, 8))
    v = rng.standard_normal((n, 2, 8))
    full_o, full_l = oatt.extend_attention(q, k, v, p)
    for chunk in (1, 5, 8, 23):
        for a in range(0, n - p, chunk):
            b = min(n - p, a + chunk)
            o, l = oatt.extend_attention(q[a:b], k[:p + b], v[:p + b], p + a)
            assert np.array_equal(o, full_o[a:b]) and np.array_equal(l, full_l[a:b])


# ---------------------------------------------------------- two-tier cache
def _tt_conservation(cache, private_pages=()):
    """Device-resident and host-resident nodes each hang from the root; every
    device page and every host page is held by one tree position, the free
    list or a pending backup, exactly once."""
    ps = cache.page_size
    dev, host = [], []
    for n in cache.nodes.values():
        if n is cache.root:
            continue
        assert cache.on_gpu(n) or cache.on_host(n), "node on neither tier"
        if cache.on_gpu(n):
            assert cache.on_gpu(n.parent), "device residency not top-connected"
            dev += [s // ps for s in n.value[::ps]]
        if cache.on_host(n):
            assert cache.on_host(n.parent), "host residency not top-connected"
            host += [s // ps for s in n.host_value[::ps]]
        if n.pending is not None:
            host += [s // ps for s in n.pending[1][::ps]]
    assert sorted(dev + list(cache.free_pages) + list(private_pages)) == \
        list(range(1, cache.num_slots // ps))
    assert sorted(host + list(cache.free_host_pages)) == list(range(1, cache.host_slots // ps))


def test_two_tier_without_backups_equals_single_tier():
    """While nothing is written through, the two-tier cache makes every
    decision of the single-tier cache (random operations)."""
    rng = random.Random(23)
    for trial in range(40):
        n_slots = rng.randint(16, 70)
        a, b = RadixCache(n_slots), TwoTierRadixCache(n_slots, 64)
        la, lb = [], []
        for step in range(100):
            seq = [rng.randrange(3) for _ in range(rng.randint(1, 12))]
            r = rng.random()
            if r < 0.55:
                sa, na = a.match_prefix(seq[:-1])
                sb, nb = b.match_prefix(seq[:-1])
                assert sa == sb and na.id == nb.id
                a.inc_lock_ref(na)
                b.inc_lock_ref(nb)
                try:
                    xa = a.alloc(len(seq) - len(sa))
                except NoSpace:
                    xa = None
                try:
                    xb = b.alloc(len(seq) - len(sb))
                except NoSpace:
                    xb = None
                assert xa == xb and a.eviction_log == b.eviction_log
                if xa is None:
                    a.dec_lock_ref(na)
                    b.dec_lock_ref(nb)
                    continue
                ka, ma = a.insert(seq, sa + xa)
                kb, mb = b.insert(seq, sb + xb)
                assert ka == kb and ma.id == mb.id
                a.free((sa + xa)[len(sa):ka])
                b.free((sb + xb)[len(sb):kb])
                a.inc_lock_ref(ma)
                b.inc_lock_ref(mb)
                a.dec_lock_ref(na)
                b.dec_lock_ref(nb)
                la.append(ma)
                lb.append(mb)
            elif r < 0.8 and la:
                i = rng.randrange(len(la))
                a.dec_lock_ref(la.pop(i))
                b.dec_lock_ref(lb.pop(i))
            else:
                k = rng.randint(1, 9)
                assert a.evict(k) == b.evict(k)
            assert (a.evictable_size_, a.protected_size_) == (b.evictable_size_, b.protected_size_)
            assert list(a.free_pages) == list(b.free_pages)


def test_worked_example_with_a_host_tier():
    """"Worked example, step by step": C locked, D arrives, A (used longest
    ago) leaves the device.  With every branch written through to a host
    tier, A stays on the host; when user A returns, A's 900 tokens come back
    from the host (900 host-matched tokens, one load) instead of being
    prefilled, and the unlocked B leaves the device to make room."""
    g = _golden_kv("worked_eviction.txt")
    cache = TwoTierRadixCache(g["capacity"] + 1, 8192)
    rng = random.Random(7)
    seq = lambda n: [rng.randrange(32000) for _ in range(n)]
    s = seq(g["S"])
    branch = {b: seq(g[b]) for b in "ABC"}
    nodes = {}
    for b in "ABC":
        toks = s + branch[b]
        slots, _ = cache.match_prefix(toks)
        _, nodes[b] = cache.insert(toks, slots + cache.alloc(len(toks) - len(slots)))
        t, dev, host = cache.write_through(nodes[b])
        cache.commit_write_through(t, True)
    assert cache.host_cached_size() == g["S"] + g["A"] + g["B"] + g["C"]
    cache.inc_lock_ref(nodes["C"])
    d = s + seq(g["D_new"])
    slots, dnode = cache.match_prefix(d[:-1])
    cache.inc_lock_ref(dnode)
    new = cache.alloc(g["D_new"])
    _, dn = cache.insert(d, slots + new)
    cache.inc_lock_ref(dn)
    cache.dec_lock_ref(dnode)
    assert cache.eviction_log == [(nodes["A"].id, g["A"])]
    assert cache.device_cached_size() == 3500 and not cache.on_gpu(nodes["A"])
    assert cache.on_host(nodes["A"])
    # user A comes back with 100 new tokens
    a2 = s + branch["A"] + seq(100)
    slots, dev_node, host_len, host_node = cache.match_prefix_tiers(a2[:-1])
    assert len(slots) == g["S"] and host_len == g["A"] and host_node is nodes["A"]
    host_slots, dev_slots = cache.load_onboard(host_node)
    assert host_slots == nodes["A"].host_value and len(dev_slots) == g["A"]
    assert cache.eviction_log[-1] == (nodes["B"].id, g["B"])
    slots, node = cache.match_prefix(a2[:-1])
    assert len(slots) == g["S"] + g["A"]          # only 100 - 1 + 1 tokens left to prefill
    _tt_conservation(cache)


def test_two_tier_random_operations_keep_invariants():
    """Random matches, loads, inserts, write-throughs (committed with success
    or failure, or left pending across other operations), locks and
    evictions on a small device pool and a small host pool: residency stays
    top-connected on each tier, pages are conserved on each tier, locked
    nodes never leave the device."""
    rng = random.Random(29)
    for trial in range(60):
        ps = rng.choice([1, 2])
        cache = TwoTierRadixCache(ps * rng.randint(12, 30), ps * rng.randint(6, 24), ps)
        locks, pending, private = [], [], []
        for step in range(120):
            seq = [rng.randrange(3) for _ in range(rng.randint(1, 10))]
            r = rng.random()
            if r < 0.45:
                _, _, host_len, host_node = cache.match_prefix_tiers(seq[:-1])
                if host_len:
                    try:
                        cache.load_onboard(host_node)
                    except NoSpace:
                        pass
                slots, node = cache.match_prefix(seq[:-1])
                cache.inc_lock_ref(node)
                before = {n.id for n in cache.nodes.values() if n.lock_ref > 0}
                try:
                    new = cache.alloc(len(seq) - len(slots))
                except NoSpace:
                    cache.dec_lock_ref(node)
                    continue
                for nid, _ in cache.eviction_log[-10:]:
                    if nid in before and nid in cache.nodes:
                        assert cache.on_gpu(cache.nodes[nid]) or cache.nodes[nid].lock_ref == 0
                already, node2 = cache.insert(seq, slots + new)
                cache.free((slots + new)[len(slots):already] +
                           (slots + new)[cache.aligned(len(seq)):])
                cache.inc_lock_ref(node2)
                cache.dec_lock_ref(node)
                locks.append(node2)
            elif r < 0.6 and locks:
                node = locks.pop(rng.randrange(len(locks)))
                cache.dec_lock_ref(node)
                try:
                    t, _, _ = cache.write_through(node)
                except NoSpace:
                    t = 0
                if t:
                    pending.append(t)
            elif r < 0.75 and pending:
                cache.commit_write_through(pending.pop(rng.randrange(len(pending))),
                                           rng.random() < 0.8)
            else:
                cache.evict(rng.randint(1, 8))
            for n in locks:
                walk = n
                while walk is not cache.root:
                    assert cache.on_gpu(walk), "a locked node left the device"
                    walk = walk.parent
            _tt_conservation(cache)


def _round_robin_chat():
    wl = workloads.multi_turn_chat(sessions=6, turns=4, system=64, user=24, decode_steps=8,
                                   layers=1)
    # one request per wave, sessions taking turns: a session's history has
    # to survive five other sessions' turns to be reused
    return [[r] for w in wl.oracle_waves() for r in w]


def test_host_tier_saves_prefill_under_a_small_device_pool():
    """A multi-turn chat whose device pool holds about two sessions'
    histories: without a host tier most returning sessions find their
    history evicted and prefill it again; with one, it comes back from the
    host.  Every page is conserved on both tiers at the end."""
    waves = _round_robin_chat()
    single, _ = run_bookkeeping(waves, 400, 8)
    tiered, cache = run_bookkeeping(waves, 400, 8, host_slots=4096)
    assert tiered.prefilled < single.prefilled
    assert len(tiered.loads) > 0 and len(tiered.backups) == len(waves)
    loaded = sum(len(h) for _, h, _ in tiered.loads)
    assert tiered.prefilled + loaded <= single.prefilled
    _tt_conservation(cache)
    # a small host tier evicts host-only leaves and still conserves pages
    small, cache = run_bookkeeping(waves, 400, 8, host_slots=700)
    assert len(small.host_eviction_log) > 0
    assert small.prefilled <= single.prefilled
    _tt_conservation(cache)


def test_write_through_commit_outcomes():
    """A committed backup makes the path resident on both tiers; a failed one
    leaves it on the device only and returns every host page; a second
    backup of an already backed-up path copies nothing; a backup below one
    still in flight is refused until that one commits."""
    cache = TwoTierRadixCache(200, 100)
    a = list(range(1, 21))
    _, na = cache.insert(a, cache.alloc(20))
    free0 = len(cache.free_host_pages)
    t, dev, host = cache.write_through(na)
    assert t and len(dev) == len(host) == 20 and len(cache.free_host_pages) == free0 - 20
    b = a[:10] + list(range(50, 60))
    slots, _ = cache.match_prefix(b)
    _, nb = cache.insert(b, slots + cache.alloc(10))      # splits a's node while in flight
    assert cache.write_through(nb) == (0, [], [])           # refused: an ancestor is in flight
    cache.commit_write_through(t, False)
    assert not cache.on_host(na) and not cache.on_host(na.parent)
    assert len(cache.free_host_pages) == free0 and cache.host_cached_size() == 0
    t, dev, host = cache.write_through(nb)
    assert len(dev) == 20                                   # the shared 10 and b's own 10
    cache.commit_write_through(t, True)
    assert cache.on_host(nb) and cache.on_host(nb.parent) and not cache.on_host(na)
    assert cache.host_cached_size() == 20
    assert cache.write_through(nb) == (0, [], [])           # nothing left to copy
    t, dev, host = cache.write_through(na)
    assert len(dev) == 10                                   # only a's own 10
    cache.commit_write_through(t, True)
    _tt_conservation(cache)
