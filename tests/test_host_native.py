"""librx host side on CPU: exported symbols, argument checks, and bit-exact
agreement of the native radix cache with the oracle (slot tables, match
lengths, prefilled counts, eviction order)."""

import os
import random
import re

import numpy as np
import pytest

from conftest import ROOT, read_golden

rx = pytest.importorskip("radix_tree_prefix_gb300.rx",
                         reason="librx.so not built (run __graft_entry__.build())")
from oracle.harness import run_bookkeeping  # noqa: E402
from oracle.radix_cache import NoSpace as ONoSpace  # noqa: E402
from oracle.radix_cache import RadixCache as ORadix  # noqa: E402
from radix_tree_prefix_gb300 import workloads  # noqa: E402
from radix_tree_prefix_gb300.engine import Engine  # noqa: E402


def header_functions():
    with open(os.path.join(ROOT, "include", "rx.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rx_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported():
    names = header_functions()
    assert len(names) >= 20
    for n in names:
        assert hasattr(rx._lib, n), f"{n} declared in rx.h but not exported"
    assert set(names) <= set(rx.EXPORTED), "binding lacks a declared entry point"


def test_argument_errors_need_no_gpu():
    c = rx.RadixCache(16)
    _, node = c.insert([1, 2], c.alloc(2))
    with pytest.raises(rx.StateError):
        c.unlock(node)
    with pytest.raises(rx.RxError) as e:
        c.lock(12345)
    assert e.value.status == rx.RX_ERR_INVALID
    with pytest.raises(rx.NoSpace):
        c.alloc(100)
    # device entry points validate before touching CUDA
    bad = rx.rx_pool_desc(16, 16, 8, 1, 1, 64, 0)     # head_dim 64 unsupported
    import ctypes as C
    st = rx._lib.rx_kv_store(C.byref(bad), 0, None, None, None, 1, None)
    assert st == rx.RX_ERR_INVALID and "head_dim" in rx.last_error()
    bad = rx.rx_pool_desc(16, 16, 8, 1, 2, 128, 0)
    st = rx._lib.rx_extend_attention(C.byref(bad), 3, None, 4, None, 0, None, None, None,
                                     None, 1, 1, 1.0, None, None, None)
    assert st == rx.RX_ERR_INVALID and "layer" in rx.last_error()
    # pool rows (layers x KV heads x slots) must stay below 2^31, the range
    # of the kernels' TMA row coordinates
    big = rx.rx_pool_desc(16, 16, 2 ** 28, 4, 2, 128, 0)     # 2^31 rows
    st = rx._lib.rx_extend_attention(C.byref(big), 0, None, 4, None, 0, None, None, None,
                                     None, 0, 0, 1.0, None, None, None)
    assert st == rx.RX_ERR_INVALID and "2^31" in rx.last_error()
    st = rx._lib.rx_kv_store(C.byref(big), 0, None, None, None, 0, None)
    assert st == rx.RX_ERR_INVALID
    under = rx.rx_pool_desc(16, 16, 2 ** 28 - 1, 4, 2, 128, 0)
    assert rx._lib.rx_extend_attention(C.byref(under), 0, None, 4, None, 0, None, None, None,
                                       None, 0, 0, 1.0, None, None, None) == rx.RX_OK
    h = C.c_void_p()
    for slots, ps in ((9, 2), (8, 0), (3, 4)):    # page size must divide the slot count
        cfg = rx.rx_config(slots, ps, 0)
        assert rx._lib.rx_cache_create(C.byref(cfg), C.byref(h)) == rx.RX_ERR_INVALID


def test_worked_eviction_example_native():
    """The worked example's victims and occupancy on the native cache."""
    g = {}
    for ln in read_golden("worked_eviction.txt"):
        p = ln.split()
        if p[0] != "case":
            g[p[0]] = int(p[1])
    for locked, victim, held in (("C", "A", 3500), ("AC", "B", 3800), ("ABC", None, None)):
        c = rx.RadixCache(g["capacity"] + 1)
        rng = random.Random(7)
        seq = lambda n: [rng.randrange(32000) for _ in range(n)]
        s = seq(g["S"])
        nodes = {}
        for b in "ABC":
            toks = s + seq(g[b])
            slots, _ = c.match_prefix(toks)
            new = c.alloc(len(toks) - len(slots))
            _, nodes[b] = c.insert(toks, np.concatenate([slots, new]))
        for b in locked:
            c.lock(nodes[b])
        d = s + seq(g["D_new"])
        slots, dn = c.match_prefix(d[:-1])
        c.lock(dn)
        if victim is None:
            with pytest.raises(rx.NoSpace):
                c.alloc(g["D_new"])
            assert c.eviction_log() == []
            continue
        new = c.alloc(g["D_new"])
        assert c.eviction_log() == [(nodes[victim], g[victim])]
        c.insert(d, np.concatenate([slots, new]))
        assert c.stats()["cached_tokens"] == held


def test_random_ops_match_oracle():
    """Same random operation sequence on both caches: identical results."""
    rng = random.Random(21)
    for trial in range(60):
        n_slots = rng.randint(16, 80)
        o, n = ORadix(n_slots), rx.RadixCache(n_slots)
        onodes, nnodes = [], []
        for step in range(120):
            r = rng.random()
            seq = [rng.randrange(rng.choice([2, 3, 5])) for _ in range(rng.randint(1, 14))]
            if r < 0.2:
                assert o.match_length(seq) == n.match_length(seq)
                os_, on = o.match_prefix(seq)
                ns_, nn = n.match_prefix(seq)
                assert list(os_) == ns_.tolist() and on.id == nn
            elif r < 0.55:
                os_, on = o.match_prefix(seq[:-1])
                ns_, nn = n.match_prefix(seq[:-1])
                assert on.id == nn
                k = len(seq) - len(os_)
                try:
                    onew = o.alloc(k)
                except ONoSpace:
                    onew = None
                try:
                    nnew = n.alloc(k).tolist()
                except rx.NoSpace:
                    nnew = None
                assert onew == nnew
                if onew is None:
                    continue
                oa, on2 = o.insert(seq, list(os_) + onew)
                na, nn2 = n.insert(seq, ns_.tolist() + nnew)
                assert (oa, on2.id) == (na, nn2)
                o.free((list(os_) + onew)[len(os_):oa])
                n.free((ns_.tolist() + nnew)[len(ns_):na])
                o.inc_lock_ref(on2)
                n.lock(nn2)
                onodes.append(on2)
                nnodes.append(nn2)
            elif r < 0.8 and onodes:
                i = rng.randrange(len(onodes))
                o.dec_lock_ref(onodes.pop(i))
                n.unlock(nnodes.pop(i))
            else:
                k = rng.randint(1, 10)
                assert o.evict(k) == n.evict(k)
            st = n.stats()
            assert st["cached_tokens"] == o.cached_size()
            assert st["evictable_tokens"] == o.evictable_size_
            assert st["protected_tokens"] == o.protected_size_
            assert st["free_slots"] == len(o.free_slots)
            assert st["num_nodes"] == o.num_nodes()
            assert n.eviction_log() == o.eviction_log


SCALED = {
    "nested_share": lambda: workloads.nested_share(),
    "agent_loop": lambda: workloads.agent_loop(),
    "fork_tree_small": lambda: workloads.fork_tree(branching=4, depth=3, level_tokens=40,
                                                   decode_steps=5),
    "multi_turn_small": lambda: workloads.multi_turn_chat(sessions=12, turns=4, system=300,
                                                         user=30, decode_steps=6, layers=1),
    "long_shared_small": lambda: workloads.long_shared(batch=8, prefix=2048, unique=128,
                                                       decode_steps=8),
}


@pytest.mark.parametrize("name", sorted(SCALED))
def test_request_flow_matches_oracle(name):
    wl = SCALED[name]()
    got = Engine(wl).run()
    want, _ = run_bookkeeping(wl.oracle_waves(), wl.num_slots, wl.decode_steps,
                                   page_size=wl.page_size)
    assert got.prefilled == want.prefilled
    assert got.as_tuple() == want.as_tuple()
    assert got.stats == want.stats
    if name == "nested_share":
        assert got.prefilled == 3060
    if name.startswith("fork_tree"):
        assert len(got.eviction_log) > 0


def test_fork_tree_full_size_bookkeeping():
    """Workload 4 at full size: eviction order and slot tables bit-exact."""
    wl = workloads.fork_tree()
    got = Engine(wl).run()
    want, _ = run_bookkeeping(wl.oracle_waves(), wl.num_slots, wl.decode_steps,
                                   page_size=wl.page_size)
    assert got.as_tuple() == want.as_tuple()
    assert len(got.eviction_log) > 100


def test_decode_plan_covers_every_context_once():
    """Shared segments are read once; each request's keys are covered once."""
    wl = workloads.fork_tree(branching=3, depth=3, level_tokens=10, decode_steps=0)
    c = rx.RadixCache(wl.num_slots + 1000)
    wave = wl.waves[0]
    nodes, lens = [], []
    for r in wave:
        toks = wl.prompt_tokens(r)
        slots, _ = c.match_prefix(toks)
        new = c.alloc(len(toks) - len(slots))
        _, node = c.insert(toks, np.concatenate([slots, new]))
        c.lock(node)
        nodes.append(node)
        lens.append(len(toks) + 2)             # two decode tokens beyond the tree
    hq, hkv, d = 32, 8, 128
    G = hq // hkv
    plan, info = c.plan_decode(nodes, lens, list(range(len(wave))), hq, hkv, d)
    W = rx.RX_WORK_WORDS
    work = plan[info.off_work:info.off_work + info.n_work * W].reshape(-1, W)
    members = plan[info.off_members:info.off_members + info.n_member_entries]
    covered = {b: [] for b in range(len(wave))}
    for row, kb, ke, moff, nm, pbase, nrows, _ in work:
        assert nrows == nm * G and nm * G <= 128
        for i in range(nm):
            b = int(members[moff + i])
            covered[b].append((int(kb), int(ke)))
            if nm > 1 or ke <= 30:   # shared chunks read a member's own row range
                assert kb < ke
    for b, rngs in covered.items():
        rngs.sort()
        pos = 0
        for kb, ke in rngs:
            assert kb == pos
            pos = ke
        assert pos == lens[b]
    # level-1 node (10 tokens) is shared by all 9 leaves, level-2 by 3 each
    assert info.n_shared_segments == 1 + 3
    assert info.distinct_kv_tokens == 10 + 3 * 10 + 9 * 10 + 9 * 2
    indptr = plan[info.off_req_part_indptr:info.off_req_part_indptr + len(wave) + 1]
    assert indptr[-1] == info.n_parts


def test_identical_prompts_share_slots():
    """Several samples from one prompt: later copies adopt the tree's slots."""
    base = workloads.nested_share()
    seg = base.seg_tokens
    waves = [[workloads.Request(0, (0, 1, 3)), workloads.Request(1, (0, 1, 3)),
              workloads.Request(2, (0, 1, 3)), workloads.Request(3, (0, 2, 4))]]
    wl = workloads.Workload("dup", 1, 8, 2, 128, 5000, 0, seg, waves)
    got = Engine(wl).run()
    want, _ = run_bookkeeping(wl.oracle_waves(), wl.num_slots, 0, page_size=wl.page_size)
    assert got.as_tuple() == want.as_tuple()
    assert [[r for r, _, _ in b] for b in got.batches] == [[0], [1], [2, 3]]
    assert got.stats == want.stats


def test_multi_step_plan_covers_each_step_once():
    """A plan for T steps, clamped at step t, covers every context once."""
    wl = workloads.agent_loop(calls=7, preamble=300, lo=50, hi=400, decode_steps=0)
    c = rx.RadixCache(wl.num_slots + 1000)
    nodes, ctx0 = [], []
    for r in wl.waves[0]:
        toks = wl.prompt_tokens(r)
        slots, _ = c.match_prefix(toks)
        new = c.alloc(len(toks) - len(slots))
        _, node = c.insert(toks, np.concatenate([slots, new]))
        c.lock(node)
        nodes.append(node)
        ctx0.append(len(toks) + 1)
    T = 200
    plan, info = c.plan_decode(nodes, ctx0, list(range(len(nodes))), 32, 8, 128, n_steps=T)
    W = rx.RX_WORK_WORDS
    work = plan[info.off_work:info.off_work + info.n_work * W].reshape(-1, W)
    members = plan[info.off_members:info.off_members + info.n_member_entries]
    for t in (0, 1, 77, T - 1):
        covered = {b: [] for b in range(len(nodes))}
        for row, kb, ke, moff, nm, pbase, nrows, grow in work:
            end = min(ke, grow + t) if grow > 0 else ke
            if end <= kb:
                continue
            for i in range(nm):
                covered[int(members[moff + i])].append((int(kb), int(end)))
        for b, rngs in covered.items():
            rngs.sort()
            pos = 0
            for kb, ke in rngs:
                assert kb == pos
                pos = ke
            assert pos == ctx0[b] + t
    # the newest token of every step lies in exactly one growing private chunk
    assert info.tails_private == 1
    for t in (0, 1, T - 1):
        owners = {b: 0 for b in range(len(nodes))}
        for row, kb, ke, moff, nm, pbase, nrows, grow in work:
            if grow > 0 and kb < grow + t <= ke:
                assert nm == 1
                owners[int(members[moff])] += 1
        assert all(v == 1 for v in owners.values())


def test_tails_private_flag():
    """The in-kernel store of the newest token needs every request's newest
    token in a private tail of the warp role; the plan says when it is."""
    c = rx.RadixCache(4096)
    toks = np.arange(1, 200, dtype=np.int32)
    slots = c.alloc(len(toks))
    _, node = c.insert(toks, slots)
    c.lock(node)
    other = np.concatenate([toks[:100], np.arange(500, 560, dtype=np.int32)])
    s2 = c.alloc(60)
    _, node2 = c.insert(other, np.concatenate([slots[:100], s2]))
    c.lock(node2)
    # contexts past the cached prompts: private tails hold the newest tokens
    _, info = c.plan_decode([node, node2], [200, 161], [0, 1], 32, 8, 128, n_steps=4)
    assert info.tails_private == 1
    # head_dim 256 takes the same warp role
    _, info = c.plan_decode([node, node2], [200, 161], [0, 1], 32, 8, 256, n_steps=4)
    assert info.tails_private == 1
    # a group above 16 rows: the store stays a launch of its own
    _, info = c.plan_decode([node, node2], [200, 161], [0, 1], 32, 1, 128)
    assert info.tails_private == 0
    # a context that ends inside the shared segment (the caller passed the
    # node of a token that is itself shared): no private tail at step 0
    mid = c.match_prefix(toks[:100])[1]
    c.lock(mid)
    _, info = c.plan_decode([mid, node, node2], [100, 200, 161], [0, 1, 2], 32, 8, 128,
                            n_steps=2)
    assert info.tails_private == 0


def test_batch_end_follows_the_in_batch_rule():
    """rx_batch_end equals the request-by-request rule: m_j from the tree,
    conflict when a member shares more than m_j tokens (exactly m_j does not)."""
    rng = np.random.default_rng(5)
    c = rx.RadixCache(100000)
    base = rng.integers(1, 50, size=300).astype(np.int32)
    slots = c.alloc(200)
    c.insert(base[:200], slots)
    prompts = []
    for i in range(30):
        cut = int(rng.choice([0, 50, 199, 200, 201, 250, 300]))
        tail = rng.integers(1, 50, size=int(rng.integers(1, 40))).astype(np.int32)
        prompts.append(np.concatenate([base[:cut], tail]))
    prompts.append(prompts[3].copy())   # an identical prompt
    prompts.append(prompts[5][:1].copy())   # a one-token prompt
    tokens = np.concatenate(prompts).astype(np.int32)
    indptr = np.zeros(len(prompts) + 1, dtype=np.int64)
    np.cumsum([len(p) for p in prompts], out=indptr[1:])
    for start in range(len(prompts)):
        want = len(prompts)
        for j in range(start + 1, len(prompts)):
            m = c.match_length(prompts[j][:-1])
            if rx.batch_conflict(prompts[j], m, tokens[indptr[start]:indptr[j]],
                                 indptr[start:j + 1] - indptr[start]):
                want = j
                break
            # the rule itself, brute force
            assert all(oracle_common(prompts[j], prompts[r]) <= m for r in range(start, j))
        assert c.batch_end(tokens, indptr, start) == want


def oracle_common(a, b):
    n = min(len(a), len(b))
    k = 0
    while k < n and a[k] == b[k]:
        k += 1
    return k


def test_pointer_forms_match_array_forms():
    """The pointer forms of the batch steps, given a batch's slice of the
    wave's offsets (offsets relative to the wave's tokens) and reused output
    buffers, give the array forms' results: same batch ends, prefixes, new
    slots, slot-table rows and prompt nodes, on twin caches."""
    rng = np.random.default_rng(11)
    base = rng.integers(1, 40, size=120).astype(np.int32)
    prompts = []
    for i in range(14):
        cut = int(rng.choice([0, 30, 119, 120]))
        tail = rng.integers(1, 40, size=int(rng.integers(1, 30))).astype(np.int32)
        prompts.append(np.concatenate([base[:cut], tail]))
    prompts.append(prompts[2].copy())
    tokens = np.concatenate(prompts).astype(np.int32)
    indptr = np.zeros(len(prompts) + 1, dtype=np.int64)
    np.cumsum([len(p) for p in prompts], out=indptr[1:])
    W, S = len(prompts), 200
    ca, cp = rx.RadixCache(5000), rx.RadixCache(5000)
    ta, tp = np.zeros((W, S), np.int32), np.zeros((W, S), np.int32)
    na, npn = np.zeros(W, np.int64), np.zeros(W, np.int64)
    b_prefix, b_nodes = np.zeros(W, np.int32), np.zeros(W, np.int64)
    b_new = np.zeros(len(tokens), np.int32)
    start = 0
    while start < W:
        end = ca.batch_end(tokens, indptr, start)
        assert cp.batch_end_p(tokens.ctypes.data, indptr.ctypes.data, start, W) == end
        R = end - start
        tok = tokens[indptr[start]:indptr[end]]
        ind = indptr[start:end + 1] - indptr[start]
        prefix, mnodes, new = ca.extend_begin(tok, ind, ta[start:end])
        ind_p = indptr.ctypes.data + 8 * start
        row_p = tp.ctypes.data + 4 * S * start
        total = cp.extend_begin_p(R, tokens.ctypes.data, ind_p, row_p, S, b_prefix.ctypes.data,
                                  b_nodes.ctypes.data, b_new.ctypes.data)
        assert total == len(new)
        assert np.array_equal(b_prefix[:R], prefix) and np.array_equal(b_new[:total], new)
        assert np.array_equal(tp[start:end], ta[start:end])
        nodes, rew = ca.extend_end(tok, ind, ta[start:end], prefix, mnodes)
        rew_p = cp.extend_end_p(R, tokens.ctypes.data, ind_p, row_p, S, b_prefix.ctypes.data,
                                b_nodes.ctypes.data, npn.ctypes.data + 8 * start)
        na[start:end] = nodes
        assert rew_p == rew
        assert np.array_equal(tp[start:end], ta[start:end])
        start = end
    assert np.array_equal(npn, na)
    assert ca.stats() == cp.stats()


# ------------------------------------------------------------------- pages
@pytest.mark.parametrize("page_size", [1, 4, 16])
def test_random_ops_match_oracle_with_pages(page_size):
    """The random operation sequence of the token-level test, on caches cut
    into pages: identical slots, nodes, eviction order and counts."""
    rng = random.Random(31 + page_size)
    for trial in range(40):
        n_slots = rng.randint(6, 20) * page_size
        o, n = ORadix(n_slots, page_size), rx.RadixCache(n_slots, page_size)
        onodes, nnodes = [], []
        for step in range(100):
            r = rng.random()
            seq = [rng.randrange(rng.choice([2, 3])) for _ in range(rng.randint(1, 5 * page_size))]
            if r < 0.2:
                assert o.match_length(seq) == n.match_length(seq)
                os_, on = o.match_prefix(seq)
                ns_, nn = n.match_prefix(seq)
                assert list(os_) == ns_.tolist() and on.id == nn
            elif r < 0.55:
                os_, on = o.match_prefix(seq[:-1])
                ns_, nn = n.match_prefix(seq[:-1])
                assert on.id == nn
                k = len(seq) - len(os_)
                try:
                    onew = o.alloc(k)
                except ONoSpace:
                    onew = None
                try:
                    nnew = n.alloc(k).tolist()
                except rx.NoSpace:
                    nnew = None
                assert onew == nnew
                if onew is None:
                    continue
                oa, on2 = o.insert(seq, list(os_) + onew)
                na, nn2 = n.insert(seq, ns_.tolist() + nnew)
                assert (oa, on2.id) == (na, nn2)
                orow = list(os_) + onew
                o.free(orow[len(os_):oa] + orow[o.aligned(len(seq)):])
                n.free(np.array(orow[len(os_):oa] + orow[o.aligned(len(seq)):], dtype=np.int32))
                o.inc_lock_ref(on2)
                n.lock(nn2)
                onodes.append(on2)
                nnodes.append(nn2)
            elif r < 0.8 and onodes:
                i = rng.randrange(len(onodes))
                o.dec_lock_ref(onodes.pop(i))
                n.unlock(nnodes.pop(i))
            else:
                k = rng.randint(1, 3 * page_size)
                assert o.evict(k) == n.evict(k)
            st = n.stats()
            assert st["cached_tokens"] == o.cached_size()
            assert st["evictable_tokens"] == o.evictable_size_
            assert st["protected_tokens"] == o.protected_size_
            assert st["free_slots"] == len(o.free_slots)
            assert st["num_nodes"] == o.num_nodes()
            assert n.eviction_log() == o.eviction_log


PAGED = {
    "nested_share": lambda: workloads.nested_share(),
    "agent_small": lambda: workloads.agent_loop(calls=9, preamble=130, lo=3, hi=50,
                                                decode_steps=21),
    "fork_tree_small": lambda: workloads.fork_tree(branching=4, depth=3, level_tokens=40,
                                                   decode_steps=5),
    "multi_turn_small": lambda: workloads.multi_turn_chat(sessions=12, turns=4, system=300,
                                                         user=30, decode_steps=6, layers=1),
    "long_shared_small": lambda: workloads.long_shared(batch=8, prefix=2048, unique=128,
                                                       decode_steps=8),
}


@pytest.mark.parametrize("page_size", [4, 16])
@pytest.mark.parametrize("name", sorted(PAGED))
def test_request_flow_with_pages_matches_oracle(name, page_size):
    """The whole request flow on a paged pool: slot tables, prefixes,
    decode slots, finishes and eviction order equal the oracle's."""
    wl = workloads.with_pages(PAGED[name](), page_size)
    got = Engine(wl).run()
    want, _ = run_bookkeeping(wl.oracle_waves(), wl.num_slots, wl.decode_steps,
                              page_size=page_size)
    assert got.as_tuple() == want.as_tuple()
    assert got.stats == want.stats
    if name.startswith("fork_tree"):
        assert len(got.eviction_log) > 0


def test_alloc_decode_steps_follows_pages():
    """A decode token that starts a page takes a new page (one allocation per
    step, in request order), any other the next slot of the request's page."""
    c = rx.RadixCache(64, 4)
    first = c.alloc(7)                    # pages 1, 2: slots 4 .. 10
    assert first.tolist() == [4, 5, 6, 7, 8, 9, 10]
    out = c.alloc_decode_steps([7, 8], [10, 99], 3)
    # step 0: request 1 (position 8) starts a page -> page 3 (slots 12..15);
    # request 0 (position 7) takes slot 11.  Step 1: request 0 (position 8)
    # starts a page -> page 4 (16..19); request 1 takes 13.  Step 2: 17, 14.
    assert out[:, 0].tolist() == [11, 16, 17]
    assert out[:, 1].tolist() == [12, 13, 14]


# -------------------------------------------------------------- scheduling
def test_schedule_matches_oracle_on_random_queues():
    """rx_schedule equals the oracle's order for every policy on random
    queues over random trees (tiny alphabets, page sizes 1 and 4)."""
    from oracle import scheduler as osched
    rng = random.Random(41)
    for trial in range(150):
        ps = rng.choice([1, 1, 4])
        o, n = ORadix(4000, ps), rx.RadixCache(4000, ps)
        base = [rng.randrange(3) for _ in range(60)]
        for _ in range(rng.randint(0, 6)):
            cut = rng.randint(0, 60)
            seq = base[:cut] + [rng.randrange(3) for _ in range(rng.randint(1, 40))]
            os_, _ = o.match_prefix(seq)
            ns_, _ = n.match_prefix(seq)
            onew = o.alloc(len(seq) - len(os_))
            nnew = n.alloc(len(seq) - len(ns_))
            o.insert(seq, list(os_) + onew)
            n.insert(seq, np.concatenate([ns_, nnew]))
        R = rng.choice([1, 3, 9, 40, 129, 140])
        prompts = []
        for _ in range(R):
            cut = rng.choice([0, 10, 33, 40, 60])
            prompts.append(base[:cut] + [rng.randrange(3) for _ in range(rng.randint(1, 45))])
        tok = np.concatenate([np.array(p, dtype=np.int32) for p in prompts])
        ind = np.zeros(R + 1, dtype=np.int64)
        np.cumsum([len(p) for p in prompts], out=ind[1:])
        for pol in ("fcfs", "lpm", "dfs-weight"):
            assert n.schedule(pol, tok, ind).tolist() == osched.order(o, prompts, pol), (trial, pol)


@pytest.mark.parametrize("policy", ["lpm", "dfs-weight"])
@pytest.mark.parametrize("page_size", [1, 4])
def test_scheduled_request_flow_matches_oracle(policy, page_size):
    """Waves of a fork tree in shuffled arrival order under a policy (the pool
    holds 60% of the distinct tokens): batches, served order, slot tables,
    decode slots, finishes and eviction order equal the oracle's."""
    wl = workloads.fork_tree(branching=3, depth=3, level_tokens=24, decode_steps=4)
    rng = random.Random(9)
    wl.waves = [rng.sample(w, len(w)) for w in wl.waves]
    if page_size > 1:
        wl = workloads.with_pages(wl, page_size)
    got = Engine(wl, policy=policy).run()
    want, _ = run_bookkeeping(wl.oracle_waves(), wl.num_slots, wl.decode_steps,
                              page_size=page_size, policy=policy)
    assert got.as_tuple() == want.as_tuple()
    assert got.stats == want.stats
    assert len(got.eviction_log) > 0
    fcfs, _ = run_bookkeeping(wl.oracle_waves(), wl.num_slots, wl.decode_steps,
                              page_size=page_size)
    # shuffled arrivals: the cache-aware order prefills no more than arrival order
    assert got.prefilled <= fcfs.prefilled


# ------------------------------------------------------- draft-tree rows
def test_verify_rows_follow_the_tree():
    """Each draft's row is its request's context then its root path (root
    first, itself last); context length and position follow its depth."""
    from oracle import speculative as ospec
    rng = random.Random(12)
    prefix_len = [5, 0, 9]
    stride = 12
    prefix_rows = np.zeros((3, stride), dtype=np.int32)
    for r, p in enumerate(prefix_len):
        prefix_rows[r, :p] = rng.sample(range(100, 200), p)
    trees = [[-1, 0, 0, 1, 3, -1], [-1], [-1, 0, 1, 2]]
    indptr = np.cumsum([0] + [len(t) for t in trees]).astype(np.int64)
    parents = np.concatenate([np.array(t, dtype=np.int32) for t in trees])
    slots = np.arange(500, 500 + len(parents), dtype=np.int32)
    rows, ctx, pos = rx.verify_rows(prefix_len, prefix_rows, indptr, parents, slots, 20)
    for r, tree in enumerate(trees):
        p = prefix_len[r]
        for li in range(len(tree)):
            i = indptr[r] + li
            path = [slots[indptr[r] + j] for j in ospec.ancestors_and_self(tree, li)]
            want = list(prefix_rows[r, :p]) + path
            assert rows[i, :len(want)].tolist() == want
            assert ctx[i] == len(want) and pos[i] == ospec.positions(p, tree)[li]
    with pytest.raises(rx.RxError):
        rx.verify_rows([2], prefix_rows[:1], [0, 2], [-1, 1], [1, 2], 20)   # parent not before
    with pytest.raises(rx.RxError):
        rx.verify_rows([9], prefix_rows[:1], [0, 4], [-1, 0, 1, 2], [1, 2, 3, 4], 12)  # too long


# --------------------------------------------------------------- two tiers
def test_two_tier_random_ops_match_oracle():
    """Random matches across tiers, loads, inserts, write-throughs (committed
    later with success or failure), locks and evictions on both caches:
    identical slots, nodes, tickets, copies, counts and eviction logs."""
    from oracle.hicache import TwoTierRadixCache
    rng = random.Random(43)
    for trial in range(50):
        ps = rng.choice([1, 2])
        ns, hs_ = ps * rng.randint(12, 30), ps * rng.randint(6, 24)
        o, n = TwoTierRadixCache(ns, hs_, ps), rx.RadixCache(ns, ps, hs_)
        olocks, nlocks, pend = [], [], []
        for step in range(100):
            seq = [rng.randrange(3) for _ in range(rng.randint(1, 10))]
            r = rng.random()
            if r < 0.45:
                os_, on, ohl, ohn = o.match_prefix_tiers(seq[:-1])
                ns_, nn, nhl, nhn = n.match_prefix_tiers(seq[:-1])
                assert (list(os_), on.id, ohl, ohn.id) == (ns_.tolist(), nn, nhl, nhn)
                if ohl:
                    try:
                        oload = o.load_onboard(ohn)
                    except ONoSpace:
                        oload = None
                    try:
                        h, d = n.load_onboard(nhn, 64)
                        nload = (h.tolist(), d.tolist())
                    except rx.NoSpace:
                        nload = None
                    assert (None if oload is None else (list(oload[0]), list(oload[1]))) == nload
                os_, on = o.match_prefix(seq[:-1])
                ns_, nn = n.match_prefix(seq[:-1])
                assert list(os_) == ns_.tolist() and on.id == nn
                o.inc_lock_ref(on)
                n.lock(nn)
                k = len(seq) - len(os_)
                try:
                    onew = o.alloc(k)
                except ONoSpace:
                    onew = None
                try:
                    nnew = n.alloc(k).tolist()
                except rx.NoSpace:
                    nnew = None
                assert onew == nnew
                if onew is None:
                    o.dec_lock_ref(on)
                    n.unlock(nn)
                    continue
                orow = list(os_) + onew
                oa, on2 = o.insert(seq, orow)
                na, nn2 = n.insert(seq, np.array(orow, dtype=np.int32))
                assert (oa, on2.id) == (na, nn2)
                extra = orow[len(os_):oa] + orow[o.aligned(len(seq)):]
                o.free(extra)
                n.free(np.array(extra, dtype=np.int32))
                o.inc_lock_ref(on2)
                n.lock(nn2)
                o.dec_lock_ref(on)
                n.unlock(nn)
                olocks.append(on2)
                nlocks.append(nn2)
            elif r < 0.6 and olocks:
                i = rng.randrange(len(olocks))
                on, nn = olocks.pop(i), nlocks.pop(i)
                o.dec_lock_ref(on)
                n.unlock(nn)
                try:
                    ot = o.write_through(on)
                except ONoSpace:
                    ot = None
                try:
                    t, d, h = n.write_through(nn, 64)
                    nt = (t, d.tolist(), h.tolist())
                except rx.NoSpace:
                    nt = None
                assert (None if ot is None else (ot[0], list(ot[1]), list(ot[2]))) == nt
                if nt and nt[0]:
                    pend.append(nt[0])
            elif r < 0.75 and pend:
                t = pend.pop(rng.randrange(len(pend)))
                ok = rng.random() < 0.8
                o.commit_write_through(t, ok)
                n.commit_write_through(t, ok)
            else:
                k = rng.randint(1, 8)
                assert o.evict(k) == n.evict(k)
            st = n.stats()
            assert st["cached_tokens"] == o.device_cached_size()
            assert st["host_cached_tokens"] == o.host_cached_size()
            assert st["evictable_tokens"] == o.evictable_size_
            assert st["protected_tokens"] == o.protected_size_
            assert st["free_slots"] == len(o.free_slots)
            assert st["host_free_slots"] == len(o.free_host_pages) * ps
            assert st["num_nodes"] == o.num_nodes()
            assert n.eviction_log() == o.eviction_log
            assert n.host_eviction_log() == o.host_eviction_log


@pytest.mark.parametrize("host_slots,page_size", [(4096, 1), (700, 1), (4096, 4)])
def test_tiered_request_flow_matches_oracle(host_slots, page_size):
    """A round-robin multi-turn chat under a device pool that holds about two
    sessions' histories, with a host tier (large, or small enough to evict):
    loads, backups, slot tables, finishes and both eviction logs equal the
    oracle's, and the host tier prefills less than one tier."""
    wl = workloads.multi_turn_chat(sessions=6, turns=4, system=64, user=24, decode_steps=8,
                                   layers=1)
    wl.waves = [[r] for w in wl.waves for r in w]
    wl.num_slots = 400
    if page_size > 1:
        wl.page_size = page_size
    got = Engine(wl, host_slots=host_slots).run()
    want, _ = run_bookkeeping(wl.oracle_waves(), wl.num_slots, wl.decode_steps,
                              page_size=page_size, host_slots=host_slots)
    assert got.as_tuple() == want.as_tuple()
    assert len(got.loads) > 0
    single, _ = run_bookkeeping(wl.oracle_waves(), wl.num_slots, wl.decode_steps,
                                page_size=page_size)
    assert got.prefilled < single.prefilled
    if host_slots == 700:
        assert len(got.host_eviction_log) > 0


# --------------------------------------------------------- fault injection
def _snapshot(c, tokens_list):
    """What a failed step must leave alone: stats, and the match (slots and
    node) of every sequence inserted so far."""
    st = c.stats()
    matches = [(c.match_length(t), c.match_prefix_tiers(t)[0].tolist()) for t in tokens_list]
    return st, matches


def test_injected_allocation_failures_leave_the_tree_unchanged():
    """A failing k-th allocation inside each batch step: the step reports
    RX_ERR_NO_SPACE (or skips, where the step skips), releases the locks it
    took, allocates nothing, and leaves every earlier sequence matched as
    before; the next step runs normally."""
    rng = np.random.default_rng(13)
    c = rx.RadixCache(4000, 1, 2000)
    seqs = [rng.integers(1, 50, size=int(rng.integers(20, 60))).astype(np.int32) for _ in range(6)]
    # cache a few sequences and back them up
    for sq in seqs[:4]:
        slots, _ = c.match_prefix(sq)
        _, node = c.insert(sq, np.concatenate([slots, c.alloc(len(sq) - len(slots))]))
        t, d, h = c.write_through(node, 200)
        if t:
            c.commit_write_through(t, True)
    before = c.stats()
    # extend_begin: the batch's one allocation fails -> no locks, no slots
    tok = np.concatenate(seqs[4:6])
    ind = np.array([0, len(seqs[4]), len(tok)], dtype=np.int64)
    table = np.zeros((2, 100), dtype=np.int32)
    c.debug_fail_alloc(1)
    with pytest.raises(rx.NoSpace):
        c.extend_begin(tok, ind, table)
    after = c.stats()
    assert after["protected_tokens"] == 0 and after["free_slots"] == before["free_slots"]
    assert after["cached_tokens"] == before["cached_tokens"]
    # alloc_steps: the second step fails, the first stays allocated
    c.debug_fail_alloc(2)
    with pytest.raises(rx.NoSpace):
        c.alloc_steps(3, 4)
    assert c.stats()["free_slots"] == before["free_slots"] - 3
    # write-through: the host allocation fails -> no ticket, nothing pending
    slots, _ = c.match_prefix(seqs[4])
    _, n4 = c.insert(seqs[4], np.concatenate([slots, c.alloc(len(seqs[4]) - len(slots))]))
    st0 = c.stats()
    c.debug_fail_alloc(1)
    with pytest.raises(rx.NoSpace):
        c.write_through(n4, 200)
    st1 = c.stats()
    assert st1["host_free_slots"] == st0["host_free_slots"] and st1["protected_tokens"] == 0
    # write-through batch skips the failing backup and takes the next
    d, h, cnt = c.write_through_batch(np.array([n4], dtype=np.int64), 200)
    assert len(d) == len(h) == cnt[0] > 0
    # evict seqs[0] from the device (it is backed up), then a failing load
    # is skipped by the batch load: the prefix is prefilled instead
    c.evict(4000)
    assert c.stats()["cached_tokens"] == 0
    c.debug_fail_alloc(1)
    hs, ds, cnt = c.load_batch(seqs[0], np.array([0, len(seqs[0])], dtype=np.int64), 200)
    assert len(hs) == 0 and cnt.tolist() == [0]
    assert c.stats()["cached_tokens"] == 0
    # off again: the load goes through
    c.debug_fail_alloc(0)
    hs, ds, cnt = c.load_batch(seqs[0], np.array([0, len(seqs[0])], dtype=np.int64), 200)
    assert cnt[0] == len(hs) > 0


def test_injected_failure_in_the_request_flow_is_reported_and_recoverable():
    """A whole request flow with the k-th allocation failing: the flow stops
    with NoSpace at that allocation; the cache's accounting stays
    consistent (evictable + protected == cached) and every lock the failing
    batch took is released."""
    wl = workloads.fork_tree(branching=3, depth=3, level_tokens=24, decode_steps=3)
    for k in (1, 2, 5, 9):
        eng = Engine(wl)
        orig = rx.RadixCache

        class Failing(orig):
            def __init__(self, *a, **kw):
                super().__init__(*a, **kw)
                self.debug_fail_alloc(k)

        rx.RadixCache = Failing
        try:
            with pytest.raises(rx.NoSpace):
                eng.run()
        finally:
            rx.RadixCache = orig
        st = eng.cache.stats()
        assert st["evictable_tokens"] + st["protected_tokens"] == st["cached_tokens"]


def _wave_prompts(rng, n, page_size):
    """Prompts with shared heads, identical copies and one-token prompts."""
    base = rng.integers(1, 40, size=400).astype(np.int32)
    out = []
    for i in range(n):
        if out and rng.random() < 0.15:
            out.append(out[int(rng.integers(0, len(out)))].copy())     # identical
            continue
        cut = int(rng.choice([0, page_size, 40, 120, 121, 300]))
        tail = rng.integers(1, 40, size=int(rng.integers(1, 60))).astype(np.int32)
        out.append(np.concatenate([base[:cut], tail]))
    out.append(base[:1].copy())
    tokens = np.concatenate(out).astype(np.int32)
    indptr = np.zeros(len(out) + 1, dtype=np.int64)
    np.cumsum([len(p) for p in out], out=indptr[1:])
    return tokens, indptr


def _by_batches(c, tokens, indptr, stride):
    """The wave through rx_batch_end / rx_extend_begin / rx_extend_end."""
    R = len(indptr) - 1
    table = np.zeros((R, stride), dtype=np.int32)
    ends, prefix, nodes, new, rew = [], np.zeros(R, np.int32), np.zeros(R, np.int64), [], []
    start = 0
    while start < R:
        end = c.batch_end(tokens, indptr, start)
        n = end - start
        pre = np.zeros(n, np.int32)
        mn = np.zeros(n, np.int64)
        nw = np.zeros(int(indptr[end] - indptr[start]), np.int32)
        ind = np.ascontiguousarray(indptr[start:end + 1])
        tot = c.extend_begin_p(n, tokens.ctypes.data, ind.ctypes.data,
                               table[start:].ctypes.data, stride, pre.ctypes.data,
                               mn.ctypes.data, nw.ctypes.data)
        new.append(nw[:tot])
        rew.append(c.extend_end_p(n, tokens.ctypes.data, ind.ctypes.data,
                                  table[start:].ctypes.data, stride, pre.ctypes.data,
                                  mn.ctypes.data, nodes[start:].ctypes.data))
        prefix[start:end] = pre
        ends.append(end)
        start = end
    return ends, prefix, nodes, np.concatenate(new), rew, table


@pytest.mark.parametrize("page_size", [1, 4])
def test_extend_wave_equals_batch_by_batch_calls(page_size):
    """rx_extend_wave makes exactly the decisions of the per-batch calls:
    batch ends, prefixes, nodes, new slots, rewritten rows, final rows, the
    eviction log and the cache's counts; identical prompts are rewritten to
    the tree's slots in both."""
    rng = np.random.default_rng(11 + page_size)
    evicted = rewritten = 0
    for trial in range(6):
        tokens, indptr = _wave_prompts(rng, 24, page_size)
        R, stride = len(indptr) - 1, int(np.max(np.diff(indptr)))
        # what the wave holds at once (a generous pool, no history)
        big = rx.RadixCache(1 << 16, page_size)
        _by_batches(big, tokens, indptr, stride)
        held = big.stats()["cached_tokens"] + R * page_size
        # odd trials: the 88-token history must be partly evicted
        slots = -(-(held + (40 if trial % 2 else 400)) // page_size) * page_size
        a = rx.RadixCache(slots, page_size)
        b = rx.RadixCache(slots, page_size)
        hist = rng.integers(40, 80, size=88).astype(np.int32)
        for c in (a, b):
            c.insert(hist, c.alloc(88))
        ends, prefix, nodes, new, rew, table = _by_batches(a, tokens, indptr, stride)
        w_table = np.zeros((R, stride), dtype=np.int32)
        w_ends = np.zeros(R, np.int32)
        w_pre = np.zeros(R, np.int32)
        w_nodes = np.zeros(R, np.int64)
        w_new = np.zeros(int(indptr[-1]), np.int32)
        w_rew = np.zeros(R, np.int64)
        nb = b.extend_wave_p(R, tokens.ctypes.data, indptr.ctypes.data, w_table.ctypes.data,
                             stride, w_ends, w_pre, w_nodes, w_new, w_rew)
        assert w_ends[:nb].tolist() == ends
        assert np.array_equal(w_pre, prefix) and np.array_equal(w_nodes, nodes)
        assert np.array_equal(w_new[:len(new)], new)
        assert w_rew[:nb].tolist() == rew
        assert np.array_equal(w_table, table)
        assert a.eviction_log() == b.eviction_log() and a.stats() == b.stats()
        evicted += len(a.eviction_log()) > 0
        rewritten += sum(rew)
    assert evicted and rewritten      # both branches were taken


def test_extend_wave_failure_keeps_earlier_batches():
    """An allocation failing in a later batch: the call reports it, the
    batches before it stay done (their nodes locked) and the failing batch
    holds no lock."""
    rng = np.random.default_rng(3)
    tokens, indptr = _wave_prompts(rng, 12, 1)
    R, stride = len(indptr) - 1, int(np.max(np.diff(indptr)))
    c = rx.RadixCache(5000)
    ref = rx.RadixCache(5000)
    ends, *_ = _by_batches(ref, tokens, indptr, stride)
    assert len(ends) >= 2
    c.debug_fail_alloc(2)       # the second batch's allocation fails
    out = [np.zeros(R, np.int32), np.zeros(R, np.int32), np.zeros(R, np.int64),
           np.zeros(int(indptr[-1]), np.int32), np.zeros(R, np.int64)]
    table = np.zeros((R, stride), dtype=np.int32)
    with pytest.raises(rx.NoSpace):
        c.extend_wave_p(R, tokens.ctypes.data, indptr.ctypes.data, table.ctypes.data, stride,
                        *out)
    st = c.stats()
    first = int(indptr[ends[0]])
    # the first batch's prompts are in the tree and protected; nothing else is
    assert st["protected_tokens"] == st["cached_tokens"]
    assert 0 < st["cached_tokens"] <= first
    c.debug_fail_alloc(0)


def test_wave_entry_points_validate_before_cuda():
    """rx_extend_batches, rx_extend_wave and the event calls reject bad
    arguments before any CUDA call (no GPU needed)."""
    import ctypes as C
    pool = rx.rx_pool_desc(16, 16, 8, 1, 2, 128, 0)
    assert rx._lib.rx_extend_batches(C.byref(pool), 0, 4, None, -1, 1.0, None, None) == rx.RX_ERR_INVALID
    assert rx._lib.rx_extend_batches(C.byref(pool), 0, 4, None, 2, 1.0, None, None) == rx.RX_ERR_INVALID
    bad = rx.rx_pool_desc(16, 16, 8, 1, 2, 64, 0)     # head_dim 64 unsupported
    recs = np.zeros(1, dtype=rx.EXTEND_BATCH_DTYPE)
    assert rx._lib.rx_extend_batches(C.byref(bad), 0, 4, recs.ctypes.data, 1, 1.0, None,
                                     None) == rx.RX_ERR_INVALID
    assert rx._lib.rx_extend_batches(C.byref(pool), 0, 4, recs.ctypes.data, 0, 1.0, None,
                                     None) == rx.RX_OK
    assert rx._lib.rx_events_create(-1, None) == rx.RX_ERR_INVALID
    assert rx._lib.rx_events_create(0, None) == rx.RX_OK
    assert rx._lib.rx_events_destroy(-1, None) == rx.RX_ERR_INVALID
    assert rx._lib.rx_event_elapsed_ms(None, None, None) == rx.RX_ERR_INVALID
    c = rx.RadixCache(64)
    n = C.c_int32()
    # a negative wave size, and a wave with no arrays
    assert rx._lib.rx_extend_wave(c._h, -1, None, None, None, 8, None, C.byref(n), None, None,
                                  None, None) == rx.RX_ERR_INVALID
    ind = np.zeros(1, dtype=np.int64)
    assert rx._lib.rx_extend_wave(c._h, 0, None, ind.ctypes.data, None, 8, None, C.byref(n),
                                  None, None, None, None) == rx.RX_OK
    assert n.value == 0


def test_extend_plan_counts_row_tiles():
    """rx_extend_plan: request r has s_r x G rows per KV head (its suffix
    tokens times the query heads sharing a KV head), cut into tiles of 128
    rows; an empty suffix has no tile.  Counts checked against that formula
    on ragged suffixes, and bad arguments rejected."""
    import ctypes as C
    rng = np.random.default_rng(5)
    for hq, hkv in ((32, 8), (16, 4), (8, 8), (64, 8)):
        G = hq // hkv
        s = rng.integers(0, 700, size=40)
        s[[3, 17]] = 0
        s[5], s[6], s[7] = 128 // G, 128 // G + 1, 1
        qo = np.zeros(len(s) + 1, dtype=np.int32)
        np.cumsum(s, out=qo[1:])
        for d in (128, 256):
            tiles, n = rx.extend_plan(qo, hq, hkv, d)
            want = np.zeros(len(s) + 1, dtype=np.int64)
            np.cumsum(-(-s * G // 128), out=want[1:])
            assert tiles.tolist() == want.tolist() and n == want[-1]
    tiles, n = rx.extend_plan(np.zeros(1, dtype=np.int32), 32, 8, 128)
    assert tiles.tolist() == [0] and n == 0
    for qo, hq, hkv, d in (([0, 5, 3], 32, 8, 128),     # not monotone
                           ([0, 5], 30, 8, 128),        # Hq % Hkv != 0
                           ([0, 5], 32, 8, 64)):        # head_dim
        with pytest.raises(rx.RxError) as e:
            rx.extend_plan(np.asarray(qo, dtype=np.int32), hq, hkv, d)
        assert e.value.status == rx.RX_ERR_INVALID
    out = np.zeros(3, dtype=np.int32)
    # at G = 256 two tiles per suffix token: 2^32 tiles overflow the int32 plan
    big = np.array([0, 2 ** 30 - 64, 2 ** 31 - 1], dtype=np.int32)
    n = C.c_int64()
    assert rx._lib.rx_extend_plan(big.ctypes.data, 1, 2048, 8, 128, out.ctypes.data,
                                  C.byref(n)) == rx.RX_OK and n.value == 2 ** 31 - 128
    assert rx._lib.rx_extend_plan(big.ctypes.data, 2, 2048, 8, 128, out.ctypes.data,
                                  C.byref(n)) == rx.RX_ERR_INVALID


def test_device_entry_points_reject_bad_arguments_without_a_gpu():
    """Each remaining device call rejects bad arguments (and returns at once
    on empty work) before any CUDA call, so none of this needs a GPU: slot
    table writes, decode (plain, static scratch, multi-step), verification,
    KV copies and page-locked allocations."""
    import ctypes as C
    L = rx._lib
    INV, OK = rx.RX_ERR_INVALID, rx.RX_OK
    pool = rx.rx_pool_desc(16, 16, 64, 2, 2, 128, 0)
    bad = rx.rx_pool_desc(16, 16, 64, 2, 2, 64, 0)            # head_dim 64
    other = rx.rx_pool_desc(32, 32, 64, 2, 4, 128, 0)         # other head count
    fake = 16                                                  # never dereferenced
    # req_to_token writes
    assert L.rx_req_to_token_write(fake, 4, 8, fake, fake, fake, -1, None) == INV
    assert L.rx_req_to_token_write(fake, 4, 0, fake, fake, fake, 1, None) == INV
    assert L.rx_req_to_token_write(fake, -1, 8, fake, fake, fake, 1, None) == INV
    assert L.rx_req_to_token_write(None, 4, 8, fake, fake, fake, 1, None) == INV
    assert L.rx_req_to_token_write(None, 4, 8, None, None, None, 0, None) == OK
    # decode and verification (the same checks)
    info = rx.rx_decode_plan_info()
    info.workspace_bytes = 4096
    for fn in (L.rx_decode_attention, L.rx_verify_attention):
        def call(p, hq=8, i=C.byref(info), B=1, q=fake, ws=fake, wsb=4096):
            return fn(C.byref(p), 0, q, hq, fake, 8, fake, i, B, 1.0, fake, fake, ws, wsb, None)
        assert call(bad) == INV and "head_dim" in rx.last_error()
        assert call(pool, hq=7) == INV                      # Hq % Hkv != 0
        assert call(pool, i=None) == INV                    # no plan info
        assert call(pool, B=-1) == INV
        assert call(pool, B=0) == OK                        # nothing to do
        assert call(pool, wsb=4095) == INV and "workspace" in rx.last_error()
        assert call(pool, ws=None) == INV
        assert call(pool, ws=fake + 8) == INV               # misaligned workspace
        assert call(pool, q=None) == INV
    # decode with the library's static scratch: a plan larger than it
    assert L.rx_decode_attention_static(C.byref(pool), 0, fake, 8, fake, 8, fake, None, 1, 1.0,
                                        fake, fake, None) == INV
    info.workspace_bytes = 16 * 2 ** 20 + 1
    assert L.rx_decode_attention_static(C.byref(pool), 0, fake, 8, fake, 8, fake,
                                        C.byref(info), 1, 1.0, fake, fake, None) == INV
    assert "static" in rx.last_error()
    # multi-step decode
    assert L.rx_decode_steps(C.byref(pool), 0, 8, fake, 8, None, -1, 1, 1.0, fake, 0,
                             None) == INV
    assert L.rx_decode_steps(C.byref(pool), 0, 8, fake, 8, None, 2, 1, 1.0, fake, 0,
                             None) == INV
    steps = (rx.rx_decode_step * 1)()
    assert L.rx_decode_steps(C.byref(bad), 0, 8, fake, 8, steps, 1, 1, 1.0, fake, 0,
                             None) == INV
    assert L.rx_decode_steps(C.byref(pool), 0, 6, fake, 8, steps, 1, 1, 1.0, fake, 0,
                             None) == INV                   # Hq % Hkv != 0
    # KV copies between pools
    assert L.rx_kv_copy(C.byref(pool), C.byref(bad), fake, fake, 1, None) == INV
    assert L.rx_kv_copy(C.byref(pool), C.byref(other), fake, fake, 1, None) == INV
    assert "shape" in rx.last_error()
    assert L.rx_kv_copy(C.byref(pool), C.byref(pool), fake, fake, -1, None) == INV
    assert L.rx_kv_copy(C.byref(pool), C.byref(pool), None, None, 0, None) == OK
    assert L.rx_kv_copy(C.byref(pool), C.byref(pool), None, fake, 1, None) == INV
    # page-locked host allocations
    out = C.c_void_p()
    assert L.rx_host_alloc(0, C.byref(out)) == INV
    assert L.rx_host_alloc(64, None) == INV


def _planned_wave(wl, wave_index, n_steps):
    """The wave's prompts inserted and locked in a fresh cache (earlier waves
    first, so later turns share their history), then one multi-step plan."""
    c = rx.RadixCache(sum(len(wl.prompt_tokens(r)) for w in wl.waves for r in w) + 4096)
    for w in wl.waves[:wave_index]:
        for r in w:
            toks = wl.prompt_tokens(r)
            slots, _ = c.match_prefix(toks)
            c.insert(toks, np.concatenate([slots, c.alloc(len(toks) - len(slots))]))
    nodes, lens = [], []
    for r in wl.waves[wave_index]:
        toks = wl.prompt_tokens(r)
        slots, _ = c.match_prefix(toks)
        _, node = c.insert(toks, np.concatenate([slots, c.alloc(len(toks) - len(slots))]))
        c.lock(node)
        nodes.append(node)
        lens.append(len(toks) + 1)
    B = len(nodes)
    plan, info = c.plan_decode(nodes, lens, list(range(B)), wl.num_q_heads, wl.num_kv_heads,
                               wl.head_dim, n_steps=n_steps)
    W = rx.RX_WORK_WORDS
    work = plan[info.off_work:info.off_work + info.n_work * W].reshape(-1, W).astype(np.int64)
    members = plan[info.off_members:info.off_members + info.n_member_entries]
    return work, members, info, lens


@pytest.mark.parametrize("name", ["long_shared", "chat_turn_3"])
def test_decode_plan_sizes_its_work_items(name):
    """The decode planner's sizing rules: warp-role items (listed first) hold
    at most 16 query rows (8 at head_dim 256), tensor-core items at most 128
    and key chunks of whole key tiles (128 keys, 64 at head_dim 256) except
    at a segment's end; tile CTAs (items x KV heads) stay within 128; each
    group runs heaviest first; every request's context over all steps is
    covered once.  On long_shared the 32,768-token prefix of 64 requests
    (512 rows per KV head: four blocks of 128) is cut into chunks of 8 keys
    per row doubled until 128 tile CTAs remain: 8,192 keys."""
    T = 4
    if name == "long_shared":
        wl = workloads.long_shared(decode_steps=T)
        work, members, info, lens = _planned_wave(wl, 0, T)
    else:
        wl = workloads.multi_turn_chat(sessions=64, turns=3, decode_steps=T, layers=1)
        work, members, info, lens = _planned_wave(wl, 2, T)
    G = wl.num_q_heads // wl.num_kv_heads
    small_rows = 16 if wl.head_dim == 128 else 8
    step = 128 if wl.head_dim == 128 else 64
    n_tc = int(info.n_work_tc)
    warp, tile = work[:len(work) - n_tc], work[len(work) - n_tc:]
    assert n_tc > 0 and len(warp) > 0
    assert (warp[:, 6] <= small_rows).all() and (warp[:, 6] == warp[:, 4] * G).all()
    assert (tile[:, 6] <= 128).all() and (tile[:, 6] > 32).all()
    assert n_tc * wl.num_kv_heads <= 128
    for grp in (warp, tile):
        weight = (grp[:, 2] - grp[:, 1]) * grp[:, 4]
        assert (np.diff(weight) <= 0).all()
    # tile chunks: whole key tiles except the last chunk of a segment
    seg_end = {}
    for row, kb, ke, *_ in tile:
        seg_end[row] = max(seg_end.get(row, 0), ke)
    for row, kb, ke, *_ in tile:
        assert (ke - kb) % step == 0 or ke == seg_end[row]
    # coverage: each request's keys 0 .. ctx + T - 1 once (the private tail
    # of the last step included)
    covered = {b: [] for b in range(len(lens))}
    for row, kb, ke, moff, nm, *_ in work:
        for i in range(nm):
            covered[int(members[moff + i])].append((kb, ke))
    for b, rng_ in covered.items():
        pos = 0
        for kb, ke in sorted(rng_):
            assert kb == pos
            pos = ke
        assert pos == lens[b] + T - 1
    if name == "long_shared":
        assert info.n_shared_segments == 1
        assert len(tile) == 16 and n_tc * wl.num_kv_heads == 128
        assert sorted(set((tile[:, 2] - tile[:, 1]).tolist())) == [8192]


def test_launch_groups_and_their_plans():
    """A wave's extend batches merge into launch groups that end after each
    batch whose rows were rewritten (and at the wave's end); each group's
    query offsets and tile plan, cut from the whole wave's, equal those of
    the group's requests planned alone."""
    from radix_tree_prefix_gb300.engine import cut_per_group, launch_groups
    assert launch_groups(np.array([0, 0, 0])) == [0, 3]
    assert launch_groups(np.array([0, 2, 0, 1])) == [0, 2, 4]   # the last batch ends anyway
    assert launch_groups(np.array([1])) == [0, 1]
    assert launch_groups(np.array([1, 1, 1])) == [0, 1, 2, 3]
    rng = np.random.default_rng(3)
    for trial in range(200):
        R = int(rng.integers(1, 40))
        sfx = rng.integers(0, 300, size=R)
        sfx[rng.random(R) < 0.1] = 0
        cuts = np.sort(rng.choice(np.arange(1, R), size=min(R - 1, int(rng.integers(0, 8))),
                                  replace=False)) if R > 1 else np.array([], dtype=np.int64)
        bounds = [0] + cuts.tolist() + [R]
        rew = (rng.random(len(bounds) - 1) < 0.3).astype(np.int64)
        gb = launch_groups(rew)
        assert gb[0] == 0 and gb[-1] == len(bounds) - 1 and gb == sorted(set(gb))
        go = np.asarray([bounds[g] for g in gb], dtype=np.int64)
        qo_w = np.zeros(R + 1, dtype=np.int32)
        np.cumsum(sfx, out=qo_w[1:])
        hq, hkv = [(32, 8), (16, 4), (8, 8)][trial % 3]
        tiles_w, _ = rx.extend_plan(qo_w, hq, hkv, 128)
        qo_c, tiles_c = cut_per_group(qo_w, go), cut_per_group(tiles_w, go)
        assert len(qo_c) == R + len(go) - 1
        for g in range(len(go) - 1):
            j0, j1 = int(go[g]), int(go[g + 1])
            want_qo = np.zeros(j1 - j0 + 1, dtype=np.int64)
            np.cumsum(sfx[j0:j1], out=want_qo[1:])
            want_tiles, _ = rx.extend_plan(want_qo.astype(np.int32), hq, hkv, 128)
            at = j0 + g
            assert qo_c[at:at + j1 - j0 + 1].tolist() == want_qo.tolist()
            assert tiles_c[at:at + j1 - j0 + 1].tolist() == want_tiles.tolist()
