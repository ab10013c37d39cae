"""GPU parity of the librx kernels against the fp64 oracle.

Every case runs the whole request flow through the C ABI (native cache +
CUDA kernels); bookkeeping must equal the oracle's bit for bit and attention
must be within max-abs 1e-2 / mean-abs 1e-3 of fp64 attention computed from
the token streams (as if every prompt were recomputed).
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU machines, skipped there
    pytest.skip("no CUDA device", allow_module_level=True)

from oracle import attention as oatt  # noqa: E402
from oracle import pool as opool  # noqa: E402
from parity_util import DeviceRun  # noqa: E402
from radix_tree_prefix_gb300 import rx, workloads  # noqa: E402
from radix_tree_prefix_gb300.workloads import Request, Workload  # noqa: E402


@pytest.mark.parametrize("d,hkv,T", [(128, 2, 1), (128, 8, 777), (256, 4, 300), (128, 1, 4096)])
def test_kv_store_bit_exact(d, hkv, T):
    dev = torch.device("cuda:0")
    L, N = 2, 5000
    g = torch.Generator(device=dev).manual_seed(T)
    kp = torch.randn((L, hkv, N, d), generator=g, device=dev).to(torch.bfloat16)
    vp = torch.randn((L, hkv, N, d), generator=g, device=dev).to(torch.bfloat16)
    k = torch.randn((T, hkv, d), generator=g, device=dev).to(torch.bfloat16)
    v = torch.randn((T, hkv, d), generator=g, device=dev).to(torch.bfloat16)
    slots = (torch.randperm(N - 1, generator=g, device=dev)[:T] + 1).to(torch.int32)
    want_k = opool.store(kp.float().cpu().numpy(), 1, slots.cpu().numpy(), k.float().cpu().numpy())
    want_v = opool.store(vp.float().cpu().numpy(), 1, slots.cpu().numpy(), v.float().cpu().numpy())
    rx.kv_store(rx.pool_desc(kp, vp), 1, slots, k, v)
    torch.cuda.synchronize()
    assert rx.device_check() == 0
    assert np.array_equal(kp.float().cpu().numpy(), want_k)
    assert np.array_equal(vp.float().cpu().numpy(), want_v)


def test_out_of_range_indices_are_skipped_and_reported():
    """A slot outside the pool (kv_store) or a row or position outside the
    slot table (req_to_token write) is skipped on the device, leaves memory
    untouched and is reported by rx_device_check (bits 0 and 4)."""
    dev = torch.device("cuda:0")
    kp = torch.zeros((1, 2, 64, 128), dtype=torch.bfloat16, device=dev)
    vp = torch.zeros_like(kp)
    k = torch.ones((3, 2, 128), dtype=torch.bfloat16, device=dev)
    slots = torch.tensor([5, 64, 7], dtype=torch.int32, device=dev)   # 64 is outside
    rx.kv_store(rx.pool_desc(kp, vp), 0, slots, k, k)
    torch.cuda.synchronize()
    with pytest.raises(rx.RxError) as e:
        rx.device_check()
    assert "(flags 1)" in str(e.value)
    assert int((kp[0, :, 5] != 0).sum()) == 256 and int((kp[0, :, 7] != 0).sum()) == 256
    assert int((kp != 0).sum()) == 512
    table = torch.zeros((4, 16), dtype=torch.int32, device=dev)
    rows = torch.tensor([0, 4, 1, -1, 2], dtype=torch.int32, device=dev)
    pos = torch.tensor([3, 0, 16, 0, 15], dtype=torch.int32, device=dev)
    vals = torch.tensor([11, 12, 13, 14, 15], dtype=torch.int32, device=dev)
    rx.req_to_token_write(table, rows, pos, vals)
    torch.cuda.synchronize()
    with pytest.raises(rx.RxError) as e:
        rx.device_check()
    assert "(flags 16)" in str(e.value)
    want = torch.zeros_like(table)
    want[0, 3], want[2, 15] = 11, 15
    assert torch.equal(table, want)
    assert rx.device_check() == 0      # flags were cleared


def test_empty_calls_launch_nothing():
    dev = torch.device("cuda:0")
    kp = torch.zeros((1, 1, 8, 128), dtype=torch.bfloat16, device=dev)
    e = torch.zeros(0, dtype=torch.int32, device=dev)
    rx.kv_store(rx.pool_desc(kp, kp), 0, e, kp, kp)
    torch.cuda.synchronize()


SMALL = {
    # the nested example at full size: 3 batches, 3,060 prefilled tokens
    "nested_share": (lambda: workloads.nested_share(), None),
    # shared preamble + ragged suffixes + decode (G = 4)
    "agent_small": (lambda: workloads.agent_loop(calls=6, preamble=300, lo=20, hi=60,
                                                 decode_steps=5), None),
    # G = 1 and G = 8
    "agent_g1": (lambda: workloads.agent_loop(calls=5, preamble=200, lo=1, hi=70, decode_steps=3,
                                              q_heads=4, kv_heads=4), None),
    "agent_g8": (lambda: workloads.agent_loop(calls=5, preamble=150, lo=30, hi=90,
                                              decode_steps=3, q_heads=64, kv_heads=8), None),
    # head_dim 256, two layers, multi-turn waves (history reuse)
    "chat_d256": (lambda: workloads.multi_turn_chat(sessions=4, turns=3, system=100, user=40,
                                                    decode_steps=4, layers=2), None),
    # branching tree with a small pool: eviction, slot reuse, nested shared segments
    "fork_evict": (lambda: workloads.fork_tree(branching=3, depth=3, level_tokens=48,
                                               decode_steps=4), None),
    # many members on one shared segment: several member blocks of a chunk
    "long_shared_small": (lambda: workloads.long_shared(batch=20, prefix=700, unique=50,
                                                        decode_steps=3), None),
    # paged pools: whole-page keys and allocation, partly filled last pages,
    # decode tokens continuing a request's page
    "agent_p16": (lambda: workloads.with_pages(
        workloads.agent_loop(calls=6, preamble=300, lo=20, hi=60, decode_steps=21), 16), None),
    "fork_evict_p4": (lambda: workloads.with_pages(
        workloads.fork_tree(branching=3, depth=3, level_tokens=48, decode_steps=4), 4), None),
    "chat_d256_p16": (lambda: workloads.with_pages(
        workloads.multi_turn_chat(sessions=4, turns=3, system=100, user=40, decode_steps=4,
                                  layers=2), 16), None),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_workload_parity(name):
    wl = SMALL[name][0]()
    run = DeviceRun(wl)
    mx, mean, n = run.assert_close()
    if name == "nested_share":
        assert run.trace.prefilled == 3060
    if name.startswith("fork_evict"):
        assert len(run.trace.eviction_log) > 0


def test_single_token_suffixes_and_duplicates():
    """Prompts that extend the previous one by one token (a 1-query extend
    over a long prefix) and an identical prompt (rows adopt tree slots)."""
    s = workloads._Segments(77)
    base = s.new(300)
    ones = [s.new(1) for _ in range(4)]
    outs = [s.new(3) for _ in range(6)]
    waves = []
    for k in range(4):
        waves.append([Request(k, (base,) + tuple(ones[:k + 1]), outs[k])])
    waves.append([Request(4, (base, ones[0]), outs[4]), Request(5, (base, ones[0]), outs[5])])
    wl = Workload("one_token", 1, 16, 4, 128, 2000, 3, s.tokens, waves, 77)
    run = DeviceRun(wl)
    run.assert_close()
    assert [len(b) for b in run.trace.batches] == [1, 1, 1, 1, 1, 1]


def test_agent_loop_full_size_sampled():
    """The benchmark workload at full size: bookkeeping bit-exact, sampled
    extend rows of 6 requests and decode rows at 3 steps."""
    wl = workloads.agent_loop()
    run = DeviceRun(wl, sample={0, 1, 7, 20, 38, 39}, extend_tokens=48, decode_steps={0, 31, 63})
    run.assert_close()


def test_long_shared_full_size_sampled():
    wl = workloads.long_shared()
    run = DeviceRun(wl, sample={0, 1, 63}, extend_tokens=24, decode_steps={0, 127})
    run.assert_close()


def test_fork_tree_full_size_sampled():
    wl = workloads.fork_tree()
    run = DeviceRun(wl, sample={0, 3, 130, 377, 624}, extend_tokens=16, decode_steps={0, 15})
    run.assert_close()
    assert len(run.trace.eviction_log) > 100


def test_multi_turn_chat_full_size_sampled():
    """head_dim 256 at full size (256 sessions x 8 turns over a 2,000-token
    system prompt, 477,137 pool slots): bookkeeping bit-exact; the first and
    the last of the 16 layers run the same launches as in the benchmark and
    are sampled in five sessions' turns at the first and last decode step."""
    wl = workloads.multi_turn_chat()
    run = DeviceRun(wl, layers=[0, 15], sample={0, 1, 255, 1024, 2047}, extend_tokens=16,
                 decode_steps={0, 31})
    run.assert_close()


@pytest.mark.parametrize("head_dim", [128, 256])
@pytest.mark.parametrize("doubling", [128, 192])
def test_running_max_grows_over_key_tiles(head_dim, doubling):
    """Keys of the shared preamble grow in norm along the sequence (x2 every
    `doubling` positions), so rows are peaked and their running max rises from
    key tile to key tile: by more than 8 (log2 units) at many tiles, where the
    tile rescales O in TMEM after waiting for the previous tile's PV product,
    and by up to 8 at others, where the dominant keys' exponents are positive
    (relative to the stale max).  A few keys carry each row here, so the
    rounding of each weight shows in the output instead of averaging out; the
    tile is held to the same tolerances."""
    # 12 calls x 4 query heads per KV head: the preamble's decode chunks have
    # 48 rows and go to the tensor-core tile as well
    wl = workloads.agent_loop(calls=12, preamble=700, lo=20, hi=60, decode_steps=3,
                              head_dim=head_dim)

    def ramp(vals):
        for layer, k in vals["k"].items():
            n = min(700, k.shape[0])
            f = torch.exp2(torch.arange(n, device=k.device, dtype=torch.float32) / doubling)
            k[:n] = (k[:n].float() * f[:, None, None]).to(torch.bfloat16)

    run = DeviceRun(wl, values_fn=ramp)
    mx, mean, n = run.assert_close()
    print(f"peaked rows, head_dim {head_dim}, doubling {doubling}: max abs {mx:.2e}, "
          f"mean abs {mean:.2e} over {n} rows")


def test_host_input_replay_with_reused_outputs_is_bit_identical():
    """The end-to-end path (inputs replayed from pinned host memory through
    per-position device buffers refilled one batch ahead on a side stream,
    output tensors reused run to run) gives, on every run, exactly the
    outputs of a run fed from device tensors."""
    from radix_tree_prefix_gb300.engine import Engine, GatherInputs, PreparedInputs

    dev = torch.device("cuda:0")
    wl = workloads.agent_loop(calls=6, preamble=300, lo=20, hi=60, decode_steps=4)
    vals = workloads.make_values(wl, dev, [0])

    def collect(store):
        def on_ext(b, rids, prefix, qo, outs):
            store[("e", b)] = tuple(x.clone() for x in outs[0])

        def on_wave(s, rids, ctx, outs, info):
            store[("d", s)] = tuple(x.clone() for x in outs[0])
        return on_ext, on_wave

    want = {}
    e, w = collect(want)
    prepared = PreparedInputs(GatherInputs(wl, vals, [0]))
    Engine(wl, device=dev, inputs=prepared, layers=[0], on_extend=e, on_decode_wave=w).run()
    prepared.freeze()
    torch.cuda.synchronize()

    host = PreparedInputs(prepared.source, host=True)
    host.adopt(prepared)
    host.freeze()
    got = {}
    e, w = collect(got)
    eng = Engine(wl, device=dev, inputs=host, layers=[0], on_extend=e, on_decode_wave=w,
                 reuse_outputs=True)
    for _ in range(3):
        got.clear()
        eng.run()
        torch.cuda.synchronize()
        assert got.keys() == want.keys()
        for k in want:
            for a, b in zip(got[k], want[k]):
                assert torch.equal(a, b), k
    assert rx.device_check() == 0


def test_output_ring_reads_back_every_output():
    """End-to-end output path: with as many ring buffers as launches, the
    host side of buffer i holds launch i's output (o then lse, fp32) exactly
    as a run into fresh device tensors computes it, on each of two runs."""
    from radix_tree_prefix_gb300.engine import Engine, GatherInputs, OutputRing, PreparedInputs

    dev = torch.device("cuda:0")
    wl = workloads.agent_loop(calls=6, preamble=300, lo=20, hi=60, decode_steps=4)
    vals = workloads.make_values(wl, dev, [0])
    want = []
    seen = []

    def on_ext(b, rids, prefix, qo, outs):
        # the batches of one launch group get views of the group's tensors
        o, lse = (x if x._base is None else x._base for x in outs[0])
        if seen and seen[-1] == (o.data_ptr(), o.numel()):
            return
        seen.append((o.data_ptr(), o.numel()))
        want.append(torch.cat([o.reshape(-1), lse.reshape(-1)]).clone())

    def on_wave(s, rids, ctx, outs, info):
        seen.clear()        # the next wave's groups may reuse freed addresses
        want.append(torch.cat([x.reshape(-1) for x in outs[0]]).clone())

    prepared = PreparedInputs(GatherInputs(wl, vals, [0]))
    Engine(wl, device=dev, inputs=prepared, layers=[0], on_extend=on_ext,
           on_decode_wave=on_wave).run()
    prepared.freeze()
    torch.cuda.synchronize()
    host = PreparedInputs(prepared.source, host=True, ring=2)
    host.adopt(prepared)
    host.freeze()
    n = max(w.numel() for w in want)
    ring = OutputRing(dev, n, slots=len(want))
    eng = Engine(wl, device=dev, inputs=host, layers=[0], out_ring=ring)
    for _ in range(2):
        ring.d2h_bytes = 0
        eng.run()
        torch.cuda.synchronize()
        for i, w in enumerate(want):
            got = ring.host[i].view(0, (w.numel(),), torch.float32)
            assert torch.equal(got, w.cpu()), i
        assert ring.d2h_bytes == 4 * sum(w.numel() for w in want)
    assert rx.device_check() == 0
    ring.close()
    host.close()


@pytest.mark.parametrize("policy", ["lpm", "dfs-weight"])
def test_scheduled_fork_tree_parity(policy):
    """A fork tree whose leaves arrive shuffled, served in the policy's order
    under a pool that holds 60% of the distinct tokens (eviction, slot
    reuse): bookkeeping bit-exact, attention within tolerance."""
    import random
    wl = workloads.fork_tree(branching=3, depth=3, level_tokens=48, decode_steps=4)
    rng = random.Random(9)
    wl.waves = [rng.sample(w, len(w)) for w in wl.waves]
    run = DeviceRun(wl, policy=policy)
    run.assert_close()
    assert len(run.trace.eviction_log) > 0


@pytest.mark.parametrize("name,chunk", [("agent_small", 37), ("chat_d256", 100),
                                        ("long_shared_small", 256), ("nested_share", 1000)])
def test_chunked_extend_parity(name, chunk):
    """Chunked prefill: every extend batch's queries in launches of at most
    `chunk` query tokens (suffixes split across launches, ragged last
    chunk): outputs within tolerance of the fp64 oracle, bookkeeping
    unchanged."""
    wl = SMALL[name][0]()
    run = DeviceRun(wl, chunk_tokens=chunk)
    run.assert_close()
    assert run.engine.gpu_launches > 0


@pytest.mark.parametrize("host_slots,page_size", [(8192, 1), (704, 1), (8192, 16)])
def test_two_tier_chat_parity(host_slots, page_size):
    """A round-robin multi-turn chat (head_dim 256, two layers) whose device
    pool holds about two sessions' histories, with a host tier: evicted
    histories come back from the page-locked host pool (written through at
    every finish, copied back by rx_kv_copy before the extend that reads
    them); bookkeeping bit-exact, every attention output within tolerance."""
    wl = workloads.multi_turn_chat(sessions=6, turns=4, system=64, user=24, decode_steps=8,
                                   layers=2)
    wl.waves = [[r] for w in wl.waves for r in w]
    wl.num_slots = 512
    wl.page_size = page_size
    run = DeviceRun(wl, host_slots=host_slots)
    run.assert_close()
    assert len(run.trace.loads) > 0
    if host_slots == 704:
        assert len(run.trace.host_eviction_log) > 0


def _dup_waves(pool=735):
    """Identical prompts in one wave: the second's row is rewritten to the
    tree's slots and its own new slot freed, and a later batch of the same
    wave, short of free slots, takes that slot again (then evicts the first
    wave's history for the rest)."""
    s = workloads._Segments(91)
    base, x, a, big, tail = s.new(300), s.new(200), s.new(40), s.new(150), s.new(60)
    outs = [s.new(3) for _ in range(5)]
    waves = [[Request(0, (base, x), outs[0])],
             [Request(1, (base, a), outs[1]), Request(2, (base, a), outs[2]),
              Request(3, (base, big), outs[3]), Request(4, (base, big, tail), outs[4])]]
    return Workload("dups", 1, 16, 4, 128, pool, 3, s.tokens, waves, 91)


@pytest.mark.parametrize("name", ["fork_evict", "chat_d256", "fork_evict_p4", "dups"])
def test_wave_launches_equal_batch_launches(name):
    """A wave's extend batches launched in groups (rx_extend_batches: per
    group one store and one attention over all its batches' requests, a
    group ending at a batch with rewritten rows) give bit for bit the outputs
    of launching batch by batch (the per-batch path), and the timing events
    bracket each group's store and attention."""
    from radix_tree_prefix_gb300.engine import Engine, GatherInputs, PreparedInputs

    dev = torch.device("cuda:0")
    wl = _dup_waves() if name == "dups" else SMALL[name][0]()
    layers = list(range(wl.num_layers))
    vals = workloads.make_values(wl, dev, layers)

    def run(**kw):
        store = {}

        def on_ext(b, rids, prefix, qo, outs):
            store[b] = [tuple(x.clone() for x in outs[ly]) for ly in layers]
        eng = Engine(wl, device=dev, inputs=PreparedInputs(GatherInputs(wl, vals, layers)),
                     layers=layers, on_extend=on_ext, **kw)
        trace = eng.run()
        torch.cuda.synchronize()
        return store, trace, eng

    per_batch, t0, _ = run(chunk_tokens=1 << 30)
    waved, t1, eng = run(timing=True)
    assert t0.as_tuple() == t1.as_tuple()
    assert len(t1.batches) > len(wl.waves)          # waves of several batches
    assert per_batch.keys() == waved.keys()
    for b in per_batch:
        for x, y in zip(per_batch[b], waved[b]):
            for a, c in zip(x, y):
                assert torch.equal(a, c), b
    kinds = [k for k, *_ in eng.kernel_events if k in ("kv_store", "extend")]
    n = kinds.count("extend")
    assert n == kinds.count("kv_store")
    assert len(wl.waves) * len(layers) <= n < len(t1.batches) * len(layers)
    if name == "dups":
        # wave 2's last batch reuses the slot its second batch's rewrite freed
        new = [int(x) for b in t1.batches[1:] for _, m, row in b for x in row[m:]]
        assert len(new) > len(set(new)) and len(t1.eviction_log) > 0
        assert n == 3       # wave 1; wave 2 split after the rewriting batch
    assert all(a.elapsed_time(e) > 0 for k, a, e, _ in eng.kernel_events if k == "extend")
    assert rx.device_check() == 0


@pytest.mark.parametrize("head_dim,hq,hkv", [(128, 16, 4), (256, 16, 4), (128, 8, 8)])
def test_row_tiles_at_the_64_row_boundary(head_dim, hq, hkv):
    """Row tiles of at most 64 rows run M = 64 tensor-core products (rows in
    the first 16 TMEM lanes of each quadrant), larger ones M = 128: suffixes
    of 16 and 17 tokens at G = 4 (64 and 68 rows), 32 and 33 (128, 132),
    and at G = 1 suffixes of 64 and 65 tokens, over a shared prefix; decode
    member blocks of 8 and 17 requests take the same split."""
    G = hq // hkv
    s = workloads._Segments(404)
    pre = s.new(300)
    lens = [16, 17, 32, 33] if G > 1 else [64, 65, 7, 1]
    outs = [s.new(2) for _ in range(25)]
    first = [Request(99, (pre,), outs[24])]        # the prefix is cached first
    wave = [Request(k, (pre, s.new(n)), outs[k]) for k, n in enumerate(lens)]
    # decode: a shared prefix over 17 requests (G x 17 rows: member blocks
    # of 128 / G requests and the rest)
    big = [Request(10 + k, (pre, s.new(3)), outs[4 + k]) for k in range(17)]
    wl = Workload("m64", 1, hq, hkv, head_dim, 8000, 2, s.tokens, [first, wave, big], 404)
    run = DeviceRun(wl)
    run.assert_close()
    assert [m for _, m, _ in run.trace.batches[1]] == [300] * 4


def test_rings_with_several_launch_groups_per_wave():
    """The end-to-end path (inputs replayed from page-locked host memory
    through the input ring, outputs read back through the output ring)
    hands its rings over group by group; on a wave split into several launch
    groups (identical prompts) every output read back equals the output of
    a run fed from device tensors, on each of two runs."""
    from radix_tree_prefix_gb300.engine import Engine, GatherInputs, OutputRing, PreparedInputs

    dev = torch.device("cuda:0")
    wl = _dup_waves()
    vals = workloads.make_values(wl, dev, [0])
    want, seen = [], []

    def on_ext(b, rids, prefix, qo, outs):
        o, lse = (x if x._base is None else x._base for x in outs[0])
        if seen and seen[-1] == (o.data_ptr(), o.numel()):
            return
        seen.append((o.data_ptr(), o.numel()))
        want.append(torch.cat([o.reshape(-1), lse.reshape(-1)]).clone())

    def on_wave(s, rids, ctx, outs, info):
        seen.clear()
        want.append(torch.cat([x.reshape(-1) for x in outs[0]]).clone())

    prepared = PreparedInputs(GatherInputs(wl, vals, [0]))
    first = Engine(wl, device=dev, inputs=prepared, layers=[0], on_extend=on_ext,
                   on_decode_wave=on_wave)
    first.run()
    prepared.freeze()
    torch.cuda.synchronize()
    assert len(want) > 2 * len(wl.waves)          # some wave has several groups
    host = PreparedInputs(prepared.source, host=True, ring=2)
    host.adopt(prepared)
    host.freeze()
    n = max(w.numel() for w in want)
    ring = OutputRing(dev, n, slots=len(want))
    eng = Engine(wl, device=dev, inputs=host, layers=[0], out_ring=ring)
    for _ in range(2):
        eng.run()
        torch.cuda.synchronize()
        for k, w in enumerate(want):
            got = ring.host[k].view(0, (w.numel(),), torch.float32)
            assert torch.equal(got, w.cpu()), k
    assert rx.device_check() == 0
    ring.close()
    host.close()


def _tile_kinds(rows, prefix, sfx, BM, BN, G):
    """The kinds of key tiles in the slot rows: 'run' (one run of BN
    slots), 'mixed' (not one run, but some of its 16-row groups are runs of
    valid slots: a tile that straddles runs of the pool) or 'gather' (no
    group is a run)."""
    kinds = set()
    for row, p, s in zip(rows, prefix, sfx):
        per = max(1, BM // G)
        for r0 in range(0, s, per):
            kend = p + min(s, r0 + per)
            for k0 in range(0, kend, BN):
                sl = np.full(BN, -1)
                seg = row[k0:min(kend, k0 + BN)]
                sl[:len(seg)] = seg
                groups = [sl[g:g + 16] for g in range(0, BN, 16)]
                ok = [x[0] >= 0 and np.all(np.diff(x) == 1) for x in groups]
                if len(seg) == BN and np.all(np.diff(sl) == 1):
                    kinds.add("run")
                else:
                    kinds.add("mixed" if any(ok) else "gather")
    return kinds


@pytest.mark.parametrize("head_dim,hq,hkv", [(128, 16, 4), (256, 16, 4), (128, 8, 8)])
def test_extend_over_slot_rows_of_mixed_runs(head_dim, hq, hkv):
    """Slot rows made of runs of the pool of mixed lengths (whole 16-row
    groups, runs of 17 and 100, single slots) give key tiles of one run
    (box loads), tiles that straddle runs and scattered tiles (gathered slot
    by slot).  Extend attention over them equals fp64 attention over the
    same slots."""
    dev = torch.device("cuda:0")
    rng = np.random.default_rng(1700 + head_dim + hkv)
    N, L, layer = 9000, 2, 1
    G = hq // hkv
    BN = 128 if head_dim == 128 else 64
    kp = (torch.randn(L, hkv, N, head_dim, generator=torch.Generator().manual_seed(5)) * 0.7)
    vp = torch.randn(L, hkv, N, head_dim, generator=torch.Generator().manual_seed(6))
    kp, vp = kp.to(torch.bfloat16), vp.to(torch.bfloat16)

    def slot_row(n):
        out = []
        while len(out) < n:
            m = int(rng.choice([16, 32, 48, 128, 17, 100, 1, 3]))
            a = int(rng.integers(0, N - m))
            out.extend(range(a, a + m))
        return np.asarray(out[:n], dtype=np.int32)

    prefix = [0, 300, 517, 64, 1000]
    sfx = [70, 1, 130, 200, 33]
    R = len(prefix)
    W = max(p + s for p, s in zip(prefix, sfx))
    rows = [slot_row(p + s) for p, s in zip(prefix, sfx)]
    rows[4][:256] = np.arange(4000, 4256)          # whole tiles of one run
    assert _tile_kinds(rows, prefix, sfx, 128, BN, G) == {"run", "mixed", "gather"}
    table = np.zeros((R + 2, W + 5), dtype=np.int32)
    req_rows = np.array([2, 0, 4, 1, 3], dtype=np.int32)
    for r in range(R):
        table[req_rows[r], :len(rows[r])] = rows[r]
    qo = np.zeros(R + 1, dtype=np.int32)
    np.cumsum(sfx, out=qo[1:])
    q = torch.randn(int(qo[-1]), hq, head_dim, generator=torch.Generator().manual_seed(7))
    q = q.to(torch.bfloat16)
    tiles, n_tiles = rx.extend_plan(qo, hq, hkv, head_dim)

    kd, vd, qd = kp.to(dev), vp.to(dev), q.to(dev)
    out = torch.full((int(qo[-1]), hq, head_dim), float("nan"), device=dev)
    lse = torch.full((int(qo[-1]), hq), float("nan"), device=dev)
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)  # noqa: E731
    pool = rx.pool_desc(kd, vd)
    rx.extend_attention(pool, layer, qd, hq, i32(table), i32(req_rows), i32(prefix), i32(qo),
                        i32(tiles), R, n_tiles, head_dim ** -0.5, out, lse)
    torch.cuda.synchronize()
    assert rx.device_check() == 0
    o, ls = out.double().cpu().numpy(), lse.double().cpu().numpy()
    k64 = kp[layer].double().numpy()
    v64 = vp[layer].double().numpy()
    q64 = q.double().numpy()
    errs = []
    for r in range(R):
        sl = rows[r]
        k = k64[:, sl, :].transpose(1, 0, 2)
        v = v64[:, sl, :].transpose(1, 0, 2)
        want_o, want_l = oatt.extend_attention(q64[qo[r]:qo[r + 1]], k, v, prefix[r])
        errs.append(np.abs(o[qo[r]:qo[r + 1]] - want_o).ravel())
        errs.append(np.abs(ls[qo[r]:qo[r + 1]] - want_l).ravel())
    e = np.concatenate(errs)
    assert e.max() <= 1e-2 and e.mean() <= 1e-3, (e.max(), e.mean())


@pytest.mark.parametrize("head_dim,hq,hkv", [(128, 16, 4), (256, 16, 4)])
def test_pool_rows_outside_the_slots_are_never_read(head_dim, hq, hkv):
    """No kernel reads a pool row that the slot rows do not name: with every
    other row NaN, extend attention over slot rows with ragged runs (partial
    last key tiles inside one run, tiles that straddle runs) equals fp64
    attention, and equals bit for bit the same call on a pool whose other
    rows are zero."""
    dev = torch.device("cuda:0")
    rng = np.random.default_rng(2900 + head_dim)
    N = 6000
    prefix = [200, 0, 333, 90]
    sfx = [57, 300, 41, 129]
    rows = [np.arange(1000, 1257, dtype=np.int32),              # one ragged run
            np.arange(2000, 2300, dtype=np.int32)]
    for p, s in zip(prefix[2:], sfx[2:]):
        out = []
        while len(out) < p + s:
            m = int(rng.choice([16, 64, 100, 7]))
            a = int(rng.integers(3000, N - m))
            out.extend(range(a, a + m))
        rows.append(np.asarray(out[:p + s], dtype=np.int32))
    used = np.unique(np.concatenate(rows))
    gen = torch.Generator().manual_seed(11)
    kp = torch.full((1, hkv, N, head_dim), float("nan"))
    vp = torch.full((1, hkv, N, head_dim), float("nan"))
    kp[:, :, used] = torch.randn(1, hkv, len(used), head_dim, generator=gen) * 0.7
    vp[:, :, used] = torch.randn(1, hkv, len(used), head_dim, generator=gen)
    kp, vp = kp.to(torch.bfloat16), vp.to(torch.bfloat16)
    R = len(rows)
    W = max(len(r) for r in rows)
    table = np.zeros((R, W), dtype=np.int32)
    for r in range(R):
        table[r, :len(rows[r])] = rows[r]
    qo = np.zeros(R + 1, dtype=np.int32)
    np.cumsum(sfx, out=qo[1:])
    q = (torch.randn(int(qo[-1]), hq, head_dim, generator=gen)).to(torch.bfloat16)
    tiles, n_tiles = rx.extend_plan(qo, hq, hkv, head_dim)
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)  # noqa: E731
    args = (i32(table), i32(np.arange(R)), i32(prefix), i32(qo), i32(tiles))

    def run(kd, vd):
        out = torch.empty((int(qo[-1]), hq, head_dim), device=dev)
        lse = torch.empty((int(qo[-1]), hq), device=dev)
        rx.extend_attention(rx.pool_desc(kd, vd), 0, q.to(dev), hq,
                            args[0], args[1], args[2], args[3], args[4], R, n_tiles,
                            head_dim ** -0.5, out, lse)
        torch.cuda.synchronize()
        assert rx.device_check() == 0
        return out, lse

    o, ls = run(kp.to(dev), vp.to(dev))
    assert torch.isfinite(o).all() and torch.isfinite(ls).all()
    k64, v64 = kp[0].double().numpy(), vp[0].double().numpy()
    q64 = q.double().numpy()
    on, lsn = o.double().cpu().numpy(), ls.double().cpu().numpy()
    for r in range(R):
        k = k64[:, rows[r], :].transpose(1, 0, 2)
        v = v64[:, rows[r], :].transpose(1, 0, 2)
        want_o, want_l = oatt.extend_attention(q64[qo[r]:qo[r + 1]], k, v, prefix[r])
        assert np.abs(on[qo[r]:qo[r + 1]] - want_o).max() <= 1e-2
        assert np.abs(lsn[qo[r]:qo[r + 1]] - want_l).max() <= 1e-2
    kz, vz = kp.nan_to_num(0.0).to(dev), vp.nan_to_num(0.0).to(dev)
    o0, l0 = run(kz, vz)
    assert torch.equal(o0, o) and torch.equal(l0, ls)
