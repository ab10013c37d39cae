"""Oracle request flow over the radix cache.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The flow follows "SGLang: Structured LLM Programs for Efficient Inference",
section "How RadixAttention reuses past work": (1) match the longest prefix,
(2) lock the matched nodes, (3) prefill only the rest, (4) decode and insert
(the prompt suffix and the output tokens become nodes), (5) on finish unlock.
Batching of extends follows the in-batch prefix rule of "SGLang: the tree, and
the language nobody remembers", section "The scheduler is where the cache is
won or lost": a request that shares more with a request already queued in the
batch than with the tree waits, so that its sibling populates the tree first.

Readings of the pages where they leave a step open:

* a wave of requests is processed as: extend batches -> ``decode_steps`` decode
  steps over the whole wave -> finish of every request, decode and finish in
  the order the requests were served;
* before every extend batch the requests still waiting are ordered by the
  scheduling policy (``oracle/scheduler.py``; first come, first served keeps
  arrival order); taking them in that order, request ``j`` joins the batch
  unless its common prefix with some member exceeds its (side-effect free)
  tree match, and the batch then runs;
* a batch runs as: for each member in order ``match_prefix`` on its prompt
  minus the last token (the last prompt token is always recomputed, so every
  request has at least one query) and ``inc_lock_ref``; then one allocation of
  all new tokens, handed out in member order; then extend; then for each member
  ``insert(prompt)``, lock the prompt's node and unlock the matched node;
* a decode step allocates one slot per request (in order), stores the token's
  K/V there and attends over the request's context including that token; decode
  tokens stay outside the tree until finish;
* when a prompt's insert finds more of it cached than its match (identical
  prompts in consecutive batches), the request's own slots for that part are
  freed and its row takes the tree's slots, which hold the same K/V;
* finish is ``insert(prompt + outputs)`` then unlock of the prompt's node; slots
  of any part that another request had already inserted are freed;
* with a host tier (``oracle/hicache.py``): before a batch matches and locks,
  each member in order matches across both tiers and brings a prefix that is
  resident on the host only back to the device; after a wave's finishes,
  each finished sequence's path is written through to the host.

With pages of more than one slot (keys page-aligned, "SGLang: the tree, and
the language nobody remembers", section "A tree, not a map"), the readings
are the same with every length counted in whole pages:

* the in-batch rule compares the common prefix rounded down to whole pages
  with the (page-aligned) tree match;
* a batch takes, in member order, ``ceil(new tokens / page_size)`` pages per
  member from one allocation, and a member's new tokens fill its pages in
  order (a request never shares a page with another);
* only the whole pages of a prompt are inserted; its last, partly filled page
  stays private to the request;
* a decode token whose position starts a page takes a new page (one
  allocation per step for all requests that need one, in request order), any
  other takes the next slot of the request's last page;
* at finish the whole pages of prompt + outputs are inserted; the request
  frees its pages that another request had already inserted and the partly
  filled page past the last whole one.

Parity: pinned by ``tests/test_oracle_pins.py`` (12,960 / 6,660 / 3,060 prefill
counts of the nested example; 2,800 of 3,000 reused at agent step 5).
"""

from . import scheduler
from .hicache import TwoTierRadixCache
from .radix_cache import NoSpace, RadixCache, common_prefix_length


class Trace:
    """Everything the bookkeeping decides, for bit-exact comparison."""

    def __init__(self):
        self.batches = []        # per extend batch: list of (rid, prefix_len, row)
        self.decode_steps = []   # per decode step: list of (rid, slot)
        self.finishes = []       # per finish: (rid, already_cached)
        self.prefilled = 0
        self.eviction_log = []
        self.stats = {}
        self.loads = []          # per load from the host tier: (rid, host slots, device slots)
        self.backups = []        # per finish with a host tier: (rid, device slots, host slots)
        self.host_eviction_log = []

    def as_tuple(self):
        return (
            [[(rid, m, tuple(row)) for rid, m, row in b] for b in self.batches],
            [list(s) for s in self.decode_steps],
            list(self.finishes),
            self.prefilled,
            list(self.eviction_log),
            [(rid, tuple(h), tuple(d)) for rid, h, d in self.loads],
            [(rid, tuple(d), tuple(h)) for rid, d, h in self.backups],
            list(self.host_eviction_log),
        )


def next_batch(cache, wave_prompts, ordered):
    """The extend batch at the head of ``ordered`` (positions into
    ``wave_prompts``): requests join in order until one shares more (in whole
    pages) with a member than its own tree match."""
    batch = []
    for j in ordered:
        prompt = wave_prompts[j]
        m = cache.match_length(prompt[:len(prompt) - 1])
        if batch and any(cache.aligned(common_prefix_length(prompt, wave_prompts[i])) > m
                         for i in batch):
            break
        batch.append(j)
    return batch


def plan_batches(cache, wave_prompts, policy="fcfs"):
    """Yield lists of positions into ``wave_prompts`` forming extend batches.

    Lazily: a batch is yielded when it is formed, and the caller runs and
    inserts it before the waiting requests are ordered again and the next
    batch is formed.
    """
    pending = list(range(len(wave_prompts)))
    while pending:
        pos = scheduler.order(cache, [wave_prompts[j] for j in pending], policy)
        batch = next_batch(cache, wave_prompts, [pending[k] for k in pos])
        yield batch
        taken = set(batch)
        pending = [j for j in pending if j not in taken]


def run_bookkeeping(waves, num_slots, decode_steps, on_extend=None,
                    on_decode=None, page_size=1, policy="fcfs", host_slots=0):
    """Run the request flow over a fresh oracle cache.

    waves: list of waves; a wave is a list of ``(rid, prompt, outputs)`` with
    ``outputs`` holding ``decode_steps`` token ids (may be empty when
    ``decode_steps == 0``).  ``on_extend(batch_records)`` and
    ``on_decode(step, rows)`` are optional callbacks for attention checks.
    Returns ``(trace, cache)``.
    """
    tiered = host_slots > 0
    cache = (TwoTierRadixCache(num_slots, host_slots, page_size) if tiered
             else RadixCache(num_slots, page_size))
    ps = page_size
    trace = Trace()
    for wave in waves:
        prompts = [list(p) for _, p, _ in wave]
        rows = {}
        prompt_nodes = {}
        served = []
        for batch in plan_batches(cache, prompts, policy):
            served += batch
            matched = []
            if tiered:
                # a prefix resident on the host only comes back to the device
                # instead of being prefilled: members in order, before the
                # batch matches and locks
                for j in batch:
                    _, _, host_len, host_node = cache.match_prefix_tiers(
                        prompts[j][:len(prompts[j]) - 1])
                    if host_len:
                        try:
                            hs, ds = cache.load_onboard(host_node)
                        except NoSpace:          # no device room: prefilled instead
                            continue
                        trace.loads.append((wave[j][0], hs, ds))
            for j in batch:
                rid, prompt, _ = wave[j]
                slots, node = cache.match_prefix(prompts[j][:len(prompts[j]) - 1])
                cache.inc_lock_ref(node)
                matched.append((j, slots, node))
            pages_of = [-(-(len(prompts[j]) - len(s)) // ps) for j, s, _ in matched]
            new_pages = cache.alloc_pages(sum(pages_of))
            records = []
            pos = 0
            for (j, slots, node), n_pages in zip(matched, pages_of):
                rid = wave[j][0]
                n_new = len(prompts[j]) - len(slots)
                row = list(slots) + cache.page_slots(new_pages[pos:pos + n_pages], n_new)
                pos += n_pages
                rows[rid] = row
                records.append((rid, len(slots), list(row)))
                trace.prefilled += n_new
            trace.batches.append(records)
            if on_extend is not None:
                on_extend(records)
            for (j, slots, node), (rid, m, row) in zip(matched, records):
                already, node2 = cache.insert(prompts[j], rows[rid])
                if already > m:
                    tree = cache.lookup_slots(prompts[j])[m:already]
                    cache.free(rows[rid][m:already])
                    rows[rid][m:already] = tree
                cache.inc_lock_ref(node2)
                cache.dec_lock_ref(node)
                prompt_nodes[rid] = node2
        wave = [wave[j] for j in served]
        for step in range(decode_steps):
            need = [len(rows[rid]) % ps == 0 for rid, _, _ in wave]
            pages = cache.alloc_pages(sum(need))
            slots = []
            for (rid, _, _), starts_page in zip(wave, need):
                slots.append(pages.pop(0) * ps if starts_page else rows[rid][-1] + 1)
            step_rec = []
            for (rid, _, _), s in zip(wave, slots):
                rows[rid].append(s)
                step_rec.append((rid, s))
            trace.decode_steps.append(step_rec)
            if on_decode is not None:
                on_decode(step, {rid: list(rows[rid]) for rid, _, _ in wave})
        finished = []
        for rid, prompt, outputs in wave:
            full = list(prompt) + list(outputs[:decode_steps])
            already, full_node = cache.insert(full, rows[rid])
            finished.append((rid, full_node))
            if already > cache.aligned(len(prompt)):
                cache.free(rows[rid][cache.aligned(len(prompt)):already])
            if cache.aligned(len(full)) < len(full):      # the partly filled last page
                cache.free(rows[rid][cache.aligned(len(full)):])
            trace.finishes.append((rid, already))
            cache.dec_lock_ref(prompt_nodes[rid])
        if tiered:
            # write-through: every finished sequence's path is backed up to
            # the host tier, in order, each committed at once (the copy is
            # stream-ordered before any later load of it); a backup the host
            # tier cannot hold is skipped
            for rid, full_node in finished:
                try:
                    ticket, ds, hs = cache.write_through(full_node)
                except NoSpace:
                    ticket, ds, hs = 0, [], []
                if ticket:
                    cache.commit_write_through(ticket, True)
                trace.backups.append((rid, ds, hs))
    trace.eviction_log = list(cache.eviction_log)
    if tiered:
        trace.host_eviction_log = list(cache.host_eviction_log)
    trace.stats = {
        "cached": cache.cached_size(),
        "evictable": cache.evictable_size_,
        "protected": cache.protected_size_,
        "free": len(cache.free_slots),
        "num_nodes": cache.num_nodes(),
    }
    return trace, cache
