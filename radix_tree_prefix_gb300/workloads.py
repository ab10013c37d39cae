"""Seeded synthetic workloads: token ids, request structure and Q/K/V values.

This module only generates inputs.  It holds none of the cache or attention
arithmetic, and both the CUDA path and the oracle read the same arrays it
produces.

Every prompt is a concatenation of *segments* (runs of token ids).  Segments
are shared between requests exactly where the workload shares text, so a
shared segment has identical token ids, and identical Q/K/V, in every request
that contains it.  This realises the property the pages rest on: the KV of a
token depends only on that token and the tokens before it ("SGLang:
Structured LLM Programs for Efficient Inference", section "A quick recap of
how an LLM generates text").  To keep that property exact, the first token of
every segment is drawn distinct from the first token of every other segment,
so two different segments that follow the same predecessor never share a tree
edge by accident.

Token ids are uniform in [0, 32000) from ``numpy.random.Generator(PCG64)``.
Q/K/V values are standard normal, drawn with a seeded ``torch.Generator`` on
the device they are used on, and rounded to bf16 (round to nearest even).  Each
distinct token position of the workload owns one row of a *store*; a request's
tokens index into the store.

The five workloads (all sizes as stated by the workload descriptions):

1. ``nested_share``   8 requests = 900 shared + 600-token document (4 requests
                      each) + 120 unique; Hq 8 / Hkv 2, d 128, 1 layer; extend
                      only.  Expect 3,060 prefilled tokens.
2. ``agent_loop``     40 calls = 3,000 shared + U[150, 250] unique; 64 decode
                      steps; Hq 32 / Hkv 8, d 128, 1 layer; pool never evicts.
3. ``multi_turn_chat`` 256 sessions x 8 turns over a 2,000-token system prompt,
                      200 new tokens + 32 decode tokens per turn; Hq 16 / Hkv 4,
                      d 256, 16 layers; one wave per turn, decode batch 256.
4. ``fork_tree``      branching 5, depth 4, 512 tokens per level (625 leaves);
                      16 decode steps; Hq 32 / Hkv 8, d 128, 1 layer; pool holds
                      60% of the distinct tokens; one wave per level-1 subtree.
5. ``long_shared``    64 requests = 32,768 shared + 1,024 unique; 128 decode
                      steps; Hq 64 / Hkv 8, d 128, 1 layer.
"""

from dataclasses import dataclass, field

import numpy as np

VOCAB = 32000
BASE_SEED = 0


@dataclass
class Request:
    rid: int
    prompt_segs: tuple
    output_seg: int = -1


@dataclass
class Workload:
    name: str
    num_layers: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    num_slots: int
    decode_steps: int
    seg_tokens: list = field(default_factory=list)
    waves: list = field(default_factory=list)
    seed: int = BASE_SEED
    page_size: int = 1

    def __post_init__(self):
        self._finalise()

    def _finalise(self):
        lens = [len(t) for t in self.seg_tokens]
        self.seg_offset = np.zeros(len(lens) + 1, dtype=np.int64)
        np.cumsum(lens, out=self.seg_offset[1:])
        self.n_store = int(self.seg_offset[-1])
        self.requests = {r.rid: r for w in self.waves for r in w}

    # ------------------------------------------------------------ tokens
    def prompt_tokens(self, req):
        return np.concatenate([self.seg_tokens[s] for s in req.prompt_segs])

    def prompt_store_index(self, req):
        return np.concatenate([
            np.arange(self.seg_offset[s], self.seg_offset[s + 1])
            for s in req.prompt_segs])

    def output_tokens(self, req):
        if req.output_seg < 0:
            return np.zeros(0, dtype=np.int32)
        return self.seg_tokens[req.output_seg]

    def output_store_index(self, req):
        if req.output_seg < 0:
            return np.zeros(0, dtype=np.int64)
        s = req.output_seg
        return np.arange(self.seg_offset[s], self.seg_offset[s + 1])

    def oracle_waves(self):
        """Waves as lists of ``(rid, prompt list, outputs list)``."""
        return [[(r.rid, self.prompt_tokens(r).tolist(),
                  self.output_tokens(r).tolist()) for r in wave]
                for wave in self.waves]

    @property
    def group(self):
        return self.num_q_heads // self.num_kv_heads

    def distinct_tokens(self):
        return self.n_store

    def describe(self):
        return {
            "workload": self.name,
            "requests": len(self.requests),
            "waves": len(self.waves),
            "layers": self.num_layers,
            "q_heads": self.num_q_heads,
            "kv_heads": self.num_kv_heads,
            "head_dim": self.head_dim,
            "decode_steps": self.decode_steps,
            "pool_slots": self.num_slots,
            "distinct_tokens": self.n_store,
            "page_size": self.page_size,
        }


class _Segments:
    """Draws segments of token ids with globally distinct first tokens."""

    def __init__(self, seed):
        self.rng = np.random.Generator(np.random.PCG64(seed))
        self.tokens = []
        self.first = set()

    def new(self, length):
        t = self.rng.integers(0, VOCAB, size=length, dtype=np.int64).astype(np.int32)
        if length:
            while int(t[0]) in self.first:
                t[0] = int(self.rng.integers(0, VOCAB))
            self.first.add(int(t[0]))
        self.tokens.append(t)
        return len(self.tokens) - 1


# ---------------------------------------------------------------- configs
def nested_share(seed=BASE_SEED, instr=900, doc=600, unique=120, per_doc=4,
                 n_docs=2):
    s = _Segments(seed * 1000 + 1)
    i_seg = s.new(instr)
    docs = [s.new(doc) for _ in range(n_docs)]
    wave = []
    rid = 0
    for d in docs:
        for _ in range(per_doc):
            wave.append(Request(rid, (i_seg, d, s.new(unique))))
            rid += 1
    distinct = instr + n_docs * doc + n_docs * per_doc * unique
    return Workload("nested_share", 1, 8, 2, 128, distinct + 1 + 64, 0,
                    s.tokens, [wave], seed)


def agent_loop(seed=BASE_SEED, calls=40, preamble=3000, lo=150, hi=250,
               decode_steps=64, q_heads=32, kv_heads=8, head_dim=128):
    s = _Segments(seed * 1000 + 2)
    p = s.new(preamble)
    lens = s.rng.integers(lo, hi + 1, size=calls)
    wave = []
    for rid in range(calls):
        u = s.new(int(lens[rid]))
        o = s.new(decode_steps) if decode_steps else -1
        wave.append(Request(rid, (p, u), o))
    distinct = preamble + int(lens.sum()) + calls * decode_steps
    return Workload("agent_loop", 1, q_heads, kv_heads, head_dim, distinct + 1,
                    decode_steps, s.tokens, [wave], seed)


def multi_turn_chat(seed=BASE_SEED, sessions=256, turns=8, system=2000,
                    user=200, decode_steps=32, layers=16, q_heads=16,
                    kv_heads=4, head_dim=256):
    s = _Segments(seed * 1000 + 3)
    sys_seg = s.new(system)
    history = [[sys_seg] for _ in range(sessions)]
    waves = []
    rid = 0
    for _ in range(turns):
        wave = []
        for sess in range(sessions):
            u = s.new(user)
            o = s.new(decode_steps)
            wave.append(Request(rid, tuple(history[sess] + [u]), o))
            history[sess] += [u, o]
            rid += 1
        waves.append(wave)
    distinct = system + sessions * turns * (user + decode_steps)
    return Workload("multi_turn_chat", layers, q_heads, kv_heads, head_dim,
                    distinct + 1, decode_steps, s.tokens, waves, seed)


def multi_turn_chat_small(seed=BASE_SEED):
    """multi_turn_chat cut to 32 sessions x 2 turns: the same head_dim-256
    kernel shapes per launch with a few GB on the device, for profiler
    captures of single launches."""
    wl = multi_turn_chat(seed, sessions=32, turns=2)
    wl.name = "multi_turn_chat_small"
    return wl


def fork_tree(seed=BASE_SEED, branching=5, depth=4, level_tokens=512,
              decode_steps=16, pool_fraction=0.6, q_heads=32, kv_heads=8,
              head_dim=128):
    s = _Segments(seed * 1000 + 4)

    def grow(prefix, level):
        if level == depth:
            return [prefix]
        leaves = []
        for _ in range(branching):
            leaves += grow(prefix + [s.new(level_tokens)], level + 1)
        return leaves

    waves = []
    rid = 0
    n_nodes = 0
    for _ in range(branching):
        top = s.new(level_tokens)
        leaves = grow([top], 1)
        wave = []
        for leaf in leaves:
            o = s.new(decode_steps) if decode_steps else -1
            wave.append(Request(rid, tuple(leaf), o))
            rid += 1
        waves.append(wave)
    n_nodes = sum(branching ** k for k in range(1, depth + 1))
    distinct_prompt = n_nodes * level_tokens
    usable = int(pool_fraction * distinct_prompt)
    return Workload("fork_tree", 1, q_heads, kv_heads, head_dim, usable + 1,
                    decode_steps, s.tokens, waves, seed)


def long_shared(seed=BASE_SEED, batch=64, prefix=32768, unique=1024,
                decode_steps=128, q_heads=64, kv_heads=8, head_dim=128):
    s = _Segments(seed * 1000 + 5)
    p = s.new(prefix)
    wave = []
    for rid in range(batch):
        u = s.new(unique)
        o = s.new(decode_steps) if decode_steps else -1
        wave.append(Request(rid, (p, u), o))
    distinct = prefix + batch * (unique + decode_steps)
    return Workload("long_shared", 1, q_heads, kv_heads, head_dim, distinct + 1,
                    decode_steps, s.tokens, [wave], seed)


def with_pages(wl, page_size):
    """The same workload over a pool cut into pages of `page_size` slots:
    every request may leave part of a page unused (its last prompt page and
    its last decode page), so the pool grows by two pages per request of the
    largest wave and rounds up to whole pages."""
    extra = 2 * max(len(w) for w in wl.waves) * page_size
    wl.num_slots = -(-(wl.num_slots + extra) // page_size) * page_size
    wl.page_size = page_size
    wl.name = f"{wl.name}_p{page_size}"
    return wl


def shard(wl, rank, world):
    """Rank `rank`'s share of the workload among `world` replicas, each with
    its own cache and pool (no data exchange between them), routed so that
    requests that share a subtree stay on one replica: fork_tree's waves (one
    level-1 subtree each) go round-robin by wave; every other workload's
    requests go round-robin by their position in the wave (a chat session, an
    agent call, a long-context request keeps its replica from turn to turn).
    The pool keeps its size; the segment tables are shared."""
    if world <= 1:
        return wl
    if wl.name.startswith("fork_tree") and len(wl.waves) >= world:
        waves = [w for i, w in enumerate(wl.waves) if i % world == rank]
    else:
        waves = [[r for i, r in enumerate(w) if i % world == rank] for w in wl.waves]
        waves = [w for w in waves if w]
    out = Workload(wl.name, wl.num_layers, wl.num_q_heads, wl.num_kv_heads, wl.head_dim,
                   wl.num_slots, wl.decode_steps, wl.seg_tokens, waves, wl.seed, wl.page_size)
    return out


WORKLOADS = {
    "nested_share": nested_share,
    "agent_loop": agent_loop,
    "multi_turn_chat": multi_turn_chat,
    "multi_turn_chat_small": multi_turn_chat_small,
    "fork_tree": fork_tree,
    "long_shared": long_shared,
}


# ----------------------------------------------------------------- values
def make_values(wl, device, layers=None, kinds=("q", "k", "v")):
    """Seeded Q/K/V stores on ``device`` as bf16 torch tensors.

    Returns ``{kind: {layer: tensor}}`` with ``k``/``v`` of shape
    ``[n_store, Hkv, d]`` and ``q`` of shape ``[n_store, Hq, d]``.
    """
    import torch

    if layers is None:
        layers = range(wl.num_layers)
    out = {k: {} for k in kinds}
    for layer in layers:
        for ki, kind in enumerate(("q", "k", "v")):
            if kind not in kinds:
                continue
            heads = wl.num_q_heads if kind == "q" else wl.num_kv_heads
            g = torch.Generator(device=device)
            g.manual_seed(wl.seed * 1_000_003 + layer * 7 + ki + 11)
            t = torch.empty((wl.n_store, heads, wl.head_dim),
                            dtype=torch.bfloat16, device=device)
            chunk = max(1, (1 << 26) // (heads * wl.head_dim))
            for lo in range(0, wl.n_store, chunk):
                hi = min(wl.n_store, lo + chunk)
                t[lo:hi] = torch.randn((hi - lo, heads, wl.head_dim),
                                       generator=g, device=device,
                                       dtype=torch.float32).to(torch.bfloat16)
            out[kind][layer] = t
    return out
