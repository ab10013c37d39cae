"""Oracle cache-aware scheduling of a waiting queue.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Source: "SGLang: the tree, and the language nobody remembers", section "The
scheduler is where the cache is won or lost":

* longest prefix match (LPM): the waiting queue is sorted so that the request
  with the most of its prompt already in the tree goes first;
* a request whose match against the tree is thin (at most 32 tokens) is also
  matched against a second, simulated radix tree built over the waiting
  queue itself; if it shares at least 32 tokens with a request already in
  that tree it is deprioritised (sorted to the very back) so that its sibling
  runs first and populates the tree, otherwise it is inserted into the queue
  tree;
* LPM turns itself off (first come, first served) when more than 128 requests
  wait;
* DFS weight: every tree node is weighted by how many waiting requests hang
  off it, and the queue is emitted in a weighted depth-first order, so a
  subtree is drained before it can be evicted.

Readings where the page is silent:

* a request's match (against the tree and against the queue tree) is taken on
  its prompt without the last token, the same match its admission takes (the
  last prompt token is always recomputed), in whole pages;
* the queue tree holds whole prompts; its match is the longest common prefix
  with any prompt in it, limited to that prompt's whole pages and rounded
  down to whole pages -- what a radix tree over those prompts returns;
* sorting is stable: requests with equal keys keep their queue order;
* a request hangs off the deepest node whose whole root path its prompt
  (minus the last token) matches; the depth-first order emits the requests
  hanging off a node (in queue order) before visiting its children, heavier
  children first, children of equal weight in the queue order of their
  earliest waiting request.

Parity: pinned by ``tests/test_oracle_pins.py`` (the served order and the
126 / 46 prefilled tokens printed by the cache-aware scheduling toy of "SGLang:
Structured LLM Programs for Efficient Inference", section "Practice: try it
yourself", the thresholds and the queue-length switch as stated, and
hand-worked depth-first orders).  The 14,688 / 5,472 figures of the page's
interactive queue simulation are parity unpinned: the simulation's inputs are
not on the page.
"""

from .radix_cache import common_prefix_length

IN_BATCH_CHECK_THRESHOLD = 32
IN_BATCH_DEPRIORITIZE_THRESHOLD = 32
LPM_QUEUE_LIMIT = 128

POLICIES = ("fcfs", "lpm", "dfs-weight")


def _key(prompt):
    return list(prompt[:len(prompt) - 1])


def queue_tree_match(cache, tokens, queued):
    """Match of ``tokens`` in a radix tree holding the prompts ``queued``."""
    best = 0
    for q in queued:
        c = common_prefix_length(tokens, q)
        best = max(best, min(c, cache.aligned(len(q))))
    return cache.aligned(best)


def lpm_order(cache, prompts):
    """Queue positions in LPM order (FCFS above the queue limit)."""
    n = len(prompts)
    if n > LPM_QUEUE_LIMIT:
        return list(range(n))
    keys = []
    queued = []
    for i, p in enumerate(prompts):
        m = cache.match_length(_key(p))
        deprioritised = False
        if m <= IN_BATCH_CHECK_THRESHOLD:
            if queue_tree_match(cache, _key(p), queued) >= IN_BATCH_DEPRIORITIZE_THRESHOLD:
                deprioritised = True
            else:
                queued.append(list(p))
        keys.append((float("inf") if deprioritised else -m, i))
    return [i for _, i in sorted(keys)]


def hanging_node(cache, tokens):
    """The deepest node whose whole root path ``tokens`` matches."""
    node = cache.root
    pos = 0
    tokens = tokens[:cache.aligned(len(tokens))]
    while pos < len(tokens):
        child = node.children.get(cache.child_key(tokens, pos))
        if child is None:
            break
        k = common_prefix_length(child.key, tokens[pos:])
        if k < len(child.key):
            break
        pos += k
        node = child
    return node


def dfs_weight_order(cache, prompts):
    """Queue positions in weighted depth-first order of the tree."""
    at = {}
    for i, p in enumerate(prompts):
        at.setdefault(hanging_node(cache, _key(p)).id, []).append(i)
    weight = {}
    first = {}

    def weigh(node):
        w = len(at.get(node.id, []))
        f = min(at.get(node.id, [len(prompts)]))
        for c in node.children.values():
            cw, cf = weigh(c)
            w += cw
            f = min(f, cf)
        weight[node.id] = w
        first[node.id] = f
        return w, f

    weigh(cache.root)
    out = []

    def visit(node):
        out.extend(at.get(node.id, []))
        kids = [c for c in node.children.values() if weight[c.id] > 0]
        kids.sort(key=lambda c: (-weight[c.id], first[c.id]))
        for c in kids:
            visit(c)

    visit(cache.root)
    return out


def order(cache, prompts, policy):
    """Queue positions of ``prompts`` in the order ``policy`` serves them."""
    if policy == "fcfs":
        return list(range(len(prompts)))
    if policy == "lpm":
        return lpm_order(cache, prompts)
    if policy == "dfs-weight":
        return dfs_weight_order(cache, prompts)
    raise ValueError(f"unknown policy {policy}")
