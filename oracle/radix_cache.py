"""Oracle radix cache over a token-granular KV slot pool.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``): plain Python, no
speed tricks, each step written in the order the pages describe it.

Sources (page title, section):

* "SGLang: the tree, and the language nobody remembers", section "A tree, not
  a map": a ``TreeNode`` carries ``key`` (a token run), ``value`` (its KV slot
  indices), ``children``, ``parent``, ``lock_ref``, ``last_access_time`` and
  ``priority``; ``inc_lock_ref`` moves a node's length from the evictable to
  the protected count when its ``lock_ref`` goes from 0 to 1; eviction heapifies
  the candidates, pops them, and pushes a parent once it is childless and
  unlocked (cascading); a node splits where a request diverges; children are
  keyed on the first token when ``page_size == 1``.
* "SGLang" (bibekananda.in), sections "One tree for everybody" and "Eviction on
  a tree": a request walks from the root as far as its tokens match; the
  divergent part becomes a new branch; eviction works from the leaves inward.
* "SGLang: Structured LLM Programs for Efficient Inference", sections "How
  RadixAttention reuses past work" (match, lock, prefill the rest, insert,
  unlock) and "Worked example, step by step" (a node is evicted whole; locked
  nodes are never candidates; if nothing can be evicted the request waits).

* same page, same section: keys are page-aligned -- every key is truncated to
  a multiple of ``page_size`` and a match is rounded down to one -- and a
  node's children are keyed on the first token at ``page_size == 1`` and on
  the tuple of the first ``page_size`` tokens otherwise.

Readings where the pages are silent:

* the pool is cut into pages of ``page_size`` consecutive slots; page 0 (slots
  ``0 .. page_size-1``) is a pad page that is never handed out, and the
  allocator hands out whole pages, so a request's positions ``[k*page_size,
  (k+1)*page_size)`` always lie in one page, in slot order (at
  ``page_size == 1`` a page is a slot);
* a match that ends inside an edge splits that edge so the returned node covers
  exactly the matched prefix; the new upper node takes a fresh id and inherits
  the lower node's ``lock_ref`` and ``last_access_time``;
* ``last_access_time`` is a logical clock that advances once per ``match_prefix``
  or ``insert`` call and is written on every node of the touched path;
* the eviction key is ``(priority, last_access_time, node id)`` with
  ``priority == 0`` everywhere, i.e. least recently used, ties by creation order;
* the allocator is a FIFO free list of pages initialised ``1 .. N/page_size -
  1``; freed pages join the tail in the order given (a page once, at the first
  of its slots);
* an allocation that cannot be met after evicting everything evictable fails
  with ``NoSpace``; nodes evicted during that attempt stay evicted.

Parity: pinned by ``tests/test_oracle_pins.py`` (the toy trie's printed reuse
counts, the nested example's prefill counts, the agent step-5 reuse, the worked
eviction example, brute-force longest-common-prefix on tiny alphabets, and the
structural invariants of locking and leaf-inward eviction).
"""

from collections import deque
import heapq


class NoSpace(Exception):
    """Raised when an allocation cannot be satisfied even after eviction."""


class StateError(Exception):
    """Raised on lock misuse (unlock below zero, unknown node)."""


class TreeNode:
    def __init__(self, node_id, key, value, parent):
        self.id = node_id
        self.key = list(key)          # token run on the edge into this node
        self.value = list(value)      # KV slot of each token in ``key``
        self.children = {}            # first token of child key -> child
        self.parent = parent
        self.lock_ref = 0
        self.last_access_time = 0
        self.priority = 0
        self.evicted = False


def common_prefix_length(a, b):
    """Number of leading positions where sequences ``a`` and ``b`` agree."""
    n = 0
    limit = min(len(a), len(b))
    while n < limit and a[n] == b[n]:
        n += 1
    return n


class RadixCache:
    """Radix tree over token prefixes plus the FIFO page allocator."""

    def __init__(self, num_slots, page_size=1):
        if page_size < 1 or num_slots < page_size or num_slots % page_size:
            raise ValueError("num_slots must be a positive multiple of page_size")
        self.num_slots = num_slots
        self.page_size = page_size
        # page 0 is the pad page
        self.free_pages = deque(range(1, num_slots // page_size))
        self.root = TreeNode(0, [], [], None)
        self.next_id = 1
        self.clock = 0
        self.evictable_size_ = 0
        self.protected_size_ = 0
        self.nodes = {0: self.root}
        self.eviction_log = []        # (node id, number of tokens) in order

    # ------------------------------------------------------------- pages
    def aligned(self, n):
        """``n`` rounded down to a whole number of pages."""
        return n - n % self.page_size

    def child_key(self, tokens, pos):
        """Key of the child that starts at ``tokens[pos]``: the token itself at
        page size 1, else the tuple of the page's tokens."""
        if self.page_size == 1:
            return tokens[pos]
        return tuple(tokens[pos:pos + self.page_size])

    @property
    def free_slots(self):
        """Slots of the free pages, in free-list order."""
        ps = self.page_size
        return [p * ps + j for p in self.free_pages for j in range(ps)]

    # ------------------------------------------------------------------ walk
    def _new_node(self, key, value, parent):
        node = TreeNode(self.next_id, key, value, parent)
        self.next_id += 1
        self.nodes[node.id] = node
        return node

    def _split(self, node, k):
        """Split ``node``'s edge after its first ``k`` tokens.

        Returns the new upper node, which covers ``key[:k]``; ``node`` keeps
        the remainder and becomes its only child.
        """
        assert 0 < k < len(node.key)
        parent = node.parent
        upper = self._new_node(node.key[:k], node.value[:k], parent)
        upper.lock_ref = node.lock_ref
        upper.last_access_time = node.last_access_time
        parent.children[self.child_key(node.key, 0)] = upper
        node.key = node.key[k:]
        node.value = node.value[k:]
        node.parent = upper
        upper.children[self.child_key(node.key, 0)] = node
        return upper

    def match_length(self, tokens):
        """Longest cached prefix of ``tokens`` (whole pages), no side effects."""
        tokens = tokens[:self.aligned(len(tokens))]
        node = self.root
        pos = 0
        while pos < len(tokens):
            child = node.children.get(self.child_key(tokens, pos))
            if child is None:
                break
            k = self.aligned(common_prefix_length(child.key, tokens[pos:]))
            pos += k
            if k < len(child.key):
                break
            node = child
        return pos

    def lookup_slots(self, tokens):
        """Slots of the longest cached prefix of ``tokens``, no side effects."""
        tokens = tokens[:self.aligned(len(tokens))]
        node = self.root
        pos = 0
        out = []
        while pos < len(tokens):
            child = node.children.get(self.child_key(tokens, pos))
            if child is None:
                break
            k = self.aligned(common_prefix_length(child.key, tokens[pos:]))
            out.extend(child.value[:k])
            pos += k
            if k < len(child.key):
                break
            node = child
        return out

    def match_prefix(self, tokens):
        """Walk from the root as far as ``tokens`` match.

        Returns ``(slots, node)``: the KV slots of the matched prefix, in
        order, and the node whose path from the root is exactly that prefix
        (the root when nothing matched).  Only whole pages match: ``tokens``
        is truncated to whole pages and the match inside an edge rounded down
        to one.  A match ending inside an edge splits that edge.  Every node
        on the matched path is touched.
        """
        self.clock += 1
        tokens = tokens[:self.aligned(len(tokens))]
        node = self.root
        slots = []
        pos = 0
        path = []
        while pos < len(tokens):
            child = node.children.get(self.child_key(tokens, pos))
            if child is None:
                break
            k = self.aligned(common_prefix_length(child.key, tokens[pos:]))
            if k < len(child.key):
                child = self._split(child, k)
            slots.extend(child.value)
            pos += k
            path.append(child)
            node = child
        for n in path:
            n.last_access_time = self.clock
        return slots, node

    def insert(self, tokens, slots):
        """Insert ``tokens`` with their KV ``slots``.

        Only the whole pages of ``tokens`` are inserted (the key is
        truncated to a multiple of the page size).  Walks (and splits) as
        ``match_prefix`` does; the part not yet in the tree becomes one new
        leaf holding the matching part of ``slots``.  Returns ``(already,
        node)``: how many leading tokens were already cached (the caller frees
        its own slots for that part beyond what it had locked) and the node
        that ends exactly at the truncated length.
        """
        if len(tokens) != len(slots):
            raise ValueError("tokens and slots differ in length")
        n = self.aligned(len(tokens))
        tokens, slots = list(tokens[:n]), list(slots[:n])
        self.clock += 1
        node = self.root
        pos = 0
        path = []
        while pos < len(tokens):
            child = node.children.get(self.child_key(tokens, pos))
            if child is None:
                break
            k = self.aligned(common_prefix_length(child.key, tokens[pos:]))
            if k < len(child.key):
                child = self._split(child, k)
            pos += k
            path.append(child)
            node = child
        already = pos
        if pos < len(tokens):
            leaf = self._new_node(tokens[pos:], slots[pos:], node)
            node.children[self.child_key(tokens, pos)] = leaf
            self.evictable_size_ += len(leaf.key)
            path.append(leaf)
            node = leaf
        for n in path:
            n.last_access_time = self.clock
        return already, node

    # ------------------------------------------------------------- locking
    def inc_lock_ref(self, node):
        """Protect ``node`` and its ancestors (the root excluded)."""
        self._check_live(node)
        while node is not self.root:
            if node.lock_ref == 0:
                self.evictable_size_ -= len(node.key)
                self.protected_size_ += len(node.key)
            node.lock_ref += 1
            node = node.parent

    def dec_lock_ref(self, node):
        """Release one protection of ``node`` and its ancestors."""
        self._check_live(node)
        walk = node
        while walk is not self.root:
            if walk.lock_ref <= 0:
                raise StateError("unlock below zero")
            walk = walk.parent
        while node is not self.root:
            if node.lock_ref == 1:
                self.evictable_size_ += len(node.key)
                self.protected_size_ -= len(node.key)
            node.lock_ref -= 1
            node = node.parent

    def _check_live(self, node):
        if node.evicted or self.nodes.get(node.id) is not node:
            raise StateError("node is not in the tree")

    # ------------------------------------------------------------ eviction
    def _leaves(self):
        out = []
        stack = [self.root]
        while stack:
            n = stack.pop()
            if n is not self.root and not n.children:
                out.append(n)
            stack.extend(n.children.values())
        return out

    def evict(self, num_tokens):
        """Free at least ``num_tokens`` slots by evicting unlocked leaves.

        Candidates are the unlocked leaves, ordered by ``(priority,
        last_access_time, id)``.  The smallest is evicted whole, its pages go
        to the tail of the free list in stored order, and its parent becomes a
        candidate once childless and unlocked.  Stops when enough is freed or
        no candidate is left; returns the number of slots freed.
        """
        heap = [(n.priority, n.last_access_time, n.id, n)
                for n in self._leaves() if n.lock_ref == 0]
        heapq.heapify(heap)
        freed = 0
        while freed < num_tokens and heap:
            _, _, _, victim = heapq.heappop(heap)
            parent = victim.parent
            del parent.children[self.child_key(victim.key, 0)]
            self.free_pages.extend(s // self.page_size
                                   for s in victim.value[::self.page_size])
            freed += len(victim.value)
            self.evictable_size_ -= len(victim.key)
            self.eviction_log.append((victim.id, len(victim.key)))
            victim.evicted = True
            del self.nodes[victim.id]
            if (parent is not self.root and not parent.children
                    and parent.lock_ref == 0):
                heapq.heappush(heap, (parent.priority, parent.last_access_time,
                                      parent.id, parent))
        return freed

    # ----------------------------------------------------------- allocator
    def alloc_pages(self, n):
        """Take ``n`` pages from the head of the free list, evicting the
        shortfall first (in slots) if too few are free."""
        if n < 0:
            raise ValueError("negative allocation")
        if len(self.free_pages) < n:
            self.evict((n - len(self.free_pages)) * self.page_size)
        if len(self.free_pages) < n:
            raise NoSpace(n)
        return [self.free_pages.popleft() for _ in range(n)]

    def page_slots(self, pages, k):
        """The first ``k`` slots of ``pages``, page after page."""
        ps = self.page_size
        return [p * ps + j for p in pages for j in range(ps)][:k]

    def alloc(self, k):
        """``k`` slots: the first ``k`` slots of the ``ceil(k / page_size)``
        pages taken from the head of the free list (evicting if short)."""
        ps = self.page_size
        return self.page_slots(self.alloc_pages(-(-k // ps)), k)

    def free(self, slots):
        """Return the pages the given slots lie in (each once, in order)."""
        seen, order = set(), []
        for s in slots:
            p = s // self.page_size
            if p not in seen:
                seen.add(p)
                order.append(p)
        self.free_pages.extend(order)

    # --------------------------------------------------------------- stats
    def cached_size(self):
        total = 0
        stack = [self.root]
        while stack:
            n = stack.pop()
            total += len(n.key)
            stack.extend(n.children.values())
        return total

    def num_nodes(self):
        return len(self.nodes) - 1
