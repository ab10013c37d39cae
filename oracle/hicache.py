"""Oracle two-tier (GPU + host) radix cache.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Source: "SGLang: the tree, and the language nobody remembers", section "What
the C++ tree is actually for": the C++ tree is a two-tier cache with
asynchronous transactions.  ``match_prefix`` returns the device indices it
matched, how many tokens matched on the host, and a node handle for each
tier; a node can be on the GPU, on the host, or on both, and
``is_leaf_device`` holds when no child is resident on the GPU;
``writing_through`` backs KV up to the host and hands back a ticket that a
later ``commit_writing_through(ticket, success)`` resolves; ``loading_onboard``
brings a host-resident node back to the device and returns the host indices
to copy from.

Readings where the page is silent (the single-tier rules of
``radix_cache.py`` hold unless stated):

* a node holds device slots (``value``), host slots (``host_value``) or both;
  the host tier is a second slot pool cut into the same pages, page 0 a pad
  page, with its own FIFO free list;
* the device-resident nodes form a subtree hanging from the root, and so do
  the host-resident ones: write-through backs up a whole root path, a
  load brings back a whole host-only path below the device part, and device
  eviction works leaf-inward over device residency;
* a match walks every tier; its device part is the leading run of
  device-resident nodes; the rest of the walk matched on the host only;
  ``match_length`` (the in-batch rule, scheduling) counts both tiers;
* device eviction takes unlocked device leaves (no child on the device) in
  least-recently-used order; a node also on the host only gives up its
  device slots and stays in the tree, a device-only node leaves the tree;
  the parent becomes a candidate once it has no child on the device;
* host eviction (when a backup needs host pages) takes host-only nodes
  without children, least recently used first, removing them; their
  parent becomes a candidate once childless and host-only;
* ``write_through(node)`` allocates host pages for the device-only nodes of
  the node's root path (in path order), locks the node until the commit
  (so the device slots being copied stay), and returns the copies to make
  (device slots -> host slots); committing with success makes those nodes
  resident on both tiers, with failure frees the host pages; while a backup
  of any node on the path is in flight the write-through is refused (ticket
  0), so a failed commit can never leave a host-resident node below a node
  that is not;
* ``load_onboard(node)`` allocates device pages (evicting as an allocation
  does, with the path's device part locked meanwhile) for the host-only
  nodes of the node's root path and makes them resident on both tiers; it
  returns the copies to make (host slots -> device slots), which the caller
  completes before any kernel reads those slots;
* an insert over a host-only node adopts the caller's device slots for it
  (the same tokens after the same predecessors, so the same K/V); the
  already-cached count is the device-resident part.

Parity: pinned by ``tests/test_oracle_pins.py`` (identical to the single-tier
cache while nothing is on the host; the worked eviction example with a host
tier, where the evicted branch comes back from the host instead of being
prefilled; residency and slot-conservation invariants under random
operations; a multi-turn chat under a small device pool prefilling less with
the host tier than without).
"""

from collections import deque
import heapq

from .radix_cache import NoSpace, RadixCache, StateError, common_prefix_length


class TwoTierRadixCache(RadixCache):
    def __init__(self, num_slots, host_slots, page_size=1):
        super().__init__(num_slots, page_size)
        if host_slots < 0 or host_slots % page_size:
            raise ValueError("host_slots must be a multiple of page_size")
        self.host_slots = host_slots
        self.free_host_pages = deque(range(1, host_slots // page_size)) if host_slots else deque()
        self.host_eviction_log = []
        self.pending = {}                  # ticket -> end node of the backed-up path
        self.next_ticket = 1
        self.root.host_value = []
        self.root.pending = None

    # ------------------------------------------------------------ residency
    def _new_node(self, key, value, parent):
        node = super()._new_node(key, value, parent)
        node.host_value = None
        node.pending = None                # (ticket, host slots) while backing up
        return node

    def on_gpu(self, node):
        return node is self.root or node.value is not None

    def on_host(self, node):
        return node is self.root or node.host_value is not None

    def _dev_children(self, node):
        return [c for c in node.children.values() if self.on_gpu(c)]

    def _split(self, node, k):
        parent = node.parent
        upper = self._new_node(node.key[:k], [] if node.value is None else node.value[:k],
                               parent)
        if node.value is None:
            upper.value = None
        if node.host_value is not None:
            upper.host_value = node.host_value[:k]
            node.host_value = node.host_value[k:]
        if node.pending is not None:
            upper.pending = (node.pending[0], node.pending[1][:k])
            node.pending = (node.pending[0], node.pending[1][k:])
        upper.lock_ref = node.lock_ref
        upper.last_access_time = node.last_access_time
        parent.children[self.child_key(node.key, 0)] = upper
        node.key = node.key[k:]
        if node.value is not None:
            node.value = node.value[k:]
        node.parent = upper
        upper.children[self.child_key(node.key, 0)] = node
        return upper

    def _walk(self, tokens, split=True):
        """Nodes matched along ``tokens`` (whole pages, every tier)."""
        tokens = tokens[:self.aligned(len(tokens))]
        node = self.root
        pos = 0
        path = []
        while pos < len(tokens):
            child = node.children.get(self.child_key(tokens, pos))
            if child is None:
                break
            k = self.aligned(common_prefix_length(child.key, tokens[pos:]))
            if k < len(child.key):
                if not split:
                    break
                child = self._split(child, k)
            pos += k
            path.append(child)
            node = child
        return path, pos

    # ---------------------------------------------------------------- match
    def lookup_slots(self, tokens):
        """Device slots of the longest device-resident cached prefix."""
        tokens = tokens[:self.aligned(len(tokens))]
        node = self.root
        pos = 0
        out = []
        while pos < len(tokens):
            child = node.children.get(self.child_key(tokens, pos))
            if child is None or not self.on_gpu(child):
                break
            k = self.aligned(common_prefix_length(child.key, tokens[pos:]))
            out.extend(child.value[:k])
            pos += k
            if k < len(child.key):
                break
            node = child
        return out

    def match_prefix_tiers(self, tokens):
        """Walk every tier.  Returns ``(slots, device_node, host_len,
        host_node)``: the device slots of the leading device-resident part,
        its last node, how many more tokens matched on the host only, and
        the last node matched (``device_node`` when nothing more matched)."""
        self.clock += 1
        path, _ = self._walk(tokens)
        for n in path:
            n.last_access_time = self.clock
        slots = []
        dev = self.root
        host_len = 0
        for n in path:
            if self.on_gpu(n) and host_len == 0:
                slots.extend(n.value)
                dev = n
            else:
                host_len += len(n.key)
        return slots, dev, host_len, (path[-1] if path else self.root)

    def match_prefix(self, tokens):
        slots, node, _, _ = self.match_prefix_tiers(tokens)
        return slots, node

    def insert(self, tokens, slots):
        if len(tokens) != len(slots):
            raise ValueError("tokens and slots differ in length")
        n = self.aligned(len(tokens))
        tokens, slots = list(tokens[:n]), list(slots[:n])
        self.clock += 1
        path, pos = self._walk(tokens)
        already = 0
        off = 0
        for x in path:
            if self.on_gpu(x):
                if off == already:
                    already += len(x.key)
            else:
                # host-only: adopt the caller's device slots for it
                x.value = slots[off:off + len(x.key)]
                if x.lock_ref > 0:
                    self.protected_size_ += len(x.key)
                else:
                    self.evictable_size_ += len(x.key)
            off += len(x.key)
        node = path[-1] if path else self.root
        if pos < len(tokens):
            leaf = self._new_node(tokens[pos:], slots[pos:], node)
            node.children[self.child_key(tokens, pos)] = leaf
            self.evictable_size_ += len(leaf.key)
            path.append(leaf)
            node = leaf
        for x in path:
            x.last_access_time = self.clock
        return already, node

    def inc_lock_ref(self, node):
        walk = node
        while walk is not self.root:
            if not self.on_gpu(walk):
                raise StateError("only device-resident paths are locked")
            walk = walk.parent
        super().inc_lock_ref(node)

    # ------------------------------------------------------------- eviction
    def evict(self, num_tokens):
        """Device eviction over device residency (see the module readings)."""
        heap = []
        stack = [self.root]
        while stack:
            x = stack.pop()
            if (x is not self.root and self.on_gpu(x) and not self._dev_children(x)
                    and x.lock_ref == 0):
                heap.append((x.priority, x.last_access_time, x.id, x))
            stack.extend(x.children.values())
        heapq.heapify(heap)
        freed = 0
        while freed < num_tokens and heap:
            _, _, _, victim = heapq.heappop(heap)
            parent = victim.parent
            self.free_pages.extend(s // self.page_size for s in victim.value[::self.page_size])
            freed += len(victim.value)
            self.evictable_size_ -= len(victim.key)
            self.eviction_log.append((victim.id, len(victim.key)))
            if self.on_host(victim):
                victim.value = None
            else:
                assert not victim.children, "a device-only node below a device leaf"
                del parent.children[self.child_key(victim.key, 0)]
                victim.evicted = True
                del self.nodes[victim.id]
            if (parent is not self.root and self.on_gpu(parent)
                    and not self._dev_children(parent) and parent.lock_ref == 0):
                heapq.heappush(heap, (parent.priority, parent.last_access_time, parent.id,
                                      parent))
        return freed

    def host_evict(self, num_tokens):
        """Host eviction: host-only childless nodes, least recent first."""
        heap = [(n.priority, n.last_access_time, n.id, n) for n in self.nodes.values()
                if n is not self.root and not self.on_gpu(n) and self.on_host(n)
                and not n.children]
        heapq.heapify(heap)
        freed = 0
        while freed < num_tokens and heap:
            _, _, _, victim = heapq.heappop(heap)
            parent = victim.parent
            self.free_host_pages.extend(s // self.page_size
                                        for s in victim.host_value[::self.page_size])
            freed += len(victim.host_value)
            self.host_eviction_log.append((victim.id, len(victim.key)))
            del parent.children[self.child_key(victim.key, 0)]
            victim.evicted = True
            del self.nodes[victim.id]
            if (parent is not self.root and not self.on_gpu(parent) and not parent.children):
                heapq.heappush(heap, (parent.priority, parent.last_access_time, parent.id,
                                      parent))
        return freed

    def host_alloc_pages(self, n):
        if len(self.free_host_pages) < n:
            self.host_evict((n - len(self.free_host_pages)) * self.page_size)
        if len(self.free_host_pages) < n:
            raise NoSpace(n)
        return [self.free_host_pages.popleft() for _ in range(n)]

    # ---------------------------------------------------------- transfers
    def _root_path(self, node):
        path = []
        while node is not self.root:
            path.append(node)
            node = node.parent
        return path[::-1]

    def write_through(self, node):
        """Back up the device-only nodes of ``node``'s root path.  Returns
        ``(ticket, device slots, host slots)`` (ticket 0 and empty lists when
        the path is on the host already)."""
        path = self._root_path(node)
        if any(x.pending is not None for x in path):
            return 0, [], []          # a backup on this path is still in flight
        todo = [x for x in path if not self.on_host(x)]
        n = sum(len(x.key) for x in todo)
        if n == 0:
            return 0, [], []
        pages = self.host_alloc_pages(n // self.page_size)
        ticket = self.next_ticket
        self.next_ticket += 1
        dev, host = [], []
        pos = 0
        for x in todo:
            hs = self.page_slots(pages[pos // self.page_size:], len(x.key))
            pos += len(x.key)
            x.pending = (ticket, hs)
            dev.extend(x.value)
            host.extend(hs)
        self.inc_lock_ref(node)
        self.pending[ticket] = node
        return ticket, dev, host

    def commit_write_through(self, ticket, success):
        node = self.pending.pop(ticket)
        x = node
        while x is not self.root:
            if x.pending is not None and x.pending[0] == ticket:
                if success:
                    x.host_value = x.pending[1]
                else:
                    self.free_host_pages.extend(s // self.page_size
                                                for s in x.pending[1][::self.page_size])
                x.pending = None
            x = x.parent
        self.dec_lock_ref(node)

    def load_onboard(self, node):
        """Bring the host-only nodes of ``node``'s root path to the device.
        Returns ``(host slots, device slots)`` to copy."""
        path = self._root_path(node)
        todo = [x for x in path if not self.on_gpu(x)]
        n = sum(len(x.key) for x in todo)
        if n == 0:
            return [], []
        dev_node = self.root
        for x in path:
            if not self.on_gpu(x):
                break
            dev_node = x
        self.inc_lock_ref(dev_node)
        try:
            pages = self.alloc_pages(n // self.page_size)
        finally:
            self.dec_lock_ref(dev_node)
        host, dev = [], []
        pos = 0
        for x in todo:
            ds = self.page_slots(pages[pos // self.page_size:], len(x.key))
            pos += len(x.key)
            x.value = ds
            self.evictable_size_ += len(x.key)
            host.extend(x.host_value)
            dev.extend(ds)
        return host, dev

    # --------------------------------------------------------------- stats
    def device_cached_size(self):
        return sum(len(n.key) for n in self.nodes.values() if n is not self.root and self.on_gpu(n))

    def host_cached_size(self):
        return sum(len(n.key) for n in self.nodes.values()
                   if n is not self.root and self.on_host(n))
