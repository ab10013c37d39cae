// Host radix cache over a token-granular KV slot pool (the rx_* host calls
// of include/rx.h).
//
// Sources, by page title and section:
//  - "SGLang: the tree, and the language nobody remembers", "A tree, not a
//    map": TreeNode{key, value, children, parent, lock_ref, last_access_time,
//    priority}; inc_lock_ref moves a node between the evictable and protected
//    counts; eviction pops a heap of candidates and pushes a parent once it is
//    childless and unlocked; a node splits at the divergence point; keys are
//    page-aligned (truncated to whole pages, matches rounded down to a page)
//    and children are keyed on the first token at page_size 1, on the first
//    page otherwise; the match inside an edge is a galloping search
//    (doubling windows, one block compare each, then a binary search of the
//    window holding the divergence).
//  - "SGLang" (bibekananda.in), "One tree for everybody" / "Eviction on a
//    tree": walk as far as the tokens match; the divergent part becomes a new
//    branch; leaves go first.
//  - "SGLang: Structured LLM Programs for Efficient Inference", "How
//    RadixAttention reuses past work" and "Worked example, step by step".
//
// Readings where the pages are silent: a logical access clock advanced once
// per match/insert and written on the whole touched path; heap key
// (priority = 0, last_access_time, node id); the pool cut into pages of
// page_size consecutive slots with page 0 a pad page, and a FIFO free list of
// pages 1..N/page_size-1 handing out whole pages (a request's positions
// [k*page_size, (k+1)*page_size) lie in one page, in slot order); a match
// ending inside an edge splits it; the split's upper half takes a fresh id and
// the lower half's lock_ref and access time.

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <deque>
#include <memory>
#include <queue>
#include <string>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "rx.h"
#include "rx_internal.h"

namespace {

thread_local std::string g_err;

rx_status fail(rx_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return s;
}

struct Node {
  int64_t id = 0;
  std::vector<int32_t> key;
  std::vector<int32_t> value;
  std::unordered_map<int32_t, Node*> children;       // page_size 1: first token
  std::unordered_map<std::string, Node*> pchildren;  // page_size > 1: first page
  Node* parent = nullptr;
  int64_t lock_ref = 0;
  int64_t last_access_time = 0;
  int32_t priority = 0;
  // Two-tier residency: device slots in `value` while `gpu`, host slots in
  // `host_value` while `host`; a backup in flight holds its host slots in
  // `pending_host` under ticket `pending_ticket`.
  bool gpu = true;
  bool host = false;
  std::vector<int32_t> host_value;
  int64_t pending_ticket = 0;
  std::vector<int32_t> pending_host;
};

// Length of the common prefix of a[0..n) and b[0..n): gallop over windows
// of doubling size with one memcmp each, then bisect the window that holds
// the first difference.
int64_t common_prefix(const int32_t* a, const int32_t* b, int64_t n) {
  int64_t i = 0, w = 16;
  while (i < n) {
    int64_t len = std::min(w, n - i);
    if (std::memcmp(a + i, b + i, size_t(len) * sizeof(int32_t)) != 0) {
      int64_t lo = i, hi = i + len;  // first difference lies in [lo, hi)
      while (hi - lo > 16) {
        int64_t mid = lo + (hi - lo) / 2;
        if (std::memcmp(a + lo, b + lo, size_t(mid - lo) * sizeof(int32_t)) == 0)
          lo = mid;
        else
          hi = mid;
      }
      while (lo < hi && a[lo] == b[lo]) ++lo;
      return lo;
    }
    i += len;
    w *= 2;
  }
  return n;
}

}  // namespace

struct rx_cache {
  int64_t num_slots = 0;
  int64_t ps = 1;  // page size in slots
  std::unordered_map<int64_t, std::unique_ptr<Node>> nodes;
  Node* root = nullptr;
  std::deque<int32_t> free_list;  // free pages (a page is a slot at page size 1)
  int64_t next_id = 1;
  int64_t clock = 0;
  int64_t evictable = 0;
  int64_t protected_ = 0;
  int64_t cached = 0;
  int64_t evicted_tokens = 0;
  std::vector<rx_evict_rec> evict_log;
  // host tier (empty when host_slots is 0)
  int64_t host_slots = 0;
  std::deque<int32_t> host_free;  // free host pages
  int64_t host_cached = 0;
  std::vector<rx_evict_rec> host_evict_log;
  std::unordered_map<int64_t, int64_t> tickets;  // ticket -> end node of the backup
  int64_t next_ticket = 1;
  // fault injection (tests): the fail_countdown-th page allocation from now
  // fails as if the pool were short after eviction; 0 = off
  int64_t fail_countdown = 0;
  bool injected_failure() {
    return fail_countdown > 0 && --fail_countdown == 0;
  }

  bool on_gpu(const Node* x) const { return x == root || x->gpu; }
  bool on_host(const Node* x) const { return x == root || x->host; }
  bool has_gpu_child(const Node* x) const {
    bool any = false;
    for_children(x, [&](const Node* c) { any = any || c->gpu; });
    return any;
  }

  // ------------------------------------------------------------- pages
  int64_t aligned(int64_t n) const { return n - n % ps; }
  int64_t pages_for(int64_t tokens) const { return (tokens + ps - 1) / ps; }
  std::string page_key(const int32_t* t) const {
    return std::string(reinterpret_cast<const char*>(t), size_t(ps) * sizeof(int32_t));
  }
  Node* child_of(const Node* n, const int32_t* t) const {
    if (ps == 1) {
      auto it = n->children.find(t[0]);
      return it == n->children.end() ? nullptr : it->second;
    }
    auto it = n->pchildren.find(page_key(t));
    return it == n->pchildren.end() ? nullptr : it->second;
  }
  void set_child(Node* n, const int32_t* t, Node* c) {
    if (ps == 1)
      n->children[t[0]] = c;
    else
      n->pchildren[page_key(t)] = c;
  }
  void erase_child(Node* n, const int32_t* t) {
    if (ps == 1)
      n->children.erase(t[0]);
    else
      n->pchildren.erase(page_key(t));
  }
  bool childless(const Node* n) const {
    return ps == 1 ? n->children.empty() : n->pchildren.empty();
  }
  template <class F>
  void for_children(const Node* n, F f) const {
    if (ps == 1)
      for (const auto& kv : n->children) f(kv.second);
    else
      for (const auto& kv : n->pchildren) f(kv.second);
  }
  // Pages of slots[0..n), each once, in order of first appearance, to the
  // free-list tail.
  void free_slot_pages(const int32_t* slots, int64_t n) {
    if (ps == 1) {
      for (int64_t i = 0; i < n; ++i) free_list.push_back(slots[i]);
      return;
    }
    std::unordered_set<int32_t> seen;
    for (int64_t i = 0; i < n; ++i) {
      const int32_t p = int32_t(slots[i] / ps);
      if (seen.insert(p).second) free_list.push_back(p);
    }
  }
  // Take n pages from the head of the free list, evicting the shortfall
  // first; false (nothing taken) if still short.
  bool alloc_pages(int64_t n, int32_t* out) {
    if (int64_t(free_list.size()) < n) evict((n - int64_t(free_list.size())) * ps);
    if (int64_t(free_list.size()) < n || injected_failure()) return false;
    for (int64_t i = 0; i < n; ++i) {
      out[i] = free_list.front();
      free_list.pop_front();
    }
    return true;
  }
  // The first k slots of pages[0..), page after page.
  void page_slots(const int32_t* pages, int64_t k, int32_t* out) const {
    for (int64_t i = 0; i < k; ++i) out[i] = int32_t(int64_t(pages[i / ps]) * ps + i % ps);
  }

  Node* new_node(const int32_t* k, const int32_t* v, int64_t n, Node* parent) {
    auto up = std::make_unique<Node>();
    Node* x = up.get();
    x->id = next_id++;
    x->key.assign(k, k + n);
    x->value.assign(v, v + n);
    x->parent = parent;
    nodes.emplace(x->id, std::move(up));
    return x;
  }

  Node* find(rx_node id) const {
    auto it = nodes.find(id);
    return it == nodes.end() ? nullptr : it->second.get();
  }

  // Split `node` after its first k tokens; returns the new upper node.
  Node* split(Node* node, int64_t k) {
    Node* parent = node->parent;
    Node* upper = new_node(node->key.data(), node->value.data(), node->gpu ? k : 0, parent);
    upper->key.assign(node->key.begin(), node->key.begin() + k);
    upper->lock_ref = node->lock_ref;
    upper->last_access_time = node->last_access_time;
    upper->gpu = node->gpu;
    if (node->host) {
      upper->host = true;
      upper->host_value.assign(node->host_value.begin(), node->host_value.begin() + k);
      node->host_value.erase(node->host_value.begin(), node->host_value.begin() + k);
    }
    if (node->pending_ticket) {
      upper->pending_ticket = node->pending_ticket;
      upper->pending_host.assign(node->pending_host.begin(), node->pending_host.begin() + k);
      node->pending_host.erase(node->pending_host.begin(), node->pending_host.begin() + k);
    }
    set_child(parent, node->key.data(), upper);
    node->key.erase(node->key.begin(), node->key.begin() + k);
    if (node->gpu) node->value.erase(node->value.begin(), node->value.begin() + k);
    node->parent = upper;
    set_child(upper, node->key.data(), node);
    return upper;
  }

  int64_t match_length(const int32_t* t, int64_t n) const {
    n = aligned(n);
    const Node* node = root;
    int64_t pos = 0;
    while (pos < n) {
      const Node* c = child_of(node, t + pos);
      if (!c) break;
      int64_t lim = std::min<int64_t>(int64_t(c->key.size()), n - pos);
      int64_t k = aligned(common_prefix(c->key.data(), t + pos, lim));
      pos += k;
      if (k < int64_t(c->key.size())) break;
      node = c;
    }
    return pos;
  }

  // Slots of the longest cached prefix of t[0..n) (no split, no touch);
  // writes them to out and returns the matched length.
  int64_t lookup_slots(const int32_t* t, int64_t n, int32_t* out) const {
    n = aligned(n);
    const Node* node = root;
    int64_t pos = 0;
    while (pos < n) {
      const Node* c = child_of(node, t + pos);
      if (!c || !c->gpu) break;
      int64_t lim = std::min<int64_t>(int64_t(c->key.size()), n - pos);
      int64_t k = aligned(common_prefix(c->key.data(), t + pos, lim));
      std::memcpy(out + pos, c->value.data(), size_t(k) * sizeof(int32_t));
      pos += k;
      if (k < int64_t(c->key.size())) break;
      node = c;
    }
    return pos;
  }

  // Walk every tier (splitting at the end of the match); returns the
  // deepest node and the matched length; *dev_len / *dev_node = the leading
  // device-resident part of the walk and its last node, whose slots are
  // written to `slots` if non-null.
  Node* walk(const int32_t* t, int64_t n, int64_t* matched,
             std::vector<Node*>* path, int32_t* slots, int64_t* dev_len = nullptr,
             Node** dev_node = nullptr) {
    n = aligned(n);
    Node* node = root;
    Node* dnode = root;
    int64_t pos = 0, dlen = 0;
    bool dev_run = true;
    while (pos < n) {
      Node* c = child_of(node, t + pos);
      if (!c) break;
      int64_t lim = std::min<int64_t>(int64_t(c->key.size()), n - pos);
      int64_t k = aligned(common_prefix(c->key.data(), t + pos, lim));
      if (k < int64_t(c->key.size())) c = split(c, k);
      if (dev_run && c->gpu) {
        if (slots) std::memcpy(slots + pos, c->value.data(), size_t(k) * sizeof(int32_t));
        dlen += k;
        dnode = c;
      } else {
        dev_run = false;
      }
      pos += k;
      path->push_back(c);
      node = c;
    }
    *matched = pos;
    if (dev_len) *dev_len = dlen;
    if (dev_node) *dev_node = dnode;
    return node;
  }

  // The device part of a match across tiers.
  Node* match_prefix(const int32_t* t, int64_t n, int32_t* slots,
                     int64_t* len) {
    clock += 1;
    std::vector<Node*> path;
    int64_t all = 0;
    Node* dnode = root;
    walk(t, n, &all, &path, slots, len, &dnode);
    for (Node* x : path) x->last_access_time = clock;
    return dnode;
  }

  // Inserts the whole pages of t[0..n) (the key truncated to a multiple of
  // the page size).
  Node* insert(const int32_t* t, const int32_t* s, int64_t n,
               int64_t* already) {
    n = aligned(n);
    clock += 1;
    std::vector<Node*> path;
    int64_t pos = 0;
    Node* node = walk(t, n, &pos, &path, nullptr, already);
    // host-only nodes of the path adopt the caller's device slots
    int64_t off = 0;
    for (Node* x : path) {
      const int64_t len = int64_t(x->key.size());
      if (!x->gpu) {
        x->value.assign(s + off, s + off + len);
        x->gpu = true;
        (x->lock_ref > 0 ? protected_ : evictable) += len;
        cached += len;
      }
      off += len;
    }
    if (pos < n) {
      Node* leaf = new_node(t + pos, s + pos, n - pos, node);
      set_child(node, t + pos, leaf);
      evictable += n - pos;
      cached += n - pos;
      path.push_back(leaf);
      node = leaf;
    }
    for (Node* x : path) x->last_access_time = clock;
    return node;
  }

  void lock(Node* node) {
    for (; node != root; node = node->parent) {
      if (node->lock_ref == 0) {
        evictable -= int64_t(node->key.size());
        protected_ += int64_t(node->key.size());
      }
      node->lock_ref += 1;
    }
  }

  bool unlock(Node* node) {
    for (Node* w = node; w != root; w = w->parent)
      if (w->lock_ref <= 0) return false;
    for (; node != root; node = node->parent) {
      if (node->lock_ref == 1) {
        evictable += int64_t(node->key.size());
        protected_ -= int64_t(node->key.size());
      }
      node->lock_ref -= 1;
    }
    return true;
  }

  int64_t evict(int64_t k) {
    struct Cand {
      int32_t priority;
      int64_t time, id;
      Node* node;
      bool operator>(const Cand& o) const {
        if (priority != o.priority) return priority > o.priority;
        if (time != o.time) return time > o.time;
        return id > o.id;
      }
    };
    std::priority_queue<Cand, std::vector<Cand>, std::greater<Cand>> heap;
    std::vector<Node*> stack{root};
    while (!stack.empty()) {
      Node* x = stack.back();
      stack.pop_back();
      if (x != root && x->gpu && !has_gpu_child(x) && x->lock_ref == 0)
        heap.push({x->priority, x->last_access_time, x->id, x});
      for_children(x, [&](Node* c) { stack.push_back(c); });
    }
    int64_t freed = 0;
    while (freed < k && !heap.empty()) {
      Node* v = heap.top().node;
      heap.pop();
      Node* parent = v->parent;
      for (size_t i = 0; i < v->value.size(); i += size_t(ps))
        free_list.push_back(int32_t(v->value[i] / ps));
      int64_t len = int64_t(v->key.size());
      freed += len;
      evictable -= len;
      cached -= len;
      evicted_tokens += len;
      evict_log.push_back({v->id, len});
      if (v->host) {  // the host copy stays: the node leaves the device only
        v->gpu = false;
        v->value.clear();
      } else {
        erase_child(parent, v->key.data());
        nodes.erase(v->id);
      }
      if (parent != root && parent->gpu && !has_gpu_child(parent) && parent->lock_ref == 0)
        heap.push({parent->priority, parent->last_access_time, parent->id,
                   parent});
    }
    return freed;
  }

  // Host eviction: host-only childless nodes, least recent first; their
  // parent joins once childless and host-only.
  int64_t host_evict(int64_t k) {
    struct Cand {
      int32_t priority;
      int64_t time, id;
      Node* node;
      bool operator>(const Cand& o) const {
        if (priority != o.priority) return priority > o.priority;
        if (time != o.time) return time > o.time;
        return id > o.id;
      }
    };
    std::priority_queue<Cand, std::vector<Cand>, std::greater<Cand>> heap;
    for (auto& kv : nodes) {
      Node* x = kv.second.get();
      if (x != root && !x->gpu && x->host && childless(x))
        heap.push({x->priority, x->last_access_time, x->id, x});
    }
    int64_t freed = 0;
    while (freed < k && !heap.empty()) {
      Node* v = heap.top().node;
      heap.pop();
      Node* parent = v->parent;
      for (size_t i = 0; i < v->host_value.size(); i += size_t(ps))
        host_free.push_back(int32_t(v->host_value[i] / ps));
      const int64_t len = int64_t(v->key.size());
      freed += len;
      host_cached -= len;
      host_evict_log.push_back({v->id, len});
      erase_child(parent, v->key.data());
      nodes.erase(v->id);
      if (parent != root && !parent->gpu && parent->host && childless(parent))
        heap.push({parent->priority, parent->last_access_time, parent->id, parent});
    }
    return freed;
  }

  bool host_alloc_pages(int64_t n, int32_t* out) {
    if (int64_t(host_free.size()) < n) host_evict((n - int64_t(host_free.size())) * ps);
    if (int64_t(host_free.size()) < n || injected_failure()) return false;
    for (int64_t i = 0; i < n; ++i) {
      out[i] = host_free.front();
      host_free.pop_front();
    }
    return true;
  }

  std::vector<Node*> root_path(Node* x) const {
    std::vector<Node*> p;
    for (; x != root; x = x->parent) p.push_back(x);
    std::reverse(p.begin(), p.end());
    return p;
  }

  // k slots: the first k slots of ceil(k / page size) pages (all of them at
  // page size 1).
  bool alloc(int64_t k, int32_t* out) {
    if (ps == 1) return alloc_pages(k, out);
    std::vector<int32_t> pages(size_t(pages_for(k)));
    if (!alloc_pages(int64_t(pages.size()), pages.data())) return false;
    page_slots(pages.data(), k, out);
    return true;
  }

  int64_t depth(const Node* x) const {
    int64_t d = 0;
    for (; x != root; x = x->parent) d += int64_t(x->key.size());
    return d;
  }
};

// ---------------------------------------------------------------- C ABI
// Whether two token sequences share more than `m` leading tokens counted in
// whole pages of `ps` tokens (m itself a multiple of ps), i.e. their first
// m + ps tokens agree: the page after position m is compared first (where
// prompts that match the tree to depth m usually part), the m tokens before
// it only when that one agrees.
static bool shares_more_than(const int32_t* a, int64_t na, const int32_t* b, int64_t nb,
                             int64_t m, int64_t ps = 1) {
  if (m < 0) return true;
  const int64_t need = m + ps;
  if (na < need || nb < need || a[m] != b[m]) return false;
  if (std::memcmp(a + m, b + m, size_t(ps) * sizeof(int32_t)) != 0) return false;
  return common_prefix(a, b, m) == m;
}

extern "C" {

size_t rx_last_error(char* buf, size_t cap) {
  if (buf && cap) {
    size_t n = std::min(cap - 1, g_err.size());
    std::memcpy(buf, g_err.data(), n);
    buf[n] = 0;
  }
  return g_err.size();
}

rx_status rx_cache_create(const rx_config* cfg, rx_cache** out) {
  if (!cfg || !out) return fail(RX_ERR_INVALID, "rx_cache_create: NULL argument");
  if (cfg->num_slots < 1 || cfg->num_slots > (int64_t(1) << 31))
    return fail(RX_ERR_INVALID, "rx_cache_create: num_slots %lld out of range",
                (long long)cfg->num_slots);
  if (cfg->page_size < 1 || cfg->num_slots < cfg->page_size ||
      cfg->num_slots % cfg->page_size != 0)
    return fail(RX_ERR_INVALID,
                "rx_cache_create: page_size %d must be >= 1 and divide num_slots %lld",
                cfg->page_size, (long long)cfg->num_slots);
  if (cfg->host_slots < 0 || cfg->host_slots % cfg->page_size != 0)
    return fail(RX_ERR_INVALID, "rx_cache_create: host_slots %lld not a multiple of page_size",
                (long long)cfg->host_slots);
  auto* c = new rx_cache();
  c->num_slots = cfg->num_slots;
  c->ps = cfg->page_size;
  c->host_slots = cfg->host_slots;
  for (int64_t p = 1; p < cfg->host_slots / cfg->page_size; ++p) c->host_free.push_back(int32_t(p));
  auto root = std::make_unique<Node>();
  root->id = 0;
  c->root = root.get();
  c->nodes.emplace(0, std::move(root));
  for (int64_t p = 1; p < cfg->num_slots / cfg->page_size; ++p)
    c->free_list.push_back(int32_t(p));
  *out = c;
  return RX_OK;
}

rx_status rx_cache_destroy(rx_cache* cache) {
  delete cache;
  return RX_OK;
}

rx_status rx_match_length(const rx_cache* c, const int32_t* tokens, int64_t n,
                          int64_t* out_len) {
  if (!c || (!tokens && n) || n < 0 || !out_len)
    return fail(RX_ERR_INVALID, "rx_match_length: bad argument");
  *out_len = c->match_length(tokens, n);
  return RX_OK;
}

rx_status rx_match_prefix(rx_cache* c, const int32_t* tokens, int64_t n,
                          int32_t* out_slots, int64_t* out_len,
                          rx_node* out_node) {
  if (!c || (!tokens && n) || n < 0 || (!out_slots && n) || !out_len || !out_node)
    return fail(RX_ERR_INVALID, "rx_match_prefix: bad argument");
  Node* x = c->match_prefix(tokens, n, out_slots, out_len);
  *out_node = x->id;
  return RX_OK;
}

rx_status rx_lock(rx_cache* c, rx_node node) {
  Node* x = c ? c->find(node) : nullptr;
  if (!x) return fail(RX_ERR_INVALID, "rx_lock: unknown node %lld", (long long)node);
  for (Node* w = x; w != c->root; w = w->parent)
    if (!w->gpu) return fail(RX_ERR_STATE, "rx_lock: node %lld not on the device", (long long)node);
  c->lock(x);
  return RX_OK;
}

rx_status rx_unlock(rx_cache* c, rx_node node) {
  Node* x = c ? c->find(node) : nullptr;
  if (!x) return fail(RX_ERR_INVALID, "rx_unlock: unknown node %lld", (long long)node);
  if (!c->unlock(x))
    return fail(RX_ERR_STATE, "rx_unlock: lock_ref of node %lld would go below 0",
                (long long)node);
  return RX_OK;
}

rx_status rx_alloc(rx_cache* c, int64_t k, int32_t* out_slots) {
  if (!c || k < 0 || (!out_slots && k)) return fail(RX_ERR_INVALID, "rx_alloc: bad argument");
  if (!c->alloc(k, out_slots))
    return fail(RX_ERR_NO_SPACE, "rx_alloc: %lld slots requested, %lld free after eviction",
                (long long)k, (long long)(int64_t(c->free_list.size()) * c->ps));
  return RX_OK;
}

rx_status rx_evict(rx_cache* c, int64_t k, int64_t* out_freed) {
  if (!c || k < 0) return fail(RX_ERR_INVALID, "rx_evict: bad argument");
  int64_t f = c->evict(k);
  if (out_freed) *out_freed = f;
  return RX_OK;
}

rx_status rx_free(rx_cache* c, const int32_t* slots, int64_t k) {
  if (!c || k < 0 || (!slots && k)) return fail(RX_ERR_INVALID, "rx_free: bad argument");
  for (int64_t i = 0; i < k; ++i) {
    if (slots[i] < c->ps || slots[i] >= c->num_slots)
      return fail(RX_ERR_INVALID, "rx_free: slot %d out of range", slots[i]);
  }
  c->free_slot_pages(slots, k);
  return RX_OK;
}

rx_status rx_insert(rx_cache* c, const int32_t* tokens, const int32_t* slots,
                    int64_t n, int64_t* out_already, rx_node* out_node) {
  if (!c || n < 0 || (n && (!tokens || !slots)) || !out_already)
    return fail(RX_ERR_INVALID, "rx_insert: bad argument");
  Node* x = c->insert(tokens, slots, n, out_already);
  if (out_node) *out_node = x->id;
  return RX_OK;
}

rx_status rx_stats(const rx_cache* c, rx_stats_t* out) {
  if (!c || !out) return fail(RX_ERR_INVALID, "rx_stats: bad argument");
  out->cached_tokens = c->cached;
  out->evictable_tokens = c->evictable;
  out->protected_tokens = c->protected_;
  out->free_slots = int64_t(c->free_list.size()) * c->ps;
  out->num_nodes = int64_t(c->nodes.size()) - 1;
  out->evicted_nodes = int64_t(c->evict_log.size());
  out->evicted_tokens = c->evicted_tokens;
  out->clock = c->clock;
  out->host_cached_tokens = c->host_cached;
  out->host_free_slots = int64_t(c->host_free.size()) * c->ps;
  out->host_evicted_nodes = int64_t(c->host_evict_log.size());
  return RX_OK;
}

rx_status rx_eviction_log(const rx_cache* c, int64_t start, rx_evict_rec* out,
                          int64_t cap, int64_t* out_total) {
  if (!c || start < 0 || cap < 0 || (cap && !out))
    return fail(RX_ERR_INVALID, "rx_eviction_log: bad argument");
  int64_t total = int64_t(c->evict_log.size());
  for (int64_t i = 0; i < cap && start + i < total; ++i) out[i] = c->evict_log[start + i];
  if (out_total) *out_total = total;
  return RX_OK;
}

rx_status rx_node_depth(const rx_cache* c, rx_node node, int64_t* out_depth) {
  const Node* x = c ? c->find(node) : nullptr;
  if (!x || !out_depth) return fail(RX_ERR_INVALID, "rx_node_depth: unknown node");
  *out_depth = c->depth(x);
  return RX_OK;
}

// ------------------------------------------------------- batch helpers
rx_status rx_extend_begin(rx_cache* c, int32_t R, const int32_t* tokens,
                          const int64_t* tok_indptr, int32_t* req_to_token,
                          int64_t row_stride, int32_t* out_prefix_len,
                          rx_node* out_match_node, int32_t* out_new_slots,
                          int64_t* out_total_new) {
  if (!c || R < 0 || !tok_indptr || (R && (!tokens || !req_to_token || !out_prefix_len ||
                                          !out_match_node || !out_new_slots)) ||
      !out_total_new)
    return fail(RX_ERR_INVALID, "rx_extend_begin: bad argument");
  for (int32_t r = 0; r < R; ++r) {
    int64_t n = tok_indptr[r + 1] - tok_indptr[r];
    if (n < 1 || n > row_stride)
      return fail(RX_ERR_INVALID, "rx_extend_begin: prompt %d has length %lld (row %lld)", r,
                  (long long)n, (long long)row_stride);
  }
  int64_t total_new = 0, total_pages = 0;
  for (int32_t r = 0; r < R; ++r) {
    const int32_t* t = tokens + tok_indptr[r];
    int64_t n = tok_indptr[r + 1] - tok_indptr[r];
    int64_t m = 0;
    Node* x = c->match_prefix(t, n - 1, req_to_token + r * row_stride, &m);
    c->lock(x);
    out_prefix_len[r] = int32_t(m);
    out_match_node[r] = x->id;
    total_new += n - m;
    total_pages += c->pages_for(n - m);
  }
  // one allocation of every member's pages, handed out in member order; a
  // member's new tokens fill its own pages in order
  std::vector<int32_t> pages;
  int32_t* page_out = out_new_slots;
  if (c->ps > 1) {
    pages.resize(size_t(total_pages));
    page_out = pages.data();
  }
  if (!c->alloc_pages(total_pages, page_out)) {
    for (int32_t r = 0; r < R; ++r) c->unlock(c->find(out_match_node[r]));
    return fail(RX_ERR_NO_SPACE, "rx_extend_begin: %lld new slots needed, %lld free after eviction",
                (long long)total_new, (long long)(int64_t(c->free_list.size()) * c->ps));
  }
  int64_t pos = 0, pg = 0;
  for (int32_t r = 0; r < R; ++r) {
    int64_t n = tok_indptr[r + 1] - tok_indptr[r];
    int64_t m = out_prefix_len[r];
    if (c->ps > 1) {
      c->page_slots(pages.data() + pg, n - m, out_new_slots + pos);
      pg += c->pages_for(n - m);
    }
    std::memcpy(req_to_token + r * row_stride + m, out_new_slots + pos,
                size_t(n - m) * sizeof(int32_t));
    pos += n - m;
  }
  *out_total_new = total_new;
  return RX_OK;
}

rx_status rx_extend_end(rx_cache* c, int32_t R, const int32_t* tokens,
                        const int64_t* tok_indptr, int32_t* req_to_token,
                        int64_t row_stride, const int32_t* prefix_len,
                        const rx_node* match_node, rx_node* out_prompt_node,
                        int64_t* out_rewritten) {
  if (!c || R < 0 || !tok_indptr || (R && (!tokens || !req_to_token || !prefix_len ||
                                          !match_node || !out_prompt_node)))
    return fail(RX_ERR_INVALID, "rx_extend_end: bad argument");
  for (int32_t r = 0; r < R; ++r) {
    if (!c->find(match_node[r]))
      return fail(RX_ERR_INVALID, "rx_extend_end: unknown node %lld", (long long)match_node[r]);
  }
  int64_t rewritten = 0;
  std::vector<int32_t> tree;
  for (int32_t r = 0; r < R; ++r) {
    const int32_t* t = tokens + tok_indptr[r];
    int64_t n = tok_indptr[r + 1] - tok_indptr[r];
    int32_t* row = req_to_token + r * row_stride;
    int64_t already = 0;
    Node* x = c->insert(t, row, n, &already);
    if (already > prefix_len[r]) {
      // Identical prompt inserted by an earlier batch: adopt the tree's slots
      // (same tokens, same predecessors, same K/V) and free this request's.
      tree.resize(size_t(n));
      c->lookup_slots(t, already, tree.data());
      c->free_slot_pages(row + prefix_len[r], already - prefix_len[r]);
      for (int64_t i = prefix_len[r]; i < already; ++i) row[i] = tree[size_t(i)];
      ++rewritten;
    }
    c->lock(x);
    c->unlock(c->find(match_node[r]));
    out_prompt_node[r] = x->id;
  }
  if (out_rewritten) *out_rewritten = rewritten;
  return RX_OK;
}

rx_status rx_finish(rx_cache* c, int32_t R, const int32_t* tokens,
                    const int64_t* tok_indptr, const int32_t* req_to_token,
                    int64_t row_stride, const int64_t* prompt_len,
                    const rx_node* prompt_node, int64_t* out_already,
                    rx_node* out_full_node) {
  if (!c || R < 0 || !tok_indptr || (R && (!tokens || !req_to_token || !prompt_len ||
                                          !prompt_node)))
    return fail(RX_ERR_INVALID, "rx_finish: bad argument");
  for (int32_t r = 0; r < R; ++r) {
    if (!c->find(prompt_node[r]))
      return fail(RX_ERR_INVALID, "rx_finish: unknown node %lld", (long long)prompt_node[r]);
    if (tok_indptr[r + 1] - tok_indptr[r] > row_stride)
      return fail(RX_ERR_INVALID, "rx_finish: sequence %d longer than the row", r);
  }
  for (int32_t r = 0; r < R; ++r) {
    const int32_t* t = tokens + tok_indptr[r];
    int64_t n = tok_indptr[r + 1] - tok_indptr[r];
    const int32_t* row = req_to_token + r * row_stride;
    int64_t already = 0;
    Node* full = c->insert(t, row, n, &already);
    if (out_full_node) out_full_node[r] = full->id;
    // the request's own pages another request had already inserted, and the
    // partly filled page past the last whole one
    const int64_t p_al = c->aligned(prompt_len[r]);
    if (already > p_al) c->free_slot_pages(row + p_al, already - p_al);
    if (c->aligned(n) < n) c->free_slot_pages(row + c->aligned(n), 1);
    if (out_already) out_already[r] = already;
    if (!c->unlock(c->find(prompt_node[r])))
      return fail(RX_ERR_STATE, "rx_finish: request %d was not locked", r);
  }
  return RX_OK;
}

rx_status rx_batch_conflict(const int32_t* tokens, int64_t n, int64_t match_len,
                            int32_t R, const int32_t* member_tokens,
                            const int64_t* member_indptr, int32_t* out_conflict) {
  if ((!tokens && n) || n < 0 || R < 0 || (R && (!member_tokens || !member_indptr)) ||
      !out_conflict)
    return fail(RX_ERR_INVALID, "rx_batch_conflict: bad argument");
  *out_conflict = 0;
  for (int32_t r = 0; r < R; ++r)
    if (shares_more_than(tokens, n, member_tokens + member_indptr[r],
                         member_indptr[r + 1] - member_indptr[r], match_len)) {
      *out_conflict = 1;
      break;
    }
  return RX_OK;
}

rx_status rx_batch_end(const rx_cache* c, const int32_t* tokens, const int64_t* indptr,
                       int32_t start, int32_t R, int32_t* out_end) {
  if (!c || !tokens || !indptr || start < 0 || start >= R || !out_end)
    return fail(RX_ERR_INVALID, "rx_batch_end: bad argument");
  for (int32_t j = start + 1; j < R; ++j) {
    const int32_t* pj = tokens + indptr[j];
    const int64_t nj = indptr[j + 1] - indptr[j];
    if (nj < 1) return fail(RX_ERR_INVALID, "rx_batch_end: empty prompt %d", j);
    const int64_t m = c->match_length(pj, nj - 1);
    for (int32_t r = start; r < j; ++r)
      if (shares_more_than(pj, nj, tokens + indptr[r], indptr[r + 1] - indptr[r], m, c->ps)) {
        *out_end = j;
        return RX_OK;
      }
  }
  *out_end = R;
  return RX_OK;
}

}  // extern "C"

// -------------------------------------------------------- decode plan
// A tree node on the root path of >= 2 requests of the decode batch is read
// once for all of them (a multi-query tile); each request's remaining context
// is private.  Runs of consecutive nodes visited by the same requests are one
// segment (a child's visitors are a subset of its parent's, so equal counts
// mean equal sets).  Segments are cut into key chunks and member blocks, one
// CTA per (chunk, block, KV head); every (chunk, member) yields a partial
// (o, lse) entry that the merge combines per request.
static rx_status plan_decode_impl(const rx_cache* c, int32_t B, int32_t n_steps,
                                  const rx_node* prompt_node, const int32_t* ctx_len,
                                  const int32_t* req_rows, int32_t num_q_heads,
                                  int32_t num_kv_heads, int32_t head_dim, int32_t* plan,
                                  int64_t plan_cap, rx_decode_plan_info* info) {
  if (n_steps < 1) return fail(RX_ERR_INVALID, "rx_plan_decode: n_steps < 1");
  if (!c || B < 0 || !info || (B && (!prompt_node || !ctx_len || !req_rows)))
    return fail(RX_ERR_INVALID, "rx_plan_decode: bad argument");
  if (num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads != 0)
    return fail(RX_ERR_INVALID, "rx_plan_decode: Hq %d not a multiple of Hkv %d", num_q_heads,
                num_kv_heads);
  const int32_t G = num_q_heads / num_kv_heads;
  if (head_dim != 128 && head_dim != 256)
    return fail(RX_ERR_INVALID, "rx_plan_decode: head_dim must be 128 or 256");
  if (G > rx_internal::decode_rows_per_item(head_dim))
    return fail(RX_ERR_INVALID, "rx_plan_decode: group size %d above %d", G,
                rx_internal::decode_rows_per_item(head_dim));
  std::vector<std::vector<const Node*>> paths(static_cast<size_t>(B));
  std::unordered_map<const Node*, int32_t> visits;
  for (int32_t b = 0; b < B; ++b) {
    const Node* x = c->find(prompt_node[b]);
    if (!x)
      return fail(RX_ERR_INVALID, "rx_plan_decode: unknown node %lld", (long long)prompt_node[b]);
    if (c->depth(x) > ctx_len[b] || ctx_len[b] < 1)
      return fail(RX_ERR_INVALID, "rx_plan_decode: ctx_len %d shorter than node depth",
                  ctx_len[b]);
    for (; x != c->root; x = x->parent) paths[b].push_back(x);
    std::reverse(paths[b].begin(), paths[b].end());
    for (const Node* n : paths[b]) visits[n] += 1;
  }
  struct Seg {
    int32_t row;
    int64_t kb, ke;
    std::vector<int32_t> members;
    int64_t grow = 0;  // private tail: its end at step t is min(ke, grow + t)
  };
  std::vector<Seg> segs;
  std::unordered_map<const Node*, size_t> seg_of;
  int64_t n_shared = 0;
  // every request's first-step token past its shared segments (the warp
  // kernel then owns each step's newest token)
  const int64_t small_rows = rx_internal::decode_small_rows(head_dim);
  bool tails_private = G <= small_rows;
  for (int32_t b = 0; b < B; ++b) {
    const auto& path = paths[b];
    int64_t pos = 0;
    size_t i = 0;
    while (i < path.size() && visits[path[i]] >= 2) {
      int32_t cnt = visits[path[i]];
      const Node* first = path[i];
      int64_t start = pos;
      while (i < path.size() && visits[path[i]] == cnt) {
        pos += int64_t(path[i]->key.size());
        ++i;
      }
      auto it = seg_of.find(first);
      if (it == seg_of.end()) {
        seg_of.emplace(first, segs.size());
        segs.push_back(Seg{req_rows[b], start, pos, {b}});
        ++n_shared;
      } else {
        segs[it->second].members.push_back(b);
      }
    }
    // private tail: covers the context of the last step; at step t it ends at
    // ctx_len[b] + t
    const int64_t last = int64_t(ctx_len[b]) + n_steps - 1;
    if (int64_t(ctx_len[b]) <= pos) tails_private = false;
    if (last > pos) segs.push_back(Seg{req_rows[b], pos, last, {b}, int64_t(ctx_len[b])});
  }
  // work items: (key chunk, member block) of each segment.  Segments with <=
  // small_rows rows go to the warp role of the decode kernel (listed
  // first), larger ones to its tensor-core tiles in member blocks of <=
  // kDecodeTcRows rows (listed last); chunks are cut at the tile's key step
  // (128 keys at head_dim 128, 64 at 256).
  struct Work {
    int32_t row, kb, ke, member_off, n_members, grow;
  };
  // A segment goes to the warp role when its rows fit one warp-role item, or
  // when it has at most kDecodeSplitRows rows: those are cut into member
  // blocks of at most small_rows rows (each block re-reads the segment's
  // keys, mostly from L2), which costs the GPU less than a 128-row tile
  // that would be mostly empty.
  const int64_t warp_block = std::max<int64_t>(1, small_rows / G);
  auto is_warp_seg = [&](int64_t members_k) {
    const int64_t rows = members_k * G;
    return rows <= small_rows || (rows <= rx_internal::kDecodeSplitRows && G <= small_rows);
  };
  auto warp_blocks = [&](int64_t members_k) {
    return members_k * G <= small_rows ? int64_t(1) : (members_k + warp_block - 1) / warp_block;
  };
  // chunk of the warp-role items: the longest that keeps enough units
  int64_t small_chunk = rx_internal::kDecodeSmallChunkMin;
  for (int64_t c = rx_internal::kDecodeSmallChunkMax; c > rx_internal::kDecodeSmallChunkMin;
       c /= 2) {
    int64_t units = 0;
    for (const Seg& s : segs)
      if (is_warp_seg(int64_t(s.members.size())))
        units += (s.ke - s.kb + c - 1) / c * warp_blocks(int64_t(s.members.size())) * num_kv_heads;
    if (units >= int64_t(rx_internal::kDecodeWarpSlots) * rx_internal::kDecodeUnitsPerWarp) {
      small_chunk = c;
      break;
    }
  }
  // chunks of the tensor-core items: kDecodeKeysPerRow keys per row (at
  // least kDecodeMinChunk), times the smallest power of two that keeps the
  // tile CTAs at or below kDecodeTcCap
  auto tc_base_chunk = [&](int64_t rows) {
    return std::max<int64_t>(rx_internal::kDecodeMinChunk, rx_internal::kDecodeKeysPerRow * rows);
  };
  int64_t tc_scale = 1;
  for (; tc_scale < 64; tc_scale *= 2) {
    int64_t ctas = 0;
    for (const Seg& s : segs) {
      const int64_t rows = int64_t(s.members.size()) * G;
      if (is_warp_seg(int64_t(s.members.size()))) continue;
      const int64_t per_block = rx_internal::kDecodeTcRows / G;
      const int64_t blocks = (int64_t(s.members.size()) + per_block - 1) / per_block;
      const int64_t c = tc_base_chunk(rows) * tc_scale;
      ctas += (s.ke - s.kb + c - 1) / c * blocks * num_kv_heads;
    }
    if (ctas <= rx_internal::kDecodeTcCap) break;
  }
  std::vector<Work> small, large;
  std::vector<int32_t> members;
  int64_t distinct = 0;
  for (const Seg& s : segs) {
    const int64_t n = s.ke - s.kb;
    distinct += s.grow ? std::max<int64_t>(0, s.grow - s.kb) : n;
    const int32_t k = int32_t(s.members.size());
    const int64_t rows = int64_t(k) * G;
    bool is_small;
    int32_t per_block;
    int64_t chunk, step;
    if (is_warp_seg(k)) {
      is_small = true;
      per_block = rows <= small_rows ? k : int32_t(warp_block);
      chunk = std::max<int64_t>(small_chunk, 2 * std::min<int64_t>(rows, small_rows));
      step = 16;
    } else {
      is_small = false;
      per_block = rx_internal::kDecodeTcRows / G;
      chunk = tc_base_chunk(rows) * tc_scale;
      step = head_dim == 128 ? 128 : 64;
    }
    const int64_t n_chunks = (n + chunk - 1) / chunk;
    int64_t len = (n + n_chunks - 1) / n_chunks;
    len = (len + step - 1) / step * step;
    const int32_t moff = int32_t(members.size());
    members.insert(members.end(), s.members.begin(), s.members.end());
    for (int64_t kb = s.kb; kb < s.ke; kb += len) {
      const int64_t ke = std::min(s.ke, kb + len);
      for (int32_t m0 = 0; m0 < k; m0 += per_block) {
        Work w{s.row, int32_t(kb), int32_t(ke), moff + m0, std::min(per_block, k - m0),
               int32_t(s.grow)};
        (is_small ? small : large).push_back(w);
      }
    }
  }
  auto heavier = [](const Work& a, const Work& b) {
    return int64_t(a.ke - a.kb) * a.n_members > int64_t(b.ke - b.kb) * b.n_members;
  };
  std::stable_sort(small.begin(), small.end(), heavier);
  std::stable_sort(large.begin(), large.end(), heavier);
  std::vector<Work> work = small;
  work.insert(work.end(), large.begin(), large.end());
  info->n_work_tc = int64_t(large.size());
  std::vector<std::vector<int32_t>> parts_of(static_cast<size_t>(B));
  int64_t n_parts = 0;
  for (const Work& w : work) {
    for (int32_t i = 0; i < w.n_members; ++i)
      parts_of[size_t(members[size_t(w.member_off + i)])].push_back(int32_t(n_parts + i));
    n_parts += w.n_members;
  }
  info->n_work = int64_t(work.size());
  info->n_parts = n_parts;
  info->n_member_entries = int64_t(members.size());
  info->off_work = 0;
  info->off_members = info->off_work + info->n_work * RX_WORK_WORDS;
  info->off_req_part_indptr = info->off_members + info->n_member_entries;
  info->off_req_parts = info->off_req_part_indptr + B + 1;
  info->plan_words = info->off_req_parts + n_parts;
  info->n_shared_segments = n_shared;
  int64_t o_bytes = n_parts * num_q_heads * int64_t(head_dim) * 4;
  int64_t l_bytes = n_parts * num_q_heads * 4;
  // partial o, partial lse, and one 256-byte block for the decode kernel's
  // work counter
  // partial results, then the work counters (one per step of the plan)
  info->workspace_bytes = ((o_bytes + 255) / 256) * 256 + ((l_bytes + 255) / 256) * 256 +
                          std::max<int64_t>(256, (4 * int64_t(n_steps) + 255) / 256 * 256);
  info->distinct_kv_tokens = distinct;
  info->tails_private = tails_private ? 1 : 0;
  if (!plan || plan_cap < info->plan_words)
    return fail(RX_ERR_INVALID, "rx_plan_decode: plan needs %lld words, capacity %lld",
                (long long)info->plan_words, (long long)plan_cap);
  int64_t part = 0;
  for (size_t w = 0; w < work.size(); ++w) {
    int32_t* o = plan + info->off_work + int64_t(w) * RX_WORK_WORDS;
    o[0] = work[w].row;
    o[1] = work[w].kb;
    o[2] = work[w].ke;
    o[3] = work[w].member_off;
    o[4] = work[w].n_members;
    o[5] = int32_t(part);
    o[6] = work[w].n_members * G;
    o[7] = work[w].grow;
    part += work[w].n_members;
  }
  std::memcpy(plan + info->off_members, members.data(), members.size() * sizeof(int32_t));
  int32_t* indptr = plan + info->off_req_part_indptr;
  int32_t* rp = plan + info->off_req_parts;
  indptr[0] = 0;
  for (int32_t b = 0; b < B; ++b) {
    std::memcpy(rp + indptr[b], parts_of[size_t(b)].data(),
                parts_of[size_t(b)].size() * sizeof(int32_t));
    indptr[b + 1] = indptr[b] + int32_t(parts_of[size_t(b)].size());
  }
  return RX_OK;
}

extern "C" rx_status rx_plan_decode(const rx_cache* c, int32_t B, const rx_node* prompt_node,
                                    const int32_t* ctx_len, const int32_t* req_rows,
                                    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                    int32_t* plan, int64_t plan_cap, rx_decode_plan_info* info) {
  return plan_decode_impl(c, B, 1, prompt_node, ctx_len, req_rows, num_q_heads, num_kv_heads,
                          head_dim, plan, plan_cap, info);
}

extern "C" rx_status rx_plan_decode_steps(const rx_cache* c, int32_t B, int32_t n_steps,
                                          const rx_node* prompt_node, const int32_t* ctx_len,
                                          const int32_t* req_rows, int32_t num_q_heads,
                                          int32_t num_kv_heads, int32_t head_dim, int32_t* plan,
                                          int64_t plan_cap, rx_decode_plan_info* info) {
  return plan_decode_impl(c, B, n_steps, prompt_node, ctx_len, req_rows, num_q_heads,
                          num_kv_heads, head_dim, plan, plan_cap, info);
}

extern "C" rx_status rx_alloc_steps(rx_cache* c, int64_t k, int32_t n_steps, int32_t* out_slots) {
  if (!c || k < 0 || n_steps < 0 || (!out_slots && k > 0 && n_steps > 0))
    return fail(RX_ERR_INVALID, "rx_alloc_steps: bad argument");
  if (c->ps != 1)
    return fail(RX_ERR_INVALID, "rx_alloc_steps: page_size %lld > 1; use rx_alloc_decode_steps",
                (long long)c->ps);
  for (int32_t t = 0; t < n_steps; ++t) {
    if (!c->alloc(k, out_slots + int64_t(t) * k))
      return fail(RX_ERR_NO_SPACE, "rx_alloc_steps: step %d: %lld slots requested, %lld free after eviction",
                  t, (long long)k, (long long)c->free_list.size());
  }
  return RX_OK;
}

extern "C" rx_status rx_alloc_decode_steps(rx_cache* c, int32_t B, int32_t n_steps,
                                          const int32_t* pos0, const int32_t* last_slot,
                                          int32_t* out_slots) {
  if (!c || B < 0 || n_steps < 0 || (B && n_steps && (!pos0 || !last_slot || !out_slots)))
    return fail(RX_ERR_INVALID, "rx_alloc_decode_steps: bad argument");
  std::vector<int32_t> pages(static_cast<size_t>(B));
  for (int32_t t = 0; t < n_steps; ++t) {
    int32_t* out = out_slots + int64_t(t) * B;
    const int32_t* prev = t ? out - B : last_slot;
    int64_t need = 0;
    for (int32_t b = 0; b < B; ++b) need += (int64_t(pos0[b]) + t) % c->ps == 0;
    if (!c->alloc_pages(need, pages.data()))
      return fail(RX_ERR_NO_SPACE,
                  "rx_alloc_decode_steps: step %d: %lld pages requested, %lld free after eviction",
                  t, (long long)need, (long long)c->free_list.size());
    int64_t k = 0;
    for (int32_t b = 0; b < B; ++b)
      out[b] = (int64_t(pos0[b]) + t) % c->ps == 0 ? int32_t(int64_t(pages[size_t(k++)]) * c->ps)
                                                   : prev[b] + 1;
  }
  return RX_OK;
}

extern "C" rx_status rx_extend_plan(const int32_t* qo_indptr, int32_t R, int32_t num_q_heads,
                                    int32_t num_kv_heads, int32_t head_dim,
                                    int32_t* tile_indptr, int64_t* out_num_tiles) {
  if (R < 0 || !qo_indptr || !tile_indptr || !out_num_tiles || num_kv_heads <= 0 ||
      num_q_heads % num_kv_heads != 0 || (head_dim != 128 && head_dim != 256))
    return fail(RX_ERR_INVALID, "rx_extend_plan: bad argument");
  const int64_t G = num_q_heads / num_kv_heads;
  const int64_t rows_per_tile = rx_internal::extend_rows_per_tile(head_dim);
  tile_indptr[0] = 0;
  for (int32_t r = 0; r < R; ++r) {
    int64_t s = qo_indptr[r + 1] - qo_indptr[r];
    if (s < 0) return fail(RX_ERR_INVALID, "rx_extend_plan: qo_indptr not monotone");
    int64_t t = (s * G + rows_per_tile - 1) / rows_per_tile;
    if (tile_indptr[r] + t > INT32_MAX) return fail(RX_ERR_INVALID, "rx_extend_plan: too many tiles");
    tile_indptr[r + 1] = int32_t(tile_indptr[r] + t);
  }
  *out_num_tiles = tile_indptr[R];
  return RX_OK;
}

namespace rx_internal {
rx_status set_error(rx_status s, const char* msg) { return fail(s, "%s", msg); }
}  // namespace rx_internal

// ---------------------------------------------------- cache-aware scheduling
// "SGLang: the tree, and the language nobody remembers", section "The
// scheduler is where the cache is won or lost".  A request's match (against
// the tree and against the queue tree) is taken on its prompt without the
// last token, in whole pages; sorts are stable.
namespace {

constexpr int64_t kInBatchCheck = 32;       // thin tree match: check the queue
constexpr int64_t kInBatchDeprioritize = 32;  // shares this much with the queue: wait
constexpr int32_t kLpmQueueLimit = 128;     // above: first come, first served

// The deepest node whose whole root path t[0..n) matches (n in whole pages).
const Node* hanging_node(const rx_cache* c, const int32_t* t, int64_t n) {
  n = c->aligned(n);
  const Node* node = c->root;
  int64_t pos = 0;
  while (pos < n) {
    const Node* ch = c->child_of(node, t + pos);
    if (!ch) break;
    const int64_t len = int64_t(ch->key.size());
    if (n - pos < len || common_prefix(ch->key.data(), t + pos, len) < len) break;
    pos += len;
    node = ch;
  }
  return node;
}

void lpm_order(const rx_cache* c, int32_t R, const int32_t* tokens, const int64_t* indptr,
               int32_t* out) {
  for (int32_t i = 0; i < R; ++i) out[i] = i;
  if (R > kLpmQueueLimit) return;
  // the simulated radix tree over the waiting queue (no slots of its own)
  rx_config qc{c->ps, int32_t(c->ps), 0};
  rx_cache* q = nullptr;
  rx_cache_create(&qc, &q);
  std::vector<int32_t> dummy;
  std::vector<std::pair<int64_t, int32_t>> keys(static_cast<size_t>(R));
  const int64_t kBack = INT64_MAX;
  for (int32_t i = 0; i < R; ++i) {
    const int32_t* p = tokens + indptr[i];
    const int64_t n = indptr[i + 1] - indptr[i];
    const int64_t m = c->match_length(p, n - 1);
    bool back = false;
    if (m <= kInBatchCheck) {
      if (q->match_length(p, n - 1) >= kInBatchDeprioritize) {
        back = true;
      } else {
        if (int64_t(dummy.size()) < n) dummy.resize(size_t(n), 0);
        int64_t already = 0;
        q->insert(p, dummy.data(), n, &already);
      }
    }
    keys[size_t(i)] = {back ? kBack : -m, i};
  }
  rx_cache_destroy(q);
  std::stable_sort(keys.begin(), keys.end(),
                   [](const std::pair<int64_t, int32_t>& a, const std::pair<int64_t, int32_t>& b) {
                     return a.first < b.first;
                   });
  for (int32_t i = 0; i < R; ++i) out[i] = keys[size_t(i)].second;
}

void dfs_weight_order(const rx_cache* c, int32_t R, const int32_t* tokens, const int64_t* indptr,
                      int32_t* out) {
  std::unordered_map<const Node*, std::vector<int32_t>> at;
  for (int32_t i = 0; i < R; ++i) {
    const int32_t* p = tokens + indptr[i];
    const int64_t n = indptr[i + 1] - indptr[i];
    at[hanging_node(c, p, n - 1)].push_back(i);
  }
  // subtree weights and earliest waiting request, children before parents
  std::unordered_map<const Node*, std::pair<int64_t, int32_t>> wf;  // weight, first
  std::vector<const Node*> order{c->root};
  for (size_t k = 0; k < order.size(); ++k)
    c->for_children(order[k], [&](const Node* ch) { order.push_back(ch); });
  for (size_t k = order.size(); k-- > 0;) {
    const Node* x = order[k];
    auto it = at.find(x);
    int64_t w = it == at.end() ? 0 : int64_t(it->second.size());
    int32_t f = it == at.end() ? R : it->second.front();
    c->for_children(x, [&](const Node* ch) {
      const auto& cw = wf[ch];
      w += cw.first;
      f = std::min(f, cw.second);
    });
    wf[x] = {w, f};
  }
  // depth first: a node's own requests, then heavier children first
  int32_t o = 0;
  std::vector<const Node*> stack{c->root};
  std::vector<const Node*> kids;
  while (!stack.empty()) {
    const Node* x = stack.back();
    stack.pop_back();
    auto it = at.find(x);
    if (it != at.end())
      for (int32_t i : it->second) out[o++] = i;
    kids.clear();
    c->for_children(x, [&](const Node* ch) {
      if (wf[ch].first > 0) kids.push_back(ch);
    });
    std::sort(kids.begin(), kids.end(), [&](const Node* a, const Node* b) {
      const auto& wa = wf[a];
      const auto& wb = wf[b];
      if (wa.first != wb.first) return wa.first > wb.first;
      return wa.second < wb.second;
    });
    for (size_t k = kids.size(); k-- > 0;) stack.push_back(kids[k]);
  }
}

}  // namespace

extern "C" rx_status rx_schedule(const rx_cache* c, int32_t policy, int32_t R,
                                 const int32_t* tokens, const int64_t* indptr,
                                 int32_t* out_order) {
  if (!c || R < 0 || (R && (!tokens || !indptr || !out_order)))
    return fail(RX_ERR_INVALID, "rx_schedule: bad argument");
  for (int32_t i = 0; i < R; ++i)
    if (indptr[i + 1] - indptr[i] < 1)
      return fail(RX_ERR_INVALID, "rx_schedule: empty prompt %d", i);
  switch (policy) {
    case RX_POLICY_FCFS:
      for (int32_t i = 0; i < R; ++i) out_order[i] = i;
      return RX_OK;
    case RX_POLICY_LPM:
      lpm_order(c, R, tokens, indptr, out_order);
      return RX_OK;
    case RX_POLICY_DFS_WEIGHT:
      dfs_weight_order(c, R, tokens, indptr, out_order);
      return RX_OK;
    default:
      return fail(RX_ERR_INVALID, "rx_schedule: unknown policy %d", policy);
  }
}

// --------------------------------------------------- draft-tree verification
// "SGLang: the tree, and the language nobody remembers", section
// "Speculative decoding puts a tree inside the tree": a draft token attends
// to the request's context and to its own ancestors in the draft tree (and
// itself).  Its slot-table row is the context's slots followed by the slots
// of its root path, so the decode kernels compute exactly the tree-masked
// attention over that row.
extern "C" rx_status rx_verify_rows(int32_t R, const int32_t* prefix_len,
                                    const int32_t* prefix_rows, int64_t prefix_stride,
                                    const int64_t* draft_indptr, const int32_t* parents,
                                    const int32_t* draft_slots, int32_t* out_rows,
                                    int64_t out_stride, int32_t* out_ctx_len,
                                    int32_t* out_positions) {
  if (R < 0 || (R && (!prefix_len || !prefix_rows || !draft_indptr || !out_rows ||
                      !out_ctx_len)) || prefix_stride < 0 || out_stride < 1)
    return fail(RX_ERR_INVALID, "rx_verify_rows: bad argument");
  std::vector<int32_t> depth, path;
  for (int32_t r = 0; r < R; ++r) {
    const int64_t b = draft_indptr[r], e = draft_indptr[r + 1];
    const int64_t p = prefix_len[r];
    if (e < b || p < 0 || p > prefix_stride)
      return fail(RX_ERR_INVALID, "rx_verify_rows: request %d: bad draft range or prefix", r);
    depth.assign(size_t(e - b), 0);
    for (int64_t i = b; i < e; ++i) {
      const int64_t li = i - b;
      const int32_t par = parents[i];
      if (par < -1 || par >= li)
        return fail(RX_ERR_INVALID, "rx_verify_rows: draft %lld: parent %d must precede it",
                    (long long)i, par);
      depth[size_t(li)] = par < 0 ? 0 : depth[size_t(par)] + 1;
      const int64_t ctx = p + depth[size_t(li)] + 1;
      if (ctx > out_stride)
        return fail(RX_ERR_INVALID, "rx_verify_rows: draft %lld needs %lld row entries, row has %lld",
                    (long long)i, (long long)ctx, (long long)out_stride);
      int32_t* row = out_rows + i * out_stride;
      std::memcpy(row, prefix_rows + int64_t(r) * prefix_stride, size_t(p) * sizeof(int32_t));
      path.clear();
      for (int64_t j = li; j >= 0; j = parents[b + j]) path.push_back(draft_slots[b + j]);
      for (size_t k = 0; k < path.size(); ++k) row[p + int64_t(k)] = path[path.size() - 1 - k];
      out_ctx_len[i] = int32_t(ctx);
      if (out_positions) out_positions[i] = int32_t(p + depth[size_t(li)]);
    }
  }
  return RX_OK;
}

// ------------------------------------------------------ two-tier transfers
// "SGLang: the tree, and the language nobody remembers", section "What the
// C++ tree is actually for": match across tiers with a node for each tier,
// write-through tickets committed later, load-onboard of host-resident nodes.
namespace {

// Host pages for the device-only nodes of node's root path; the path stays
// locked until the commit.  *ticket = 0 (nothing to copy) when the path is
// on the host already or a backup on it is in flight.
rx_status write_through_impl(rx_cache* c, Node* node, int32_t* out_dev, int32_t* out_host,
                             int64_t cap, int64_t* out_n, int64_t* out_ticket) {
  *out_n = 0;
  *out_ticket = 0;
  const std::vector<Node*> path = c->root_path(node);
  for (const Node* x : path)
    if (x->pending_ticket) return RX_OK;
  int64_t n = 0;
  for (const Node* x : path)
    if (!x->host) n += int64_t(x->key.size());
  if (n == 0) return RX_OK;
  if (n > cap)
    return fail(RX_ERR_INVALID, "rx_write_through: %lld tokens to copy, capacity %lld",
                (long long)n, (long long)cap);
  if (c->host_slots == 0) return fail(RX_ERR_NO_SPACE, "rx_write_through: no host tier");
  std::vector<int32_t> pages(static_cast<size_t>(n / c->ps));
  if (!c->host_alloc_pages(int64_t(pages.size()), pages.data()))
    return fail(RX_ERR_NO_SPACE, "rx_write_through: %lld host slots needed, %lld free",
                (long long)n, (long long)(int64_t(c->host_free.size()) * c->ps));
  const int64_t ticket = c->next_ticket++;
  int64_t pos = 0;
  for (Node* x : path) {
    if (x->host) continue;
    const int64_t len = int64_t(x->key.size());
    x->pending_ticket = ticket;
    x->pending_host.resize(size_t(len));
    c->page_slots(pages.data() + pos / c->ps, len, x->pending_host.data());
    std::memcpy(out_dev + pos, x->value.data(), size_t(len) * sizeof(int32_t));
    std::memcpy(out_host + pos, x->pending_host.data(), size_t(len) * sizeof(int32_t));
    pos += len;
  }
  c->lock(node);
  c->tickets[ticket] = node->id;
  *out_n = n;
  *out_ticket = ticket;
  return RX_OK;
}

rx_status commit_impl(rx_cache* c, int64_t ticket, bool success) {
  auto it = c->tickets.find(ticket);
  if (it == c->tickets.end())
    return fail(RX_ERR_INVALID, "rx_commit_write_through: unknown ticket %lld", (long long)ticket);
  Node* node = c->find(it->second);
  c->tickets.erase(it);
  for (Node* x = node; x != c->root; x = x->parent) {
    if (x->pending_ticket != ticket) continue;
    if (success) {
      x->host_value = std::move(x->pending_host);
      x->host = true;
      c->host_cached += int64_t(x->key.size());
    } else {
      for (size_t i = 0; i < x->pending_host.size(); i += size_t(c->ps))
        c->host_free.push_back(int32_t(x->pending_host[i] / c->ps));
    }
    x->pending_host.clear();
    x->pending_ticket = 0;
  }
  c->unlock(node);
  return RX_OK;
}

// Device pages for the host-only nodes of node's root path (the path's
// device part locked while allocating); they become resident on both tiers.
rx_status load_impl(rx_cache* c, Node* node, int32_t* out_host, int32_t* out_dev, int64_t cap,
                    int64_t* out_n) {
  *out_n = 0;
  const std::vector<Node*> path = c->root_path(node);
  int64_t n = 0;
  Node* dev_node = c->root;
  bool dev_run = true;
  for (Node* x : path) {
    if (x->gpu && dev_run) {
      dev_node = x;
    } else {
      dev_run = false;
      if (!x->gpu) n += int64_t(x->key.size());
    }
  }
  if (n == 0) return RX_OK;
  if (n > cap)
    return fail(RX_ERR_INVALID, "rx_load_onboard: %lld tokens to load, capacity %lld",
                (long long)n, (long long)cap);
  std::vector<int32_t> pages(static_cast<size_t>(n / c->ps));
  c->lock(dev_node);
  const bool ok = c->alloc_pages(int64_t(pages.size()), pages.data());
  c->unlock(dev_node);
  if (!ok)
    return fail(RX_ERR_NO_SPACE, "rx_load_onboard: %lld device slots needed, %lld free",
                (long long)n, (long long)(int64_t(c->free_list.size()) * c->ps));
  int64_t pos = 0;
  for (Node* x : path) {
    if (x->gpu) continue;
    const int64_t len = int64_t(x->key.size());
    x->value.resize(size_t(len));
    c->page_slots(pages.data() + pos / c->ps, len, x->value.data());
    x->gpu = true;
    c->evictable += len;
    c->cached += len;
    std::memcpy(out_host + pos, x->host_value.data(), size_t(len) * sizeof(int32_t));
    std::memcpy(out_dev + pos, x->value.data(), size_t(len) * sizeof(int32_t));
    pos += len;
  }
  *out_n = n;
  return RX_OK;
}

}  // namespace

extern "C" rx_status rx_match_prefix_tiers(rx_cache* c, const int32_t* tokens, int64_t n,
                                           int32_t* out_slots, int64_t* out_device_len,
                                           int64_t* out_host_len, rx_node* out_device_node,
                                           rx_node* out_host_node) {
  if (!c || (!tokens && n) || n < 0 || (!out_slots && n) || !out_device_len || !out_host_len ||
      !out_device_node || !out_host_node)
    return fail(RX_ERR_INVALID, "rx_match_prefix_tiers: bad argument");
  c->clock += 1;
  std::vector<Node*> path;
  int64_t all = 0;
  Node* dnode = c->root;
  Node* last = c->walk(tokens, n, &all, &path, out_slots, out_device_len, &dnode);
  for (Node* x : path) x->last_access_time = c->clock;
  *out_host_len = all - *out_device_len;
  *out_device_node = dnode->id;
  *out_host_node = last->id;
  return RX_OK;
}

extern "C" rx_status rx_load_onboard(rx_cache* c, rx_node node, int32_t* out_host_slots,
                                     int32_t* out_device_slots, int64_t cap, int64_t* out_n) {
  Node* x = c ? c->find(node) : nullptr;
  if (!x || !out_n || (cap && (!out_host_slots || !out_device_slots)))
    return fail(RX_ERR_INVALID, "rx_load_onboard: bad argument or unknown node");
  return load_impl(c, x, out_host_slots, out_device_slots, cap, out_n);
}

extern "C" rx_status rx_write_through(rx_cache* c, rx_node node, int32_t* out_device_slots,
                                      int32_t* out_host_slots, int64_t cap, int64_t* out_n,
                                      int64_t* out_ticket) {
  Node* x = c ? c->find(node) : nullptr;
  if (!x || !out_n || !out_ticket || (cap && (!out_device_slots || !out_host_slots)))
    return fail(RX_ERR_INVALID, "rx_write_through: bad argument or unknown node");
  for (Node* w = x; w != c->root; w = w->parent)
    if (!w->gpu) return fail(RX_ERR_STATE, "rx_write_through: path not on the device");
  return write_through_impl(c, x, out_device_slots, out_host_slots, cap, out_n, out_ticket);
}

extern "C" rx_status rx_commit_write_through(rx_cache* c, int64_t ticket, int32_t success) {
  if (!c) return fail(RX_ERR_INVALID, "rx_commit_write_through: NULL cache");
  return commit_impl(c, ticket, success != 0);
}

extern "C" rx_status rx_load_batch(rx_cache* c, int32_t R, const int32_t* tokens,
                                   const int64_t* indptr, int32_t* out_host_slots,
                                   int32_t* out_device_slots, int64_t cap, int64_t* out_n,
                                   int64_t* out_counts) {
  if (!c || R < 0 || !indptr || (R && (!tokens || !out_counts)) || !out_n)
    return fail(RX_ERR_INVALID, "rx_load_batch: bad argument");
  *out_n = 0;
  std::vector<Node*> path;
  for (int32_t r = 0; r < R; ++r) {
    out_counts[r] = 0;
    const int64_t n = indptr[r + 1] - indptr[r];
    if (n < 1) return fail(RX_ERR_INVALID, "rx_load_batch: empty prompt %d", r);
    c->clock += 1;
    path.clear();
    int64_t all = 0, dlen = 0;
    Node* dnode = c->root;
    Node* last = c->walk(tokens + indptr[r], n - 1, &all, &path, nullptr, &dlen, &dnode);
    for (Node* x : path) x->last_access_time = c->clock;
    if (all == dlen) continue;
    int64_t got = 0;
    const rx_status st = load_impl(c, last, out_host_slots + *out_n, out_device_slots + *out_n,
                                   cap - *out_n, &got);
    if (st == RX_ERR_NO_SPACE) continue;  // prefilled instead
    if (st != RX_OK) return st;
    out_counts[r] = got;
    *out_n += got;
  }
  return RX_OK;
}

extern "C" rx_status rx_write_through_batch(rx_cache* c, int32_t R, const rx_node* nodes,
                                            int32_t* out_device_slots, int32_t* out_host_slots,
                                            int64_t cap, int64_t* out_n, int64_t* out_counts) {
  if (!c || R < 0 || (R && (!nodes || !out_counts)) || !out_n)
    return fail(RX_ERR_INVALID, "rx_write_through_batch: bad argument");
  *out_n = 0;
  for (int32_t r = 0; r < R; ++r) {
    out_counts[r] = 0;
    Node* x = c->find(nodes[r]);
    if (!x) return fail(RX_ERR_INVALID, "rx_write_through_batch: unknown node %lld",
                        (long long)nodes[r]);
    int64_t got = 0, ticket = 0;
    const rx_status st = write_through_impl(c, x, out_device_slots + *out_n,
                                            out_host_slots + *out_n, cap - *out_n, &got, &ticket);
    if (st == RX_ERR_NO_SPACE) continue;  // the host tier cannot hold it: not backed up
    if (st != RX_OK) return st;
    if (ticket) commit_impl(c, ticket, true);
    out_counts[r] = got;
    *out_n += got;
  }
  return RX_OK;
}

extern "C" rx_status rx_host_eviction_log(const rx_cache* c, int64_t start, rx_evict_rec* out,
                                          int64_t cap, int64_t* out_total) {
  if (!c || start < 0 || cap < 0 || (cap && !out))
    return fail(RX_ERR_INVALID, "rx_host_eviction_log: bad argument");
  const int64_t total = int64_t(c->host_evict_log.size());
  for (int64_t i = 0; i < cap && start + i < total; ++i) out[i] = c->host_evict_log[start + i];
  if (out_total) *out_total = total;
  return RX_OK;
}

// Fault injection for tests: the k-th page allocation from now (device or
// host pool, counted together; k >= 1) fails with RX_ERR_NO_SPACE after the
// evictions it would do anyway, as if the pool were still short.  k = 0
// turns it off.
extern "C" rx_status rx_debug_fail_alloc(rx_cache* c, int64_t k) {
  if (!c || k < 0) return fail(RX_ERR_INVALID, "rx_debug_fail_alloc: bad argument");
  c->fail_countdown = k;
  return RX_OK;
}

// ------------------------------------------------------------- whole waves
// The in-batch rule's batch loop over a whole wave in one call: for each
// batch in turn rx_batch_end, rx_extend_begin, rx_extend_end, exactly as a
// caller making those calls batch by batch would ("SGLang: the tree, and the
// language nobody remembers", section "The overlap that pays for itself":
// the host decides slots ahead of the GPU, which needs only slot numbers).
extern "C" rx_status rx_extend_wave(rx_cache* c, int32_t R, const int32_t* tokens,
                                    const int64_t* indptr, int32_t* req_to_token,
                                    int64_t row_stride, int32_t* out_batch_end,
                                    int32_t* out_n_batches, int32_t* out_prefix_len,
                                    rx_node* out_prompt_node, int32_t* out_new_slots,
                                    int64_t* out_batch_rewritten) {
  if (!c || R < 0 || !indptr || !out_n_batches ||
      (R && (!tokens || !req_to_token || !out_batch_end || !out_prefix_len ||
             !out_prompt_node || !out_new_slots || !out_batch_rewritten)))
    return fail(RX_ERR_INVALID, "rx_extend_wave: bad argument");
  *out_n_batches = 0;
  std::vector<rx_node> match(static_cast<size_t>(R));
  int64_t new_off = 0;
  int32_t start = 0;
  while (start < R) {
    int32_t end = R;
    rx_status st = rx_batch_end(c, tokens, indptr, start, R, &end);
    if (st != RX_OK) return st;
    const int32_t n = end - start;
    int64_t total = 0;
    st = rx_extend_begin(c, n, tokens, indptr + start, req_to_token + int64_t(start) * row_stride,
                         row_stride, out_prefix_len + start, match.data() + start,
                         out_new_slots + new_off, &total);
    if (st != RX_OK) return st;
    new_off += total;
    int64_t rew = 0;
    st = rx_extend_end(c, n, tokens, indptr + start, req_to_token + int64_t(start) * row_stride,
                       row_stride, out_prefix_len + start, match.data() + start,
                       out_prompt_node + start, &rew);
    if (st != RX_OK) return st;
    out_batch_end[*out_n_batches] = end;
    out_batch_rewritten[*out_n_batches] = rew;
    *out_n_batches += 1;
    start = end;
  }
  return RX_OK;
}
