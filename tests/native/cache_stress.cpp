// Randomised stress of the host radix cache through its C ABI, built with
// AddressSanitizer and UndefinedBehaviorSanitizer by tests/test_sanitizers.py.
// Every call of the host cache is exercised (match, lock, alloc, insert,
// evict, free, pages, batch steps, whole-wave extends, decode planning,
// scheduling, the two tiers, draft rows, fault injection) on small pools so that eviction, splits and
// page boundaries are frequent; after every operation the cache's counts must
// agree: evictable + protected == cached.  Any memory error or undefined
// behaviour aborts the run through the sanitizers.
//
// usage: cache_stress <seed> <iterations>

#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <random>
#include <vector>

#include "rx.h"

namespace {

int fails = 0;

void check_counts(rx_cache* c, const char* where) {
  rx_stats_t st{};
  if (rx_stats(c, &st) != RX_OK) {
    std::printf("rx_stats failed at %s\n", where);
    ++fails;
    return;
  }
  if (st.evictable_tokens + st.protected_tokens != st.cached_tokens ||
      st.evictable_tokens < 0 || st.protected_tokens < 0 || st.free_slots < 0) {
    std::printf("counts disagree at %s: evictable %lld protected %lld cached %lld\n", where,
                (long long)st.evictable_tokens, (long long)st.protected_tokens,
                (long long)st.cached_tokens);
    ++fails;
  }
}

}  // namespace

int main(int argc, char** argv) {
  const unsigned seed = argc > 1 ? unsigned(std::atoi(argv[1])) : 1u;
  const int iters = argc > 2 ? std::atoi(argv[2]) : 2000;
  std::mt19937 rng(seed);
  auto uni = [&](int lo, int hi) { return std::uniform_int_distribution<int>(lo, hi)(rng); };

  for (int trial = 0; trial < 12; ++trial) {
    const int ps = trial % 3 == 0 ? 1 : (trial % 3 == 1 ? 2 : 4);
    rx_config cfg{};
    cfg.num_slots = int64_t(ps) * uni(16, 64);
    cfg.page_size = ps;
    cfg.host_slots = trial % 2 ? int64_t(ps) * uni(8, 48) : 0;
    rx_cache* c = nullptr;
    if (rx_cache_create(&cfg, &c) != RX_OK) return 2;
    std::vector<rx_node> locked;
    std::vector<int64_t> tickets;
    std::vector<int32_t> slots(4096), slots2(4096), plan(1 << 16);
    for (int it = 0; it < iters / 12; ++it) {
      const int n = uni(1, 14);
      std::vector<int32_t> t(static_cast<size_t>(n));
      for (auto& x : t) x = uni(0, 2);
      const int op = uni(0, 16);
      int64_t len = 0, already = 0, hl = 0, got = 0, tk = 0;
      rx_node node = 0, node2 = 0, hn = 0;
      switch (op) {
        case 0:
        case 1:
        case 2: {  // request: (load) match, lock, alloc, insert, move lock
          if (cfg.host_slots) {
            rx_match_prefix_tiers(c, t.data(), n - 1, slots.data(), &len, &hl, &node, &hn);
            if (hl) rx_load_onboard(c, hn, slots2.data(), slots.data(), 4096, &got);
          }
          rx_match_prefix(c, t.data(), n - 1, slots.data(), &len, &node);
          rx_lock(c, node);
          if (rx_alloc(c, n - len, slots.data() + len) != RX_OK) {
            rx_unlock(c, node);
            break;
          }
          rx_insert(c, t.data(), slots.data(), n, &already, &node2);
          // free the part already cached and the partly filled page
          const int64_t al = n - n % ps;
          if (already > len) rx_free(c, slots.data() + len, already - len);
          if (al < n) rx_free(c, slots.data() + al, 1);
          if (rx_lock(c, node2) == RX_OK) locked.push_back(node2);
          rx_unlock(c, node);
          break;
        }
        case 3:
          if (!locked.empty()) {
            const size_t i = size_t(uni(0, int(locked.size()) - 1));
            rx_unlock(c, locked[i]);
            locked.erase(locked.begin() + long(i));
          }
          break;
        case 4: {
          int64_t freed = 0;
          rx_evict(c, uni(1, 12), &freed);
          break;
        }
        case 5:
          if (!locked.empty() && cfg.host_slots) {
            if (rx_write_through(c, locked.back(), slots.data(), slots2.data(), 4096, &got, &tk) ==
                    RX_OK &&
                tk)
              tickets.push_back(tk);
          }
          break;
        case 6:
          if (!tickets.empty()) {
            rx_commit_write_through(c, tickets.back(), uni(0, 3) != 0);
            tickets.pop_back();
          }
          break;
        case 7: {  // scheduling over a small queue
          std::vector<int32_t> toks;
          std::vector<int64_t> ind{0};
          const int R = uni(1, 6);
          for (int r = 0; r < R; ++r) {
            const int m = uni(1, 12);
            for (int k = 0; k < m; ++k) toks.push_back(uni(0, 2));
            ind.push_back(int64_t(toks.size()));
          }
          std::vector<int32_t> order(static_cast<size_t>(R));
          rx_schedule(c, uni(0, 2), R, toks.data(), ind.data(), order.data());
          int32_t end = 0;
          rx_batch_end(c, toks.data(), ind.data(), 0, R, &end);
          std::vector<int32_t> hs(512), ds(512);
          std::vector<int64_t> cnt(static_cast<size_t>(R));
          if (cfg.host_slots)
            rx_load_batch(c, R, toks.data(), ind.data(), hs.data(), ds.data(), 512, &got,
                          cnt.data());
          break;
        }
        case 8:
          if (!locked.empty()) {  // decode plan over the locked requests
            std::vector<int32_t> ctx, rows;
            for (size_t i = 0; i < locked.size(); ++i) {
              int64_t d = 0;
              rx_node_depth(c, locked[i], &d);
              ctx.push_back(int32_t(d + 2));
              rows.push_back(int32_t(i));
            }
            rx_decode_plan_info info{};
            rx_plan_decode_steps(c, int32_t(locked.size()), 3, locked.data(), ctx.data(),
                                 rows.data(), 8, 2, 128, plan.data(), int64_t(plan.size()), &info);
          }
          break;
        case 9: {  // decode slots of two requests that own one page each
          std::vector<int32_t> own(size_t(2 * ps)), out(size_t(3) * 2);
          if (rx_alloc(c, 2 * ps, own.data()) != RX_OK) break;
          // request 0 has filled ps - 1 positions of its page, request 1 all ps
          const int32_t pos0[2] = {ps - 1, ps};
          const int32_t last[2] = {ps > 1 ? own[size_t(ps - 2)] : 0, own[size_t(2 * ps - 1)]};
          if (rx_alloc_decode_steps(c, 2, 3, pos0, last, out.data()) == RX_OK) {
            // the new pages (slots past the two owned pages)
            std::vector<int32_t> fresh;
            for (int32_t x : out)
              if (x / ps != own[0] / ps && x / ps != own[size_t(ps)] / ps) fresh.push_back(x);
            if (!fresh.empty()) rx_free(c, fresh.data(), int64_t(fresh.size()));
          }
          rx_free(c, own.data(), int64_t(own.size()));
          break;
        }
        case 10:
          rx_debug_fail_alloc(c, uni(0, 3));
          break;
        case 11: {  // draft rows
          const int32_t pl[1] = {3};
          const int32_t pr[4] = {ps, ps + 1, ps + 2, 0};
          const int64_t di[2] = {0, 4};
          const int32_t par[4] = {-1, 0, 0, 1};
          const int32_t ds[4] = {9, 10, 11, 12};
          std::vector<int32_t> rows(4 * 8), ctx(4), pos(4);
          rx_verify_rows(1, pl, pr, 4, di, par, ds, rows.data(), 8, ctx.data(), pos.data());
          break;
        }
        case 12: {  // a whole wave's extend bookkeeping, then its locks released
          std::vector<int32_t> toks;
          std::vector<int64_t> ind{0};
          const int R = uni(1, 5);
          for (int r = 0; r < R; ++r) {
            const int m = uni(1, 10);
            for (int k = 0; k < m; ++k) toks.push_back(uni(0, 2));
            ind.push_back(int64_t(toks.size()));
          }
          std::vector<int32_t> table(static_cast<size_t>(R) * 10), ends(static_cast<size_t>(R)),
              pre(static_cast<size_t>(R)), fresh(toks.size());
          std::vector<rx_node> nodes(static_cast<size_t>(R));
          std::vector<int64_t> rew(static_cast<size_t>(R));
          int32_t nb = 0;
          if (rx_extend_wave(c, R, toks.data(), ind.data(), table.data(), 10, ends.data(), &nb,
                             pre.data(), nodes.data(), fresh.data(), rew.data()) == RX_OK) {
            for (int r = 0; r < R; ++r) {
              // the partly filled last page stays with the request: free it
              const int64_t n = ind[size_t(r) + 1] - ind[size_t(r)];
              if (n % ps) rx_free(c, table.data() + size_t(r) * 10 + (n - n % ps), 1);
              rx_unlock(c, nodes[size_t(r)]);
            }
          } else {
            for (int32_t b = 0, r = 0; b < nb; ++b)
              for (; r < ends[size_t(b)]; ++r) rx_unlock(c, nodes[size_t(r)]);
          }
          break;
        }
        default: {
          int64_t ml = 0;
          rx_match_length(c, t.data(), n, &ml);
          if (ml > n) {
            std::printf("match length %lld > %d\n", (long long)ml, n);
            ++fails;
          }
          break;
        }
      }
      check_counts(c, "after an operation");
    }
    for (int64_t tkt : tickets) rx_commit_write_through(c, tkt, 1);
    for (rx_node x : locked) rx_unlock(c, x);
    check_counts(c, "after unlocking");
    rx_stats_t st{};
    rx_stats(c, &st);
    if (st.protected_tokens != 0) {
      std::printf("protected tokens left: %lld\n", (long long)st.protected_tokens);
      ++fails;
    }
    rx_cache_destroy(c);
  }
  std::printf("cache_stress seed %u: %d failures\n", seed, fails);
  return fails ? 1 : 0;
}
