"""Mutation check of the oracle's pins.

Each case copies the oracle (with the pins, their fixtures and the input
generator) into a scratch directory, plants one plausible mistake in the copy
by a text substitution, and runs ``tests/test_oracle_pins.py`` there.  At
least one pin must fail for every planted mistake; an unmutated copy must
pass.  Every substitution must match the oracle's source exactly once, so a
change to the oracle that makes a mutation inapplicable fails here too.

The mistakes cover the cache (heap order, split attributes, the cascade
condition, allocator order, access times, lock paths, eviction candidates,
page alignment of keys, matches and child keys),
the request flow (in-batch rule, what is matched, adoption of identical
prompts, what finish inserts and frees, decode tokens kept out of the tree,
lock release), the scheduler (LPM direction, the in-batch thresholds, the
queue-length switch, the depth-first weights and order) and attention (scale,
GQA head, causal boundary, log-sum-exp).

Not planted: a split that does not copy the lower node's access time to the
upper one.  Splits happen only inside a match or an insert, and both write
the new clock on every node of the path they walk, the upper node included,
so that inherited value is overwritten in the same call and no result can
depend on it.
"""

import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# name -> (oracle file, [(exact text, replacement), ...])
MUTANTS = {
    "eviction_heap_most_recent_first": ("radix_cache.py", [
        ("heap = [(n.priority, n.last_access_time, n.id, n)",
         "heap = [(n.priority, -n.last_access_time, n.id, n)"),
        ("heapq.heappush(heap, (parent.priority, parent.last_access_time,",
         "heapq.heappush(heap, (parent.priority, -parent.last_access_time,")]),
    "split_forgets_lock_ref": ("radix_cache.py", [
        ("        upper.lock_ref = node.lock_ref\n", "")]),
    "cascade_pushes_parent_with_children": ("radix_cache.py", [
        ("if (parent is not self.root and not parent.children\n"
         "                    and parent.lock_ref == 0):",
         "if parent is not self.root and parent.lock_ref == 0:")]),
    "no_cascade": ("radix_cache.py", [
        ("if (parent is not self.root and not parent.children\n"
         "                    and parent.lock_ref == 0):",
         "if False:")]),
    "allocator_lifo": ("radix_cache.py", [
        ("return [self.free_pages.popleft() for _ in range(n)]",
         "return [self.free_pages.pop() for _ in range(n)]")]),
    "match_does_not_touch": ("radix_cache.py", [
        ("        for n in path:\n            n.last_access_time = self.clock\n"
         "        return slots, node",
         "        return slots, node")]),
    "evicted_slots_reversed": ("radix_cache.py", [
        ("for s in victim.value[::self.page_size])",
         "for s in victim.value[::-self.page_size])")]),
    "evicted_pages_keep_only_first": ("radix_cache.py", [
        ("for s in victim.value[::self.page_size])",
         "for s in victim.value[:1])")]),
    "lock_only_the_node": ("radix_cache.py", [
        ("            node.lock_ref += 1\n            node = node.parent",
         "            node.lock_ref += 1\n            break")]),
    "match_does_not_split": ("radix_cache.py", [
        ("            if k < len(child.key):\n                child = self._split(child, k)\n"
         "            slots.extend(child.value)\n",
         "            if k < len(child.key):\n                slots.extend(child.value[:k])\n"
         "                pos += k\n                break\n            slots.extend(child.value)\n")]),
    "locked_leaves_evictable": ("radix_cache.py", [
        ("for n in self._leaves() if n.lock_ref == 0]", "for n in self._leaves()]")]),
    "lock_keeps_evictable_count": ("radix_cache.py", [
        ("            if node.lock_ref == 0:\n                self.evictable_size_ -= len(node.key)\n",
         "            if node.lock_ref == 0:\n")]),
    "scale_doubled": ("attention.py", [
        ("scale = 1.0 / math.sqrt(d)", "scale = 2.0 / math.sqrt(d)")]),
    "gqa_head_modulo": ("attention.py", [
        ("kv_head = h // group", "kv_head = h % hkv")]),
    "causal_excludes_self": ("attention.py", [
        ("visible = [prefix_len + i + 1 for i in range(s)]",
         "visible = [prefix_len + i + (i == 0) for i in range(s)]")]),
    "lse_without_max": ("attention.py", [
        ("lse[i, h] = m + math.log(total)", "lse[i, h] = math.log(total)")]),
    "merge_lse_without_max": ("attention.py", [
        ("lse = m + np.log(total)", "lse = np.log(total)")]),
    "store_into_layer_0": ("pool.py", [
        ("out[layer, h, int(s), :] = kv[i, h, :]", "out[0, h, int(s), :] = kv[i, h, :]")]),
    "finish_drops_outputs": ("harness.py", [
        ("already, full_node = cache.insert(full, rows[rid])",
         "already, full_node = cache.insert(list(prompt), rows[rid][:len(prompt)])")]),
    "decode_tokens_inserted_each_step": ("harness.py", [
        ("            for (rid, _, _), s in zip(wave, slots):\n"
         "                rows[rid].append(s)\n",
         "            for (rid, p_, o_), s in zip(wave, slots):\n"
         "                rows[rid].append(s)\n"
         "                cache.insert(list(p_) + list(o_[:step + 1]), rows[rid])\n")]),
    "finish_keeps_duplicate_slots": ("harness.py", [
        ("            if already > cache.aligned(len(prompt)):\n"
         "                cache.free(rows[rid][cache.aligned(len(prompt)):already])\n", "")]),
    "finish_keeps_partial_page": ("harness.py", [
        ("                cache.free(rows[rid][cache.aligned(len(full)):])\n",
         "                pass\n")]),
    "match_not_rounded_to_pages": ("radix_cache.py", [
        ("            k = self.aligned(common_prefix_length(child.key, tokens[pos:]))\n"
         "            if k < len(child.key):\n                child = self._split(child, k)\n"
         "            slots.extend(child.value)",
         "            k = common_prefix_length(child.key, tokens[pos:])\n"
         "            if k < len(child.key):\n                child = self._split(child, k)\n"
         "            slots.extend(child.value)")]),
    "insert_keeps_partial_page": ("radix_cache.py", [
        ("        n = self.aligned(len(tokens))\n", "        n = len(tokens)\n")]),
    "children_keyed_on_first_token": ("radix_cache.py", [
        ("        if self.page_size == 1:\n            return tokens[pos]\n",
         "        if True:\n            return tokens[pos]\n")]),
    "decode_page_not_started": ("harness.py", [
        ("need = [len(rows[rid]) % ps == 0 for rid, _, _ in wave]",
         "need = [len(rows[rid]) % ps == 1 % ps for rid, _, _ in wave]")]),
    "in_batch_rule_unrounded": ("harness.py", [
        ("if batch and any(cache.aligned(common_prefix_length(prompt, wave_prompts[i])) > m",
         "if batch and any(common_prefix_length(prompt, wave_prompts[i]) > m")]),
    "no_adoption_of_identical_prompt": ("harness.py", [
        ("                if already > m:\n"
         "                    tree = cache.lookup_slots(prompts[j])[m:already]\n"
         "                    cache.free(rows[rid][m:already])\n"
         "                    rows[rid][m:already] = tree\n", "")]),
    "no_in_batch_rule": ("harness.py", [
        ("        if batch and any(", "        if False and any(")]),
    "lpm_shortest_prefix_first": ("scheduler.py", [
        ("keys.append((float(\"inf\") if deprioritised else -m, i))",
         "keys.append((float(\"inf\") if deprioritised else m, i))")]),
    "in_batch_deprioritise_strictly_above": ("scheduler.py", [
        (">= IN_BATCH_DEPRIORITIZE_THRESHOLD:", "> IN_BATCH_DEPRIORITIZE_THRESHOLD:")]),
    "in_batch_check_strictly_below": ("scheduler.py", [
        ("if m <= IN_BATCH_CHECK_THRESHOLD:", "if m < IN_BATCH_CHECK_THRESHOLD:")]),
    "in_batch_queue_never_filled": ("scheduler.py", [
        ("                queued.append(list(p))\n", "                pass\n")]),
    "lpm_limit_inclusive": ("scheduler.py", [
        ("if n > LPM_QUEUE_LIMIT:", "if n >= LPM_QUEUE_LIMIT:")]),
    "dfs_lighter_children_first": ("scheduler.py", [
        ("kids.sort(key=lambda c: (-weight[c.id], first[c.id]))",
         "kids.sort(key=lambda c: (weight[c.id], first[c.id]))")]),
    "dfs_own_requests_last": ("scheduler.py", [
        ("        out.extend(at.get(node.id, []))\n        kids = [",
         "        kids = [")]),
    "draft_mask_without_diagonal": ("speculative.py", [
        ("        path.append(i)\n        i = parents[i]\n",
         "        i = parents[i]\n        if i >= 0:\n            path.append(i)\n")]),
    "draft_path_without_root": ("speculative.py", [
        ("    while i >= 0:\n", "    while i >= 0 and parents[i] >= 0:\n")]),
    "draft_depth_from_one": ("speculative.py", [
        ("out.append(0 if p < 0 else out[p] + 1)", "out.append(1 if p < 0 else out[p] + 1)")]),
    "move_writes_before_reads": ("speculative.py", [
        ("    rows = [np.array(pool[:, :, int(s), :], copy=True) for s in src]\n"
         "    for t, r in zip(tgt, rows):\n        out[:, :, int(t), :] = r\n",
         "    for t, s in zip(tgt, src):\n        out[:, :, int(t), :] = out[:, :, int(s), :]\n")]),
    "tier_eviction_drops_host_copy": ("hicache.py", [
        ("            if self.on_host(victim):\n                victim.value = None\n",
         "            if False:\n                victim.value = None\n")]),
    "tier_match_counts_host_as_device": ("hicache.py", [
        ("            if self.on_gpu(n) and host_len == 0:", "            if host_len == 0:")]),
    "tier_failed_commit_keeps_backup": ("hicache.py", [
        ("                if success:\n                    x.host_value = x.pending[1]\n",
         "                if True:\n                    x.host_value = x.pending[1]\n")]),
    "tier_host_eviction_ignores_children": ("hicache.py", [
        ("                if n is not self.root and not self.on_gpu(n) and self.on_host(n)\n"
         "                and not n.children]",
         "                if n is not self.root and not self.on_gpu(n) and self.on_host(n)]")]),
    "tier_insert_skips_host_only_nodes": ("hicache.py", [
        ("                x.value = slots[off:off + len(x.key)]\n",
         "                pass\n")]),
    "tier_device_leaf_ignores_host_children": ("hicache.py", [
        ("        return [c for c in node.children.values() if self.on_gpu(c)]",
         "        return list(node.children.values())")]),
    "dfs_weight_without_subtree": ("scheduler.py", [
        ("            w += cw\n", "")]),
    "match_whole_prompt": ("harness.py", [
        ("slots, node = cache.match_prefix(prompts[j][:len(prompts[j]) - 1])",
         "slots, node = cache.match_prefix(prompts[j])")]),
    "matched_lock_never_released": ("harness.py", [
        ("                cache.inc_lock_ref(node2)\n                cache.dec_lock_ref(node)\n",
         "                cache.inc_lock_ref(node2)\n")]),
}


def _copy(dst):
    """The pins and everything they import, under dst."""
    shutil.copytree(os.path.join(ROOT, "oracle"), os.path.join(dst, "oracle"),
                    ignore=shutil.ignore_patterns("__pycache__"))
    os.makedirs(os.path.join(dst, "tests"))
    for f in ("conftest.py", "test_oracle_pins.py"):
        shutil.copy(os.path.join(ROOT, "tests", f), os.path.join(dst, "tests", f))
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), os.path.join(dst, "tests", "golden"))
    pkg = os.path.join(dst, "radix_tree_prefix_gb300")
    os.makedirs(pkg)
    for f in ("__init__.py", "workloads.py"):
        shutil.copy(os.path.join(ROOT, "radix_tree_prefix_gb300", f), os.path.join(pkg, f))
    shutil.copy(os.path.join(ROOT, "pytest.ini"), os.path.join(dst, "pytest.ini"))


def _run_pins(d):
    env = dict(os.environ)
    env.pop("PYTHONPATH", None)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        "tests/test_oracle_pins.py"], cwd=d, env=env, capture_output=True,
                       text=True, timeout=600)
    return r.returncode, r.stdout + r.stderr


def test_unmutated_copy_passes_every_pin(tmp_path):
    _copy(str(tmp_path))
    rc, out = _run_pins(str(tmp_path))
    assert rc == 0, out[-3000:]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_fails_a_pin(name, tmp_path):
    fname, edits = MUTANTS[name]
    _copy(str(tmp_path))
    path = os.path.join(str(tmp_path), "oracle", fname)
    with open(path) as f:
        src = f.read()
    for old, new in edits:
        assert src.count(old) == 1, f"{name}: text to mutate not found once in {fname}"
        src = src.replace(old, new)
    with open(path, "w") as f:
        f.write(src)
    rc, out = _run_pins(str(tmp_path))
    # 1 = tests ran and at least one failed (not a collection or usage error)
    assert rc == 1, f"{name}: no pin failed (exit {rc})\n{out[-2000:]}"
