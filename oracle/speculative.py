"""Oracle of draft-tree verification over the KV pool and of KV moves.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Source: "SGLang: the tree, and the language nobody remembers", section
"Speculative decoding puts a tree inside the tree":

* the drafts of a request form a tree; each draft token attends only to its
  own ancestors (and, as every token does, to the request's context before
  the tree), so every branch is an independent continuation and one target
  forward pass verifies all of them;
* a draft token's position is the prompt length plus its depth in the tree
  (depths [0, 1, 1, 2] after a 7-token prompt give positions [7, 8, 8, 9]);
* the full mask holds one entry per (draft token, key): for a batch of ``bs``
  requests with ``num_verify`` draft tokens each, ``seq_lens_sum *
  num_verify + num_verify**2 * bs`` entries;
* the KV of the accepted path, written by the drafts into scattered slots,
  is moved to the slots the request's next positions use before the tree
  adopts it (``move_kv_cache(tgt, src)``).

Readings where the page is silent:

* a draft tree is given as parent indices: ``parents[i]`` is the draft token
  that ``i`` continues, or -1 when ``i`` continues the request's last
  verified token; parents come before their children;
* a draft token sees its ancestors and itself (the diagonal of the mask);
* a move reads every source row before it writes any target row.

Parity: pinned by ``tests/test_oracle_pins.py`` (the page's positions
example; a chain-shaped tree equals causal extend attention over prefix plus
drafts; a tree of depth-0 drafts equals independent decode attention of each
draft; the full mask's entry count against the page's formula; moves against
explicit copies).
"""

import numpy as np

from .attention import softmax_attention


def depths(parents):
    """Depth of every draft token (0 for a child of the verified token)."""
    out = []
    for i, p in enumerate(parents):
        if p >= i:
            raise ValueError("a parent must come before its child")
        out.append(0 if p < 0 else out[p] + 1)
    return out


def positions(prefix_len, parents):
    """Sequence position of every draft token: prefix length + depth."""
    return [prefix_len + d for d in depths(parents)]


def ancestors_and_self(parents, i):
    """Draft indices on the path from the tree's root to ``i``, root first."""
    path = []
    while i >= 0:
        path.append(i)
        i = parents[i]
    return path[::-1]


def tree_mask(prefix_len, parents):
    """Full mask of one request: bool [n, prefix_len + n]; row i is true on
    every prefix column and on the columns of i's ancestors and i."""
    n = len(parents)
    mask = np.zeros((n, prefix_len + n), dtype=bool)
    mask[:, :prefix_len] = True
    for i in range(n):
        for j in ancestors_and_self(parents, i):
            mask[i, prefix_len + j] = True
    return mask


def verify_attention(q, k_prefix, v_prefix, k_draft, v_draft, parents, scale=None):
    """Attention of every draft token under the tree mask, fp64.

    q: [n, Hq, d] draft queries; k_prefix, v_prefix: [p, Hkv, d] the
    request's context before the tree; k_draft, v_draft: [n, Hkv, d].
    Returns ``(o [n, Hq, d], lse [n, Hq])``.
    """
    n = len(parents)
    p = k_prefix.shape[0]
    mask = tree_mask(p, parents)
    keys = np.concatenate([k_prefix, k_draft])
    vals = np.concatenate([v_prefix, v_draft])
    o = np.zeros(q.shape, dtype=np.float64)
    lse = np.zeros(q.shape[:2], dtype=np.float64)
    for i in range(n):
        sel = np.nonzero(mask[i])[0]
        oi, li = softmax_attention(q[i:i + 1], keys[sel], vals[sel], [len(sel)], scale)
        o[i], lse[i] = oi[0], li[0]
    return o, lse


def move_kv(pool, tgt, src):
    """``pool[:, :, tgt[i], :] = pool[:, :, src[i], :]`` for every i, every
    layer and head, all sources read before any target is written."""
    out = np.array(pool, copy=True)
    rows = [np.array(pool[:, :, int(s), :], copy=True) for s in src]
    for t, r in zip(tgt, rows):
        out[:, :, int(t), :] = r
    return out
