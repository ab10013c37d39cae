"""Oracle attention: fp64 naive softmax attention over a request's full context.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

What the method computes, per the pages:

* "SGLang: Structured LLM Programs for Efficient Inference", section "A quick
  recap of how an LLM generates text": during decode each new token attends
  over the KV cache and its own keys and values are appended; the KV of a
  token depends only on that token and the ones before it.
* same page, section "How RadixAttention reuses past work", step 3: only the
  unmatched suffix is prefilled, attending to the reused entries as if they
  had just been computed.

So the result a radix cache must reproduce is plain causal softmax attention
over each request's whole token sequence, as if the whole prompt had been
recomputed.  This module computes exactly that from the per-token Q/K/V the
caller passes in; it never looks at a cache.

Readings (the pages give no attention formula): scores are ``q . k * scale``
with ``scale = 1/sqrt(d)``; a query at position ``i`` sees keys ``0 .. i``
(itself included); query head ``h`` reads KV head ``h // G`` with
``G = Hq / Hkv``; outputs are fp32-representable fp64 values plus the natural
log-sum-exp of the scaled scores.

Parity: pinned by closed forms in ``tests/test_oracle_pins.py`` (a single key
returns its value row; two keys with score gap ``ln 3`` weigh 1/4 and 3/4;
equal keys average the visible values, which fixes the causal boundary; a
constant-per-KV-head value fixes the GQA head mapping) and by the log-sum-exp
split identity.
"""

import math

import numpy as np


def softmax_attention(q, k, v, visible, scale=None):
    """Causal GQA attention, one query at a time, in fp64.

    q:       [nq, Hq, d]   queries
    k, v:    [n, Hkv, d]   keys and values of the whole context
    visible: [nq] ints     query ``i`` sees keys ``0 .. visible[i]-1``
    Returns ``(o [nq, Hq, d], lse [nq, Hq])``.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    nq, hq, d = q.shape
    hkv = k.shape[1]
    if hq % hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    group = hq // hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = np.zeros((nq, hq, d), dtype=np.float64)
    lse = np.zeros((nq, hq), dtype=np.float64)
    for i in range(nq):
        n_vis = int(visible[i])
        if n_vis < 1:
            raise ValueError("a query must see at least one key")
        for h in range(hq):
            kv_head = h // group
            keys = k[:n_vis, kv_head, :]
            vals = v[:n_vis, kv_head, :]
            scores = keys @ q[i, h] * scale
            m = scores.max()
            p = np.exp(scores - m)
            total = p.sum()
            o[i, h] = (p @ vals) / total
            lse[i, h] = m + math.log(total)
    return o, lse


def extend_attention(q_suffix, k_full, v_full, prefix_len, scale=None):
    """Suffix queries of one request against its prefix plus causal suffix.

    q_suffix: [s, Hq, d] queries of tokens ``prefix_len .. prefix_len+s-1``;
    k_full, v_full: [prefix_len + s, Hkv, d] the request's whole context.
    """
    s = q_suffix.shape[0]
    visible = [prefix_len + i + 1 for i in range(s)]
    return softmax_attention(q_suffix, k_full, v_full, visible, scale)


def decode_attention(q_token, k_full, v_full, scale=None):
    """One decode token (whose K/V is the last context row) over its context.

    q_token: [Hq, d]; k_full, v_full: [n, Hkv, d] including the token itself.
    Returns ``(o [Hq, d], lse [Hq])``.
    """
    n = k_full.shape[0]
    o, lse = softmax_attention(q_token[None], k_full, v_full, [n], scale)
    return o[0], lse[0]


def lse_merge(parts):
    """Combine partial attention results over disjoint key sets.

    ``parts`` is a list of ``(o [.., d], lse [..])`` each normalised over its
    own key subset.  Returns the result over the union:
    ``lse = log sum exp(lse_s)``, ``o = sum exp(lse_s - lse) * o_s``.
    """
    lses = np.stack([np.asarray(p[1], dtype=np.float64) for p in parts])
    m = lses.max(axis=0)
    w = np.exp(lses - m)
    total = w.sum(axis=0)
    lse = m + np.log(total)
    o = sum(w[i][..., None] * np.asarray(parts[i][0], dtype=np.float64)
            for i in range(len(parts))) / total[..., None]
    return o, lse
