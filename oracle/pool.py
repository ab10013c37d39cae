"""Oracle KV pool store: the definition of writing a token's K/V to its slot.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

"SGLang: Structured LLM Programs for Efficient Inference", section "A quick
recap of how an LLM generates text": each computed token's keys and values are
stored in the KV cache.  With a pool laid out ``[layer][kv_head][slot][d]`` the
store of token ``i`` at ``slots[i]`` is ``pool[layer, h, slots[i], :] =
kv[i, h, :]`` for every head ``h``.

Parity: pinned by ``tests/test_oracle_pins.py`` (stores then reads back rows
by slot; distinct slots leave every other row untouched).
"""

import numpy as np


def store(pool, layer, slots, kv):
    """Return a copy of ``pool`` with ``kv[i]`` written at ``slots[i]``."""
    out = np.array(pool, copy=True)
    for i, s in enumerate(slots):
        for h in range(kv.shape[1]):
            out[layer, h, int(s), :] = kv[i, h, :]
    return out
