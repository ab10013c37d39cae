"""rx_decode_attention_static: decode attention with the library's own fixed
scratch array, for callers that cannot provide device memory (for example a
host whose device memory is all reserved by its own pool, or a plugin given a
stream and tensors but no allocator).

The test builds a small decode batch by itself (cache, pool, table, plan),
runs the regular entry point with a caller-owned workspace, then the static
entry point twice in a row (the second time on a different batch, so a stale
array from the first call would show), and checks that each result equals the
regular one bit for bit (and so lies within the tolerance the other GPU tests
use).  The file is named
so that pytest collects it last.
"""

import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from radix_tree_prefix_gb300 import rx, workloads  # noqa: E402

MAX_ABS = 1e-2
MEAN_ABS = 1e-3


def _decode_batch(wl, dev, extra):
    """Cache + pool holding every prompt and `extra` decode tokens per request."""
    cache = rx.RadixCache(wl.num_slots + len(wl.requests) * 8)
    vals = workloads.make_values(wl, dev)
    reqs = wl.waves[0]
    B = len(reqs)
    width = max(len(wl.prompt_tokens(r)) for r in reqs) + extra
    table = np.zeros((B, width), dtype=np.int32)
    nodes, ctx, slots_all, store_all = [], [], [], []
    for b, r in enumerate(reqs):
        toks = wl.prompt_tokens(r)
        slots, _ = cache.match_prefix(toks)
        new = cache.alloc(len(toks) - len(slots))
        row = np.concatenate([slots, new]).astype(np.int32)
        _, node = cache.insert(toks, row)
        cache.lock(node)
        dec = cache.alloc(extra)
        full = np.concatenate([row, dec])
        table[b, :len(full)] = full
        nodes.append(node)
        ctx.append(len(full))
        sidx = np.concatenate([wl.prompt_store_index(r), wl.output_store_index(r)[:extra]])
        keep = np.concatenate([np.arange(len(slots), len(full))])
        slots_all.append(full[keep])
        store_all.append(sidx[keep])
    hkv, d, hq = wl.num_kv_heads, wl.head_dim, wl.num_q_heads
    kp = torch.zeros((1, hkv, cache.num_slots, d), dtype=torch.bfloat16, device=dev)
    vp = torch.zeros_like(kp)
    pool = rx.pool_desc(kp, vp)
    sl = torch.from_numpy(np.concatenate(slots_all)).to(dev)
    si = torch.from_numpy(np.concatenate(store_all).astype(np.int64)).to(dev)
    rx.kv_store(pool, 0, sl, vals["k"][0].index_select(0, si), vals["v"][0].index_select(0, si))
    plan, info = cache.plan_decode(nodes, ctx, list(range(B)), hq, hkv, d)
    d_plan = torch.from_numpy(plan[:int(info.plan_words)].copy()).to(dev)
    d_table = torch.from_numpy(table).to(dev)
    qi = torch.from_numpy(np.array([wl.output_store_index(r)[extra - 1] for r in reqs],
                                   dtype=np.int64)).to(dev)
    q = vals["q"][0].index_select(0, qi).contiguous()
    return dict(cache=cache, kp=kp, vp=vp, pool=pool, plan=d_plan, info=info, table=d_table,
                q=q, B=B, hq=hq, d=d)


def _run(batch, static):
    out = torch.empty((batch["B"], batch["hq"], batch["d"]), dtype=torch.float32,
                      device=batch["q"].device)
    lse = torch.empty((batch["B"], batch["hq"]), dtype=torch.float32, device=batch["q"].device)
    scale = 1.0 / math.sqrt(batch["d"])
    if static:
        rx.decode_attention_static(batch["pool"], 0, batch["q"], batch["hq"], batch["table"],
                                   batch["plan"], batch["info"], batch["B"], scale, out, lse)
    else:
        ws = torch.empty(int(batch["info"].workspace_bytes) + 256, dtype=torch.uint8,
                         device=batch["q"].device)
        rx.decode_attention(batch["pool"], 0, batch["q"], batch["hq"], batch["table"],
                            batch["plan"], batch["info"], batch["B"], scale, out, lse, ws)
    torch.cuda.synchronize()
    return out, lse


def _close(a, b):
    # Both entry points run the same kernels on the same plan and inputs, and
    # each partial result is written to a place the plan fixes, so the static
    # scratch must give the workspace path's outputs bit for bit (a stale or
    # misplaced scratch region would show here).  The attention tolerance is
    # checked as well, as in the other GPU tests.
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    err = torch.cat([(a[0] - b[0]).abs().flatten(), (a[1] - b[1]).abs().flatten()])
    assert float(err.max()) <= MAX_ABS and float(err.mean()) <= MEAN_ABS


def test_static_scratch_decode_matches_workspace_decode():
    dev = torch.device("cuda:0")
    first = _decode_batch(workloads.agent_loop(calls=9, preamble=400, lo=30, hi=120,
                                               decode_steps=4), dev, 4)
    second = _decode_batch(workloads.long_shared(batch=5, prefix=700, unique=90,
                                                 decode_steps=3, q_heads=16, kv_heads=8),
                           dev, 3)
    assert second["info"].workspace_bytes <= rx.RX_DECODE_STATIC_SCRATCH_BYTES
    want1 = _run(first, static=False)
    want2 = _run(second, static=False)
    got1 = _run(first, static=True)      # first call on this device: set-up
    _close(got1, want1)
    got2 = _run(second, static=True)     # second call in a row, other batch
    _close(got2, want2)
    assert rx.device_check() == 0


def test_static_scratch_rejects_oversized_plan():
    info = rx.rx_decode_plan_info()
    info.workspace_bytes = rx.RX_DECODE_STATIC_SCRATCH_BYTES + 1
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda:0")
    kp = torch.zeros((1, 1, 8, 128), dtype=torch.bfloat16, device="cuda:0")
    with pytest.raises(rx.RxError) as e:
        rx.decode_attention_static(rx.pool_desc(kp, kp), 0, kp, 1, dummy.view(1, 16), dummy,
                                   info, 1, 1.0, kp, kp)
    assert e.value.status == rx.RX_ERR_INVALID and "static scratch" in str(e.value)
