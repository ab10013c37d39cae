"""GPU parity of draft-tree verification and KV moves/copies.

Verify attention runs through the C ABI (rx_verify_rows on the host, the
decode plan over the drafts, rx_kv_store of the drafts' K/V,
rx_verify_attention) and is compared with the fp64 oracle under the tree mask
(max-abs 1e-2, mean-abs 1e-3).  KV copies are compared bit for bit with the
oracle's move (within the pool) and with the source rows (between a device
pool and a page-locked host pool).
"""

import math
import random

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from oracle import speculative as ospec  # noqa: E402
from radix_tree_prefix_gb300 import rx  # noqa: E402

MAX_ABS, MEAN_ABS = 1e-2, 1e-3


def _rand_tree(rng, n, shape):
    if shape == "chain":
        return list(range(-1, n - 1))
    if shape == "star":
        return [-1] * n
    return [rng.randrange(-1, i) if i else -1 for i in range(n)]


def _bf16(g, shape, dev):
    return torch.randn(shape, generator=g, device=dev).to(torch.bfloat16)


@pytest.mark.parametrize("d,hq,hkv,n_req,shape", [
    (128, 32, 8, 3, "random"), (128, 32, 8, 2, "chain"), (128, 8, 8, 4, "star"),
    (256, 16, 4, 3, "random"), (128, 64, 8, 5, "random")])
def test_verify_attention_matches_oracle(d, hq, hkv, n_req, shape):
    """Requests that share a system prompt (one tree segment for every draft
    of every request) and have their own continuations, each verifying a
    draft tree: every draft's output equals tree-masked fp64 attention."""
    dev = torch.device("cuda:0")
    rng = random.Random(d + hq + n_req)
    g = torch.Generator(device=dev).manual_seed(7)
    system = [rng.randrange(1, 30000) for _ in range(300)]
    prompts = [system + [rng.randrange(1, 30000) for _ in range(rng.randint(1, 90))]
               for _ in range(n_req)]
    trees = [_rand_tree(rng, rng.randint(1, 40), shape) for _ in range(n_req)]
    N = sum(len(t) for t in trees)
    cache = rx.RadixCache(20000)
    nodes, rows_p, prefix_len = [], [], []
    for p in prompts:
        slots, _ = cache.match_prefix(p)
        row = np.concatenate([slots, cache.alloc(len(p) - len(slots))]).astype(np.int32)
        _, node = cache.insert(p, row)
        cache.lock(node)
        nodes.append(node)
        rows_p.append(row)
        prefix_len.append(len(p))
    stride = max(prefix_len)
    prefix_rows = np.zeros((n_req, stride), dtype=np.int32)
    for r, row in enumerate(rows_p):
        prefix_rows[r, :len(row)] = row
    draft_slots = cache.alloc(N)
    indptr = np.cumsum([0] + [len(t) for t in trees]).astype(np.int64)
    parents = np.concatenate([np.array(t, dtype=np.int32) for t in trees])
    out_stride = stride + 41
    rows, ctx, pos = rx.verify_rows(prefix_len, prefix_rows, indptr, parents, draft_slots,
                                    out_stride)
    # K/V of every context token (by slot) and of every draft; queries of drafts
    N_slots = cache.num_slots
    kp = torch.zeros((1, hkv, N_slots, d), dtype=torch.bfloat16, device=dev)
    vp = torch.zeros_like(kp)
    pool = rx.pool_desc(kp, vp)
    ctx_slots = sorted({int(s) for row in rows_p for s in row})
    ks = _bf16(g, (len(ctx_slots), hkv, d), dev)
    vs = _bf16(g, (len(ctx_slots), hkv, d), dev)
    rx.kv_store(pool, 0, torch.tensor(ctx_slots, dtype=torch.int32, device=dev), ks, vs)
    kd = _bf16(g, (N, hkv, d), dev)
    vd = _bf16(g, (N, hkv, d), dev)
    rx.kv_store(pool, 0, torch.from_numpy(draft_slots.copy()).to(dev), kd, vd)
    q = _bf16(g, (N, hq, d), dev)
    req_of = np.repeat(np.arange(n_req), [len(t) for t in trees])
    plan, info = cache.plan_decode([nodes[r] for r in req_of], ctx, np.arange(N), hq, hkv, d)
    assert info.n_shared_segments >= 1
    d_plan = torch.from_numpy(plan[:int(info.plan_words)].copy()).to(dev)
    d_table = torch.from_numpy(rows).to(dev)
    ws = torch.empty(int(info.workspace_bytes) + 256, dtype=torch.uint8, device=dev)
    out = torch.empty((N, hq, d), dtype=torch.float32, device=dev)
    lse = torch.empty((N, hq), dtype=torch.float32, device=dev)
    rx.verify_attention(pool, 0, q, hq, d_table, d_plan, info, N, 1.0 / math.sqrt(d), out, lse, ws)
    torch.cuda.synchronize()
    assert rx.device_check() == 0
    kpos = {s: i for i, s in enumerate(ctx_slots)}
    K = ks.double().cpu().numpy()
    V = vs.double().cpu().numpy()
    errs = []
    for r, tree in enumerate(trees):
        idx = [kpos[int(s)] for s in rows_p[r]]
        sl = slice(indptr[r], indptr[r + 1])
        wo, wl = ospec.verify_attention(q[sl].double().cpu().numpy(), K[idx], V[idx],
                                        kd[sl].double().cpu().numpy(),
                                        vd[sl].double().cpu().numpy(), tree)
        errs.append(np.abs(out[sl].double().cpu().numpy() - wo).ravel())
        errs.append(np.abs(lse[sl].double().cpu().numpy() - wl).ravel())
        assert pos[sl].tolist() == ospec.positions(prefix_len[r], tree)
    e = np.concatenate(errs)
    assert e.max() <= MAX_ABS and e.mean() <= MEAN_ABS, (e.max(), e.mean())


@pytest.mark.parametrize("d,L,hkv", [(128, 2, 8), (256, 3, 4)])
def test_move_within_pool_matches_oracle(d, L, hkv):
    """The accepted path's KV moved to the request's next slots, every layer
    and head: bit for bit the oracle's move; other rows untouched."""
    dev = torch.device("cuda:0")
    g = torch.Generator(device=dev).manual_seed(d + L)
    N = 3000
    kp = _bf16(g, (L, hkv, N, d), dev)
    vp = _bf16(g, (L, hkv, N, d), dev)
    perm = torch.randperm(N - 1, generator=g, device=dev) + 1
    src, tgt = perm[:700].to(torch.int32), perm[700:1400].to(torch.int32)
    want_k = ospec.move_kv(kp.float().cpu().numpy(), tgt.cpu().numpy(), src.cpu().numpy())
    want_v = ospec.move_kv(vp.float().cpu().numpy(), tgt.cpu().numpy(), src.cpu().numpy())
    pool = rx.pool_desc(kp, vp)
    rx.kv_copy(pool, pool, src, tgt)
    torch.cuda.synchronize()
    assert rx.device_check() == 0
    assert np.array_equal(kp.float().cpu().numpy(), want_k)
    assert np.array_equal(vp.float().cpu().numpy(), want_v)


def test_copy_to_host_pool_and_back():
    """Rows copied from the device pool into a page-locked host pool (read
    and written by the kernel directly), then into a second device pool at
    other slots: bit for bit the source rows."""
    dev = torch.device("cuda:0")
    g = torch.Generator(device=dev).manual_seed(3)
    L, hkv, d, N, H = 2, 4, 256, 2000, 900
    kp = _bf16(g, (L, hkv, N, d), dev)
    vp = _bf16(g, (L, hkv, N, d), dev)
    hk = torch.zeros((L, hkv, H, d), dtype=torch.bfloat16, pin_memory=True)
    hv = torch.zeros_like(hk).pin_memory()
    k2 = torch.zeros_like(kp)
    v2 = torch.zeros_like(vp)
    src = (torch.randperm(N - 1, generator=g, device=dev)[:500] + 1).to(torch.int32)
    mid = (torch.randperm(H - 1, generator=g, device=dev)[:500] + 1).to(torch.int32)
    dst = (torch.randperm(N - 1, generator=g, device=dev)[:500] + 1).to(torch.int32)
    dev_pool, host_pool, dev2 = rx.pool_desc(kp, vp), rx.pool_desc(hk, hv), rx.pool_desc(k2, v2)
    rx.kv_copy(dev_pool, host_pool, src, mid)
    rx.kv_copy(host_pool, dev2, mid, dst)
    torch.cuda.synchronize()
    assert rx.device_check() == 0
    s, m, t = src.long().cpu(), mid.long().cpu(), dst.long().cpu()
    assert torch.equal(hk[:, :, m], kp[:, :, s.to(dev)].cpu())
    assert torch.equal(hv[:, :, m], vp[:, :, s.to(dev)].cpu())
    assert torch.equal(k2[:, :, t.to(dev)], kp[:, :, s.to(dev)])
    assert torch.equal(v2[:, :, t.to(dev)], vp[:, :, s.to(dev)])


def test_copy_refuses_pageable_host_memory_and_skips_bad_slots():
    """A pageable host pool is refused before any launch; a slot outside
    its pool is skipped on the device and reported (bit 5)."""
    dev = torch.device("cuda:0")
    kp = torch.zeros((1, 1, 64, 128), dtype=torch.bfloat16, device=dev)
    host = torch.zeros((1, 1, 64, 128), dtype=torch.bfloat16)          # pageable
    one = torch.ones(1, dtype=torch.int32, device=dev)
    with pytest.raises(rx.RxError) as e:
        rx.kv_copy(rx.pool_desc(kp, kp), rx.pool_desc(host, host), one, one)
    assert e.value.status == rx.RX_ERR_INVALID
    vp = torch.ones_like(kp)
    bad = torch.tensor([70, 3], dtype=torch.int32, device=dev)
    dst = torch.tensor([5, 6], dtype=torch.int32, device=dev)
    rx.kv_copy(rx.pool_desc(vp, vp), rx.pool_desc(kp, kp), bad, dst)
    torch.cuda.synchronize()
    with pytest.raises(rx.RxError) as e:
        rx.device_check()
    assert "(flags 32)" in str(e.value)
    assert int((kp[0, 0, 5] != 0).sum()) == 0 and int((kp[0, 0, 6] != 0).sum()) == 128
