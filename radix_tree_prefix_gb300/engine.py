"""Request flow over librx: extend batches, decode steps and finish.

This drives the native calls in the order the pages give ("SGLang: Structured
LLM Programs for Efficient Inference", section "How RadixAttention reuses past
work": match the longest prefix, lock it, prefill only the rest, decode and
insert, release) with the in-batch prefix rule of "SGLang: the tree, and the
language nobody remembers", section "The scheduler is where the cache is won
or lost" (a request sharing more with a queued batch member than with the
tree waits for that member to populate the tree).

Every cache decision is taken by the C++ library and every tensor operation
of the method by the CUDA kernels; this module only moves arrays between
them.  Per wave of requests:

* extend: ``rx_extend_wave`` makes the bookkeeping of every extend batch of
  the wave in one native call (consecutive requests join the open batch
  until one shares more with a member than its own tree match; per batch:
  match, lock, one allocation, then insert of the prompt and the lock moved
  to the prompt's node); one staged upload carries every batch's
  req_to_token rows and tile plans; then per layer ``rx_extend_batches``
  launches, batch group by batch group, ``rx_kv_store`` and
  ``rx_extend_attention`` on one stream (with a host tier or chunked
  prefill the per-batch calls ``rx_batch_end`` / ``rx_extend_begin`` /
  ``rx_extend_end`` are used instead);
* decode: the wave's ``decode_steps`` steps are allocated at once
  (``rx_alloc_steps``; ``rx_alloc_decode_steps`` with pages), appended to
  the device rows (``rx_req_to_token_write``) and planned once
  (``rx_plan_decode_steps``: the tree does not change while the wave
  decodes); per layer ``rx_decode_steps`` runs every step (new token's K/V
  stored, attention over shared segments and private tails, log-sum-exp
  merge);
* finish: ``rx_finish`` (insert prompt + outputs, unlock).
"""

import ctypes
import math

import numpy as np

from . import rx


def launch_groups(rewritten):
    """Launch groups of a wave's nb extend batches, as batch boundaries
    [0, .., nb]: a group ends after a batch whose rows rx_extend_end
    rewrote (``rewritten[b] > 0``), and at the wave's last batch."""
    nb = len(rewritten)
    return [0] + [b + 1 for b in range(nb - 1) if rewritten[b] > 0] + [nb]


def cut_per_group(x, go):
    """``x``: R + 1 prefix sums over a wave's requests; ``go``: the groups'
    request boundaries [0, .., R].  Returns every group's R_g + 1 entries,
    rebased to start at 0, concatenated (group g's at position go[g] + g)."""
    cnt = np.diff(go) + 1
    first = np.repeat(np.cumsum(cnt) - cnt, cnt)
    idx = np.repeat(go[:-1], cnt) + (np.arange(int(cnt.sum())) - first)
    return x[idx] - np.repeat(x[go[:-1]], cnt)


class Trace:
    """The bookkeeping decisions, in the same form as the oracle's trace."""

    def __init__(self):
        self.batches = []
        self.decode_steps = []
        self.finishes = []
        self.prefilled = 0
        self.eviction_log = []
        self.stats = {}
        self.loads = []          # per load from the host tier: (rid, host slots, device slots)
        self.backups = []        # per written-through sequence: (rid, device slots, host slots)
        self.host_eviction_log = []

    def as_tuple(self):
        steps = []
        for rec in self.decode_steps:
            steps.extend(rec.steps())
        t = lambda a: tuple(int(x) for x in a)
        return (
            [[(rid, m, tuple(int(x) for x in row)) for rid, m, row in b] for b in self.batches],
            steps,
            list(self.finishes),
            self.prefilled,
            list(self.eviction_log),
            [(rid, t(h), t(d)) for rid, h, d in self.loads],
            [(rid, t(d), t(h)) for rid, d, h in self.backups],
            list(self.host_eviction_log),
        )


class _DecodeRecord:
    """Slots of every decode step of a wave, kept as arrays until compared."""

    def __init__(self, rids, slots):
        self.rids = rids
        self.slots = slots

    def steps(self):
        return [[(int(r), int(x)) for r, x in zip(self.rids, row)] for row in self.slots]


class GatherInputs:
    """Q/K/V of the tokens a batch computes, gathered from seeded stores."""

    def __init__(self, wl, values, layers):
        import torch
        self.torch = torch
        self.wl = wl
        self.values = values
        self.layers = list(layers)
        dev = next(iter(values["k"].values())).device
        self.device = dev

    def _idx(self, idx):
        return self.torch.from_numpy(np.ascontiguousarray(idx, dtype=np.int64)).to(self.device)

    def extend(self, batch_no, reqs, prefix):
        idx = np.concatenate([self.wl.prompt_store_index(r)[int(m):]
                              for r, m in zip(reqs, prefix)])
        ti = self._idx(idx)
        return {layer: (self.values["q"][layer].index_select(0, ti),
                        self.values["k"][layer].index_select(0, ti),
                        self.values["v"][layer].index_select(0, ti)) for layer in self.layers}

    def decode_wave(self, step0, reqs, T):
        """Q/K/V of the new tokens of T decode steps of a wave, [T][B][heads][d]
        per layer (step t, request b: the token at output position t)."""
        idx = np.array([[self.wl.output_store_index(r)[t] for r in reqs] for t in range(T)],
                       dtype=np.int64).reshape(-1)
        ti = self._idx(idx)
        B = len(reqs)

        def rows(kind, layer):
            x = self.values[kind][layer].index_select(0, ti)
            return x.view(T, B, *x.shape[1:])
        return {layer: (rows("q", layer), rows("k", layer), rows("v", layer))
                for layer in self.layers}


class HostBuffer:
    """Page-locked host memory of an exact size.  By default it comes from
    the library (``rx_host_alloc``: cudaHostAlloc, mapped into the device
    address space); with ``mode="register"`` it is a numpy array registered
    with CUDA (cudaHostRegister).  Copies from and to it run asynchronously,
    without the power-of-two rounding of the framework's pinned-memory
    cache.  ``tensor`` views it as uint8; ``close`` releases it."""

    def __init__(self, nbytes, mode="alloc"):
        import torch
        self.torch = torch
        self.nbytes = max(1, int(nbytes))
        self.mode = mode
        self.ptr = None
        self.array = None
        if mode == "alloc":
            self.ptr = rx.host_alloc(self.nbytes)
            buf = (ctypes.c_uint8 * self.nbytes).from_address(self.ptr)
            self.tensor = torch.frombuffer(buf, dtype=torch.uint8)
        else:
            self.array = np.empty(self.nbytes, dtype=np.uint8)
            err = torch._C._cudart.cudaHostRegister(self.array.ctypes.data, self.nbytes, 0)
            if int(getattr(err, "value", err)) != 0:
                raise RuntimeError(f"cudaHostRegister failed: {err}")
            self.tensor = torch.from_numpy(self.array)

    def view(self, offset, shape, dtype):
        n = int(np.prod(shape)) * _itemsize(dtype)
        return self.tensor[offset:offset + n].view(dtype).view(shape)

    def close(self):
        if self.tensor is None:
            return
        self.tensor = None
        if self.ptr is not None:
            rx.host_free(self.ptr)
            self.ptr = None
        elif self.array is not None:
            self.torch._C._cudart.cudaHostUnregister(self.array.ctypes.data)
            self.array = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _itemsize(dtype):
    import torch
    return torch.empty(0, dtype=dtype).element_size()


def _layout(per_layer):
    """Offsets (256-byte aligned) of a position's tensors packed in one flat
    buffer: [(layer, [(offset, shape, dtype), ...]), ...] and the total."""
    off = 0
    out = []
    for layer, qkv in per_layer.items():
        ents = []
        for t in qkv:
            ents.append((off, tuple(t.shape), t.dtype))
            off += (t.numel() * t.element_size() + 255) // 256 * 256
        out.append((layer, ents))
    return out, off


class PreparedInputs:
    """Inputs gathered once (by a recording run) and replayed in order.

    ``source`` is any provider; the first pass records what it returns per
    extend batch and per decode wave, later passes replay it.  ``host=True``
    keeps the recorded tensors in page-locked host memory and copies them to
    the device when they are used (the end-to-end path): when the engine asks
    for one batch's inputs, the next batch's (in the recorded order) are
    already being copied on a side stream, so the copies overlap the kernels.
    The device side is a ring of ``ring`` flat buffers, each as large as the
    largest position, filled in turn, and the ``ring - 1`` positions after the
    one handed out are kept in flight: a buffer is refilled once the work that
    read its previous occupant on the consumer's stream (everything the
    consumer had enqueued when it asked for the position after that one) has
    completed."""

    def __init__(self, source, host=False, ring=3):
        self.source = source
        self.host = host
        self.ring = max(2, int(ring))
        self.ext = {}
        self.dec = {}
        self.order = []        # (store, key) in the order a run asks for them
        self.recording = True
        self.h2d_bytes = 0
        self._pos = 0
        self._ahead = []       # [(position, event: its copy landed, views, buffer)]
        self._copy_stream = None
        self._dev = {}         # ring slot -> flat device buffer
        self._last_use = {}    # ring slot -> event after its last reader
        self._handed = None    # ring buffer of the position handed out last
        self._seq = 0          # ring buffers filled so far
        self._host_bufs = []
        self._lay = {}         # position -> (layout, bytes)

    def adopt(self, other):
        """Replay what `other` recorded (same order and tensors)."""
        self.ext, self.dec, self.order = dict(other.ext), dict(other.dec), list(other.order)

    def freeze(self):
        self.recording = False
        if not self.host:
            return
        import torch
        # one exact-size page-locked buffer per position, filled from the
        # recorded tensors; the recorded device tensors are then dropped
        for pos, (name, key) in enumerate(self.order):
            if pos in self._lay:            # frozen before
                continue
            store = self.ext if name == "ext" else self.dec
            per_layer = store[key]
            lay, nbytes = _layout(per_layer)
            hb = HostBuffer(nbytes)
            self._host_bufs.append(hb)
            host = {}
            for layer, ents in lay:
                views = []
                for (off, shape, dtype), t in zip(ents, per_layer[layer]):
                    h = hb.view(off, shape, dtype)
                    h.copy_(t)
                    views.append(h)
                host[layer] = tuple(views)
            store[key] = host
            self._lay[pos] = (lay, nbytes)
        torch.cuda.synchronize()
        self._slot_bytes = max((b for _, b in self._lay.values()), default=0)

    def close(self):
        for hb in self._host_bufs:
            hb.close()
        self._host_bufs = []

    def _fill(self, pos, slot, stream):
        """Copies position pos's recorded inputs into ring buffer `slot` on
        `stream`, after that buffer's previous readers."""
        import torch
        name, key = self.order[pos]
        src = (self.ext if name == "ext" else self.dec)[key]
        buf = self._dev.get(slot)
        if buf is None:
            buf = torch.empty(max(1, self._slot_bytes), dtype=torch.uint8,
                              device=self.source.device)
            self._dev[slot] = buf
        ev = self._last_use.get(slot)
        if ev is not None:
            stream.wait_event(ev)
        lay, _ = self._lay[pos]
        out = {}
        with torch.cuda.stream(stream):
            for (layer, ents) in lay:
                views = []
                for (off, shape, dtype), h in zip(ents, src[layer]):
                    n = h.numel() * h.element_size()
                    d = buf[off:off + n].view(dtype).view(shape)
                    d.copy_(h, non_blocking=True)
                    self.h2d_bytes += n
                    views.append(d)
                out[layer] = tuple(views)
        return out

    def _next_slot(self):
        # consecutive fills take consecutive ring buffers, so a buffer is
        # refilled only after `ring - 1` other positions were handed out
        slot = self._seq % self.ring
        self._seq += 1
        return slot

    def _get(self, name, store, key, make):
        if self.recording:
            store[key] = make()
            self.order.append((name, key))
            return store[key]
        if not self.host:
            return store[key]
        import torch
        cur = torch.cuda.current_stream(self.source.device)
        if self._handed is not None:
            # the consumer has enqueued all its work on the previous position
            ev = self._last_use.get(self._handed)
            if ev is None:
                ev = self._last_use[self._handed] = torch.cuda.Event()
            ev.record(cur)
        pos = self._pos
        if self.order[pos] != (name, key):     # not the recorded order: start over
            pos = self.order.index((name, key))
            self._ahead = []
        if self._ahead and self._ahead[0][0] == pos:
            _, ready, out, slot = self._ahead.pop(0)
            cur.wait_event(ready)
        else:
            self._ahead = []
            slot = self._next_slot()
            out = self._fill(pos, slot, cur)
        self._handed = slot
        self._pos = (pos + 1) % len(self.order)
        # keep the next ring - 1 positions in flight on the copy stream
        if self._copy_stream is None:
            self._copy_stream = torch.cuda.Stream(self.source.device)
        nxt = (self._ahead[-1][0] + 1) % len(self.order) if self._ahead else self._pos
        while len(self._ahead) < self.ring - 1:
            nslot = self._next_slot()
            views = self._fill(nxt, nslot, self._copy_stream)
            ready = torch.cuda.Event()
            ready.record(self._copy_stream)
            self._ahead.append((nxt, ready, views, nslot))
            nxt = (nxt + 1) % len(self.order)
        return out

    def extend(self, batch_no, reqs, prefix):
        return self._get("ext", self.ext, batch_no,
                         lambda: self.source.extend(batch_no, reqs, prefix))

    def decode_wave(self, step0, reqs, T):
        return self._get("dec", self.dec, step0,
                         lambda: self.source.decode_wave(step0, reqs, T))


class OutputRing:
    """Attention outputs of the end-to-end path, read back to the host
    through a bounded ring: ``slots`` device buffers paired with as many
    page-locked host buffers, each as large as the largest launch's output
    and lse.  ``take(shape)`` hands out the next pair's device tensors; the
    one handed out before it is then complete on the consumer's stream, so
    its device-to-host copy is issued on a side stream, and the kernel that
    writes a buffer next waits for that copy.  ``flush()`` issues the last
    copy.  The host buffers keep only the latest outputs of each slot: a
    reader that wants every output consumes them as they land."""

    def __init__(self, device, max_elems, slots=4):
        import torch
        self.torch = torch
        self.device = device
        self.slots = int(slots)
        self.cap = int(max_elems)
        self.dev = [torch.empty(self.cap, dtype=torch.float32, device=device)
                    for _ in range(self.slots)]
        self.host = [HostBuffer(self.cap * 4) for _ in range(self.slots)]
        self.copied = [None] * self.slots     # event: slot's last copy done
        self.stream = torch.cuda.Stream(device)
        self.pending = None                   # (slot, o elems, lse elems)
        self.i = 0
        self.d2h_bytes = 0

    def _retire(self, cur):
        if self.pending is None:
            return
        slot, no, nl = self.pending
        self.pending = None
        written = self.torch.cuda.Event()
        written.record(cur)
        self.stream.wait_event(written)
        n = no + nl
        with self.torch.cuda.stream(self.stream):
            self.host[slot].view(0, (n,), self.torch.float32).copy_(self.dev[slot][:n],
                                                                    non_blocking=True)
        ev = self.torch.cuda.Event()
        ev.record(self.stream)
        self.copied[slot] = ev
        self.d2h_bytes += 4 * n

    def take(self, shape, cur):
        no = int(np.prod(shape))
        nl = int(np.prod(shape[:-1]))
        if no + nl > self.cap:
            raise ValueError(f"output of {no + nl} values exceeds the ring's {self.cap}")
        self._retire(cur)
        slot = self.i
        self.i = (self.i + 1) % self.slots
        if self.copied[slot] is not None:
            cur.wait_event(self.copied[slot])
        buf = self.dev[slot]
        self.pending = (slot, no, nl)
        return buf[:no].view(shape), buf[no:no + nl].view(shape[:-1])

    def flush(self, cur):
        self._retire(cur)

    def close(self):
        for h in self.host:
            h.close()


def total_new_bytes(T, wl):
    """Bytes of the K (or V) rows of T tokens of one layer (bf16)."""
    return T * wl.num_kv_heads * wl.head_dim * 2


class _DevSpan:
    """A span of int32 values in a staging buffer on the device: the part of a
    tensor the librx binding reads (data_ptr, numel, shape), without the cost
    of making a tensor view per array."""

    __slots__ = ("ptr", "n", "shape")

    def __init__(self, ptr, n, shape=None):
        self.ptr, self.n = ptr, n
        self.shape = (n,) if shape is None else shape

    def data_ptr(self):
        return self.ptr

    def numel(self):
        return self.n


class _Staging:
    """Host->device uploads through a ring of pinned buffers.

    Each upload packs int32 arrays into one pinned buffer and issues a single
    asynchronous copy on the engine's stream; a ring slot's pinned buffer is
    refilled only after its previous copy has completed (event), so the host
    never blocks on the GPU in the common case.  Device-side reuse of a slot
    is ordered by the stream itself."""

    def __init__(self, torch, device, stream, explicit, n=4):
        self.torch, self.device, self.stream = torch, device, stream
        self.explicit = explicit    # False: ``stream`` is the current stream
        self.host = [None] * n
        self.host_np = [None] * n
        self.dev = [None] * n
        self.events = [torch.cuda.Event() for _ in range(n)]
        self.used = [False] * n
        self.i = 0

    def upload(self, arrays, as_tensors=False):
        """Device spans (or, with as_tensors, tensor views) of the arrays."""
        torch = self.torch
        n = sum(len(a) for a in arrays)
        i = self.i
        self.i = (i + 1) % len(self.host)
        if self.used[i]:
            self.events[i].synchronize()
        if self.host[i] is None or self.host[i].numel() < n:
            cap = max(2 * n, 1 << 21)
            self.host[i] = torch.empty(cap, dtype=torch.int32, pin_memory=True)
            self.host_np[i] = self.host[i].numpy()
            self.dev[i] = torch.empty(cap, dtype=torch.int32, device=self.device)
        h = self.host_np[i]
        off = 0
        spans = []
        for a in arrays:
            k = len(a)
            h[off:off + k] = a
            spans.append((off, k))
            off += k
        stream = self.stream
        if self.explicit:
            with torch.cuda.stream(stream):
                self.dev[i][:n].copy_(self.host[i][:n], non_blocking=True)
        else:
            self.dev[i][:n].copy_(self.host[i][:n], non_blocking=True)
        self.events[i].record(stream)
        self.used[i] = True
        d = self.dev[i]
        if as_tensors:
            return [d[o:o + k] for o, k in spans]
        base = d.data_ptr()
        return [_DevSpan(base + 4 * o, k) for o, k in spans]


class Engine:
    """Runs a workload through librx.

    ``device=None`` runs the host bookkeeping only (no CUDA).  With a device,
    ``inputs`` supplies the Q/K/V of computed tokens (``extend`` per batch,
    ``decode_wave`` for all decode steps of a wave) and ``on_extend`` /
    ``on_decode`` receive the attention outputs per layer, per batch and per
    decode step; ``on_decode_wave`` receives a wave's decode outputs at once
    ([T][B] tensors per layer).  Every copy and
    launch goes to ``stream``; left as None it is the device's current stream
    when the engine is made, which must then stay current while it runs.
    With ``reuse_outputs`` the output tensors of each extend batch and decode
    wave (per layer) are allocated on the first run and written again by
    every later run: they stay valid until the next run starts, and whoever
    reads them on another stream must be done (e.g. synchronized) by then.
    ``policy`` ("fcfs", "lpm" or "dfs-weight") orders each wave's waiting
    requests before every extend batch (``rx_schedule``).  ``chunk_tokens``
    (chunked prefill, "SGLang: Structured LLM Programs for Efficient
    Inference", section "How the runtime and frontend work together") cuts an
    extend batch's queries into launches of at most that many query tokens,
    in query order: a request's suffix may span several chunks, and a chunk's
    part of it attends over the prefix plus the suffix tokens before it.
    ``host_slots`` > 0 adds a host tier ("SGLang: the tree, and the language
    nobody remembers", section "What the C++ tree is actually for"): a
    page-locked host pool of that many slots; before each extend batch the
    members' prefixes resident on the host only are loaded back into the
    device pool (``rx_load_batch`` + ``rx_kv_copy``) instead of being
    prefilled, and after each wave's finish every finished sequence is
    written through to the host pool (``rx_write_through_batch`` +
    ``rx_kv_copy``).
    With ``out_ring`` (an ``OutputRing``) every launch writes into the ring's
    next device buffer and the ring copies each buffer back to the host once
    the next launch takes a buffer (and at the end of a run); the tensors the
    callbacks receive are then overwritten when the ring comes round.
    """

    def __init__(self, wl, device=None, inputs=None, layers=None, on_extend=None,
                 on_decode=None, stream=None, timing=False, on_decode_wave=None,
                 reuse_outputs=False, out_ring=None, policy="fcfs", chunk_tokens=None,
                 host_slots=0):
        self.wl = wl
        self.device = device
        self.inputs = inputs
        self.layers = list(range(wl.num_layers)) if layers is None else list(layers)
        self.on_extend = on_extend
        self.on_decode = on_decode
        self.on_decode_wave = on_decode_wave
        self.stream = stream
        # launches with no explicit stream go to the device's current stream
        # as of construction, resolved once (a lookup per launch costs more
        # host time than some of the kernels it launches)
        self._explicit_stream = stream is not None
        self.scale = 1.0 / math.sqrt(wl.head_dim)
        self.max_ctx = max(len(wl.prompt_tokens(r)) for r in wl.requests.values()) + \
            wl.decode_steps
        self.max_wave = max(len(w) for w in wl.waves)
        self.gpu_launches = 0
        self.timing = timing
        self.reuse_outputs = reuse_outputs
        self.out_ring = out_ring
        self.policy = policy
        self.chunk_tokens = chunk_tokens
        self.host_slots = int(host_slots)
        self._out_bufs = {}
        self.kernel_events = []   # (kind, start event, end event, algorithmic work)
        if device is not None:
            import torch
            self.torch = torch
            if self.stream is None:
                self.stream = torch.cuda.current_stream(device)
            L, hkv, d = wl.num_layers, wl.num_kv_heads, wl.head_dim
            self.k_pool = torch.empty((L, hkv, wl.num_slots, d), dtype=torch.bfloat16,
                                      device=device)
            self.v_pool = torch.empty_like(self.k_pool)
            self.pool = rx.pool_desc(self.k_pool, self.v_pool)
            if self.host_slots:
                self.hk_pool = torch.empty((L, hkv, self.host_slots, d), dtype=torch.bfloat16,
                                           pin_memory=True)
                self.hv_pool = torch.empty_like(self.hk_pool).pin_memory()
                self.host_pool = rx.pool_desc(self.hk_pool, self.hv_pool)
            self.d_table = torch.zeros((self.max_wave, self.max_ctx), dtype=torch.int32,
                                       device=device)
            self.d_ws = torch.empty(0, dtype=torch.uint8, device=device)
            self.staging = _Staging(torch, device, self.stream, self._explicit_stream)
        # host staging
        self.h_table = np.zeros((self.max_wave, self.max_ctx), dtype=np.int32)
        self._h_table_p = self.h_table.ctypes.data
        self._wave_arrays = {}
        # one extend batch's outputs of rx_extend_begin, reused batch to batch
        # (what outlives the batch is copied out of them)
        max_wave_tokens = max(sum(len(wl.prompt_tokens(r)) for r in w) for w in wl.waves)
        self._b_prefix = np.zeros(self.max_wave, dtype=np.int32)
        self._b_nodes = np.zeros(self.max_wave, dtype=np.int64)
        self._b_new = np.zeros(max(1, max_wave_tokens), dtype=np.int32)
        self._b_ptrs = (self._b_prefix.ctypes.data, self._b_nodes.ctypes.data,
                        self._b_new.ctypes.data)
        self._w_ends = np.zeros(self.max_wave, dtype=np.int32)
        self._w_rew = np.zeros(self.max_wave, dtype=np.int64)
        self._events = rx.EventPool() if device is not None else None
        self.max_extend_rows = 0      # query rows of the largest extend launch so far
        self.plan_buf = np.empty(1 << 16, dtype=np.int32)

    def close(self):
        """Releases the library timing events this engine made (the kernel
        events of earlier timed runs are invalid afterwards)."""
        if self._events is not None:
            self._events.close()

    # ------------------------------------------------------------------ run
    def run(self):
        self.cache = rx.RadixCache(self.wl.num_slots, self.wl.page_size, self.host_slots)
        self.trace = Trace()
        self.batch_no = 0
        self.step_no = 0
        for wi, wave in enumerate(self.wl.waves):
            self._run_wave(wi, wave)
        if self.out_ring is not None and self.device is not None:
            self.out_ring.flush(self.stream)
        self.trace.eviction_log = self.cache.eviction_log()
        if self.host_slots:
            self.trace.host_eviction_log = self.cache.host_eviction_log()
        st = self.cache.stats()
        self.trace.stats = {
            "cached": st["cached_tokens"], "evictable": st["evictable_tokens"],
            "protected": st["protected_tokens"], "free": st["free_slots"],
            "num_nodes": st["num_nodes"]}
        return self.trace

    def _wave_host(self, wi, wave):
        """The token arrays of a wave's requests, as they arrive: prompt
        lengths, the prompts concatenated (int32) with their int64 offsets, and
        each prompt followed by its decode outputs, with offsets.  They depend
        only on the requests, so they are built on the first run and reused."""
        h = self._wave_arrays.get(wi)
        if h is None:
            wl = self.wl
            prompts = [np.asarray(wl.prompt_tokens(r), dtype=np.int32) for r in wave]
            lens = np.array([len(p) for p in prompts], dtype=np.int64)
            indptr = np.zeros(len(wave) + 1, dtype=np.int64)
            np.cumsum(lens, out=indptr[1:])
            tokens = np.concatenate(prompts).astype(np.int32, copy=False)
            outs = [np.asarray(wl.output_tokens(r)[:wl.decode_steps], dtype=np.int32)
                    for r in wave]
            full = np.concatenate([np.concatenate([p, o]) for p, o in zip(prompts, outs)])
            full = full.astype(np.int32, copy=False)
            findptr = np.zeros(len(wave) + 1, dtype=np.int64)
            np.cumsum(lens + wl.decode_steps, out=findptr[1:])
            for arr in (lens, indptr, tokens, full, findptr):
                arr.setflags(write=False)
            h = (lens, indptr, tokens, full, findptr, tokens.ctypes.data, indptr.ctypes.data)
            self._wave_arrays[wi] = h
        return h

    def _run_wave(self, wi, wave):
        if self.policy != "fcfs":
            return self._run_wave_scheduled(wi, wave)
        wl = self.wl
        lens, indptr, tokens, full, findptr, tokens_p, indptr_p = self._wave_host(wi, wave)
        self.h_table[:len(wave)] = 0
        prompt_nodes = np.zeros(len(wave), dtype=np.int64)
        if self.host_slots or self.chunk_tokens:
            ptrs = (tokens_p, indptr_p, prompt_nodes.ctypes.data)
            # in-batch prefix rule: each batch runs to the first request that
            # would share more with an earlier member than the tree gives it
            start = 0
            while start < len(wave):
                end = self.cache.batch_end_p(tokens_p, indptr_p, start, len(wave))
                self._extend_batch(wave, start, end, indptr, ptrs)
                start = end
        else:
            self._extend_wave(wave, lens, tokens_p, indptr_p, prompt_nodes)
        if wl.decode_steps:
            self._decode_phase(wave, lens.astype(np.int32), prompt_nodes)
        # finish: insert prompt ++ outputs, unlock
        self._finish(wave, full, findptr, lens, prompt_nodes)

    def _load_from_host(self, reqs, R, tokens_p, ind_p, cap):
        """rx_load_batch for a batch's members and the copy of the loaded KV
        from the host pool into the device pool."""
        h, d, cnt = self.cache.load_batch_p(R, tokens_p, ind_p, cap)
        pos = 0
        for r, c in zip(reqs, cnt.tolist()):
            if c:
                self.trace.loads.append((r.rid, h[pos:pos + c].copy(), d[pos:pos + c].copy()))
            pos += c
        if self.device is not None and len(h):
            d_src, d_dst = self.staging.upload([h, d])
            rx.kv_copy(self.host_pool, self.pool, d_src, d_dst, self.stream)
            self.gpu_launches += 1

    def _chunks(self, prefix, qo):
        """The batch's query rows [0, total) cut into consecutive chunks of at
        most chunk_tokens rows.  Per chunk: the first row q0, and for each
        request it touches its batch row, prefix (its own prefix plus its
        suffix rows before the chunk), query offsets relative to q0 and the
        tile plan.  One chunk (the whole batch) without chunk_tokens."""
        total = int(qo[-1])
        C = self.chunk_tokens
        if not C or total <= C:
            return [None]
        wl = self.wl
        out = []
        for a in range(0, total, C):
            b = min(total, a + C)
            rows, pre, offs = [], [], [0]
            for r in range(len(prefix)):
                lo, hi = max(a, int(qo[r])), min(b, int(qo[r + 1]))
                if lo >= hi:
                    continue
                rows.append(r)
                pre.append(int(prefix[r]) + lo - int(qo[r]))
                offs.append(offs[-1] + hi - lo)
            cq = np.array(offs, dtype=np.int32)
            tiles, n_tiles = rx.extend_plan(cq, wl.num_q_heads, wl.num_kv_heads, wl.head_dim)
            out.append({"q0": a, "rows": np.array(rows, dtype=np.int32),
                        "prefix": np.array(pre, dtype=np.int32), "qo": cq, "tiles": tiles,
                        "n_tiles": n_tiles})
        return out

    def _run_wave_scheduled(self, wi, wave):
        """A wave under a cache-aware policy: before every extend batch the
        waiting requests are ordered by ``rx_schedule`` and the batch is taken
        from the head of that order by the in-batch rule; requests take slot
        table rows in the order they are served, and decode and finish run in
        that order."""
        wl = self.wl
        lens, indptr, tokens, full, findptr, _, _ = self._wave_host(wi, wave)
        R = len(wave)
        self.h_table[:R] = 0
        prompt_nodes = np.zeros(R, dtype=np.int64)
        pending = list(range(R))
        served = []

        def gather(pos, tok, ind):
            parts = [tok[ind[j]:ind[j + 1]] for j in pos]
            out_ind = np.zeros(len(pos) + 1, dtype=np.int64)
            np.cumsum([len(x) for x in parts], out=out_ind[1:])
            return np.concatenate(parts).astype(np.int32, copy=False), out_ind

        while pending:
            ptok, pind = gather(pending, tokens, indptr)
            ordered = [pending[k] for k in self.cache.schedule(self.policy, ptok, pind)]
            otok, oind = gather(ordered, tokens, indptr)
            end = self.cache.batch_end(otok, oind, 0)
            ptrs = (otok.ctypes.data, oind.ctypes.data, prompt_nodes.ctypes.data)
            self._extend_batch([wave[j] for j in ordered], 0, end, oind, ptrs,
                               row0=len(served))
            served += ordered[:end]
            taken = set(ordered[:end])
            pending = [j for j in pending if j not in taken]
        swave = [wave[j] for j in served]
        slens = lens[served]
        if wl.decode_steps:
            self._decode_phase(swave, slens.astype(np.int32), prompt_nodes)
        sfull, sfind = gather(served, full, findptr)
        self._finish(swave, sfull, sfind, slens, prompt_nodes)

    def _finish(self, wave, full, findptr, lens, prompt_nodes):
        """rx_finish of a wave (rows 0 .. len(wave)-1), then with a host tier
        the write-through of every finished sequence and its copy to the
        host pool."""
        R = len(wave)
        nodes = np.zeros(R, dtype=np.int64)
        already = self.cache.finish(full, findptr, self.h_table[:R], lens, prompt_nodes, nodes)
        for r, a in zip(wave, already):
            self.trace.finishes.append((r.rid, int(a)))
        if not self.host_slots:
            return
        d, h, cnt = self.cache.write_through_batch(nodes, int(findptr[-1] - findptr[0]))
        pos = 0
        for r, c in zip(wave, cnt.tolist()):
            self.trace.backups.append((r.rid, d[pos:pos + c].copy(), h[pos:pos + c].copy()))
            pos += c
        if self.device is not None and len(d):
            d_src, d_dst = self.staging.upload([d, h])
            rx.kv_copy(self.pool, self.host_pool, d_src, d_dst, self.stream)
            self.gpu_launches += 1

    def _extend_batch(self, wave, j0, j1, indptr, ptrs, row0=0):
        """Requests j0 .. j1-1 of the wave as one extend batch.  ``indptr`` is
        the wave's token offsets (this batch's slice of it is passed as is:
        offsets are relative to the wave's tokens); ``ptrs`` = addresses of
        the wave's tokens, its offsets and its prompt-node array.  Request j
        uses row row0 + j of the slot table (and of the prompt-node array)."""
        tokens_p, indptr_p, nodes_out_p = ptrs
        reqs = wave[j0:j1]
        R = j1 - j0
        ind = indptr[j0:j1 + 1]
        ind_p = indptr_p + 8 * j0
        r0 = row0 + j0
        table = self.h_table[r0:r0 + R]
        table_p = self._h_table_p + 4 * self.max_ctx * r0
        prefix_p, mnodes_p, new_p = self._b_ptrs
        if self.host_slots:
            self._load_from_host(reqs, R, tokens_p, ind_p, int(ind[-1] - ind[0]))
        total = self.cache.extend_begin_p(R, tokens_p, ind_p, table_p, self.max_ctx, prefix_p,
                                          mnodes_p, new_p)
        prefix = self._b_prefix[:R]
        new_slots = self._b_new[:total]
        lens = ind[1:] - ind[:-1]
        # the trace keeps each row as extend_begin wrote it (one copy per batch)
        rows = table[:, :int(lens.max())].copy()
        pre, ln = prefix.tolist(), lens.tolist()
        self.trace.batches.append([(r.rid, pre[i], rows[i, :ln[i]]) for i, r in enumerate(reqs)])
        self.trace.prefilled += int(lens.sum()) - sum(pre)
        if self.device is not None:
            self._extend_device(reqs, r0, r0 + R, prefix, ind, new_slots)
        self.cache.extend_end_p(R, tokens_p, ind_p, table_p, self.max_ctx, prefix_p, mnodes_p,
                                nodes_out_p + 8 * r0)
        self.batch_no += 1

    def _extend_wave(self, wave, lens, tokens_p, indptr_p, prompt_nodes):
        """Every extend batch of a wave: the bookkeeping of all its batches in
        one native call (``rx_extend_wave``: the in-batch rule, match, lock,
        allocation, insert, batch after batch), then, with a device, one
        upload of every batch's rows and plans and one native call per layer
        that launches each batch's store and attention in batch order
        (``rx_extend_batches``)."""
        R = len(wave)
        ends, prefix, new = self._w_ends, self._b_prefix, self._b_new
        nb = self.cache.extend_wave_p(R, tokens_p, indptr_p, self._h_table_p, self.max_ctx, ends,
                                      prefix, prompt_nodes, new, self._w_rew)
        prefix = prefix[:R].copy()
        sfx = lens - prefix
        total = int(sfx.sum())
        new_slots = new[:total].copy()
        bounds = [0] + ends[:nb].tolist()
        # each row as its batch's kernels read it: the matched slots, then the
        # request's new slots (rx_extend_end may since have swapped the new
        # slots of a prompt an earlier batch inserted whole for the tree's)
        W = int(lens.max())
        rows = self.h_table[:R, :W].copy()
        rew = self._w_rew[:nb]
        if rew.any():
            col = np.arange(W)
            rows[(col[None, :] >= prefix[:, None]) & (col[None, :] < lens[:, None])] = new_slots
        pre, ln = prefix.tolist(), lens.tolist()
        for b in range(nb):
            self.trace.batches.append([(wave[j].rid, pre[j], rows[j, :ln[j]])
                                       for j in range(bounds[b], bounds[b + 1])])
        self.trace.prefilled += total
        if self.device is not None:
            self._extend_wave_device(wave, bounds, prefix, sfx, rows, new_slots)
        self.batch_no += nb

    def _extend_wave_device(self, wave, bounds, prefix, sfx, rows, new_slots):
        """A wave's extend batches on the device, in launch groups: a group is
        a run of consecutive batches in which only the last may have rows that
        rx_extend_end rewrote.  Per group and layer one store of all its new
        tokens' K/V, then one attention over all its requests.  That equals
        launching batch by batch: a batch's prefix may end in tokens an
        earlier batch of its group stored, which the group's store has
        written before its attention runs; no slot is stored twice within a
        group, since slots become free during a wave's bookkeeping only by
        eviction (of nodes no batch of the wave reads, which are locked) or
        by a rewrite, which ends the group; and a rewritten request's row as
        its kernels read it holds its own new slots, which later groups
        reuse only after its attention ran (one stream)."""
        wl = self.wl
        R, nb = len(wave), len(bounds) - 1
        gb = launch_groups(self._w_rew[:nb])
        gbounds = [bounds[g] for g in gb]
        ng = len(gb) - 1
        # query offsets and tile plans of the whole wave (a request's tiles
        # depend on its own suffix only), cut per group: group g's R_g + 1
        # entries start at position gbounds[g] + g of the concatenated arrays
        qo_w = np.zeros(R + 1, dtype=np.int32)
        np.cumsum(sfx, out=qo_w[1:])
        tiles_w, _ = rx.extend_plan(qo_w, wl.num_q_heads, wl.num_kv_heads, wl.head_dim)
        go = np.asarray(gbounds, dtype=np.int64)
        qo_c = cut_per_group(qo_w, go)
        tiles_c = cut_per_group(tiles_w, go)
        W = rows.shape[1]
        d_rows, d_prefix, d_qo, d_tiles, d_slots, d_tab = self.staging.upload([
            np.arange(R, dtype=np.int32), prefix, qo_c, tiles_c, new_slots, rows.ravel()])
        rec = np.zeros(ng, dtype=rx.EXTEND_BATCH_DTYPE)
        qo_at = qo_w[go].astype(np.int64)
        rec["n_new"] = qo_at[1:] - qo_at[:-1]
        rec["num_tiles"] = tiles_w[go[1:]] - tiles_w[go[:-1]]
        rec["row_stride"] = W
        rec["R"] = go[1:] - go[:-1]
        rec["d_req_to_token"] = d_tab.ptr
        rec["d_req_rows"] = d_rows.ptr + 4 * go[:-1]
        rec["d_prefix_len"] = d_prefix.ptr + 4 * go[:-1]
        off = 4 * (go[:-1] + np.arange(ng))
        rec["d_qo_indptr"] = d_qo.ptr + off
        rec["d_tile_indptr"] = d_tiles.ptr + off
        rec["d_new_slots"] = d_slots.ptr + 4 * qo_at[:-1]
        b0 = self.batch_no
        n_new = rec["n_new"].tolist()
        self.max_extend_rows = max([self.max_extend_rows] + n_new)
        flops = [self._extend_flops(prefix[gbounds[g]:gbounds[g + 1]],
                                    qo_c[gbounds[g] + g:gbounds[g + 1] + g + 1])
                 for g in range(ng)] if self.timing else None
        outs = [dict() for _ in range(ng)]

        def group_inputs(g):
            j0, j1 = gbounds[g], gbounds[g + 1]
            return self.inputs.extend(b0 + gb[g], wave[j0:j1], prefix[j0:j1])

        def fill(g, inp, layer):
            q, k, v = inp[layer]
            o, l = self._outputs(("ext", b0 + gb[g], layer),
                                 (n_new[g], wl.num_q_heads, wl.head_dim))
            for f, t in (("d_q", q), ("d_k", k), ("d_v", v), ("d_out", o), ("d_lse", l)):
                rec[f][g] = t.data_ptr()
            outs[g][layer] = (o, l)

        def launch(layer, lo, hi):
            ev = self._events.take(4 * (hi - lo)) if self.timing else None
            rx.extend_batches(self.pool, layer, wl.num_q_heads, rec[lo:hi], self.scale, ev,
                              self.stream)
            self.gpu_launches += 2 * (hi - lo)
            if ev is not None:
                for g in range(lo, hi):
                    e = [rx.NativeEvent(x) for x in ev[4 * (g - lo):4 * (g - lo) + 4]]
                    self.kernel_events.append(
                        ("kv_store", e[0], e[1],
                         float(4 * total_new_bytes(n_new[g], wl) + 4 * n_new[g])))
                    self.kernel_events.append(("extend", e[2], e[3], flops[g]))

        if self.out_ring is not None or getattr(self.inputs, "host", False):
            # rings of inputs or outputs hand a buffer out on the understanding
            # that the work on the one before it is enqueued: group by group
            for g in range(ng):
                inp = group_inputs(g)
                for layer in self.layers:
                    fill(g, inp, layer)
                    launch(layer, g, g + 1)
        else:
            inputs = [group_inputs(g) for g in range(ng)]
            for layer in self.layers:
                for g in range(ng):
                    fill(g, inputs[g], layer)
                launch(layer, 0, ng)
        if self.on_extend is not None:
            qo_l = qo_w.tolist()
            for g in range(ng):
                for b in range(gb[g], gb[g + 1]):
                    j0, j1 = bounds[b], bounds[b + 1]
                    q0, q1 = qo_l[j0] - qo_l[gbounds[g]], qo_l[j1] - qo_l[gbounds[g]]
                    qo = qo_w[j0:j1 + 1] - qo_w[j0]
                    self.on_extend(b0 + b, [r.rid for r in wave[j0:j1]], prefix[j0:j1].copy(),
                                   qo, {ly: (o[q0:q1], l[q0:q1])
                                        for ly, (o, l) in outs[g].items()})

    def _extend_device(self, reqs, j0, j1, prefix, ind, new_slots):
        torch = self.torch
        wl = self.wl
        R = j1 - j0
        qo = np.zeros(R + 1, dtype=np.int32)
        np.cumsum((ind[1:] - ind[:-1]) - prefix, out=qo[1:])
        tiles, n_tiles = rx.extend_plan(qo, wl.num_q_heads, wl.num_kv_heads, wl.head_dim)
        # the kernels read the batch's rows of the slot table from the staged
        # copy (rows 0 .. R-1); the engine's device table gets the wave's rows
        # once, before its decode steps
        width = int(max(ind[1:] - ind[:-1]))
        chunks = self._chunks(prefix, qo)
        d_rows, d_prefix, d_qo, d_tiles, d_slots, d_tab, *d_extra = self.staging.upload([
            np.arange(R, dtype=np.int32), prefix, qo, tiles, new_slots,
            self.h_table[j0:j1, :width].ravel()] + ([c for ch in chunks for c in (
                ch["rows"], ch["prefix"], ch["qo"], ch["tiles"])] if len(chunks) > 1 else []))
        d_tab.shape = (R, width)
        inputs = self.inputs.extend(self.batch_no, reqs, prefix)
        total_q = int(qo[-1])
        self.max_extend_rows = max(self.max_extend_rows, total_q)
        flops = self._extend_flops(prefix, qo) if self.timing else 0.0
        outs = {}
        store_bytes = float(4 * total_new_bytes(len(new_slots), wl) + 4 * len(new_slots))
        for layer in self.layers:
            q, k, v = inputs[layer]
            ev = self._event_start()
            rx.kv_store(self.pool, layer, d_slots, k, v, self.stream)
            self._event_end(ev, "kv_store", store_bytes)
            out, lse = self._outputs(("ext", self.batch_no, layer),
                                     (total_q, wl.num_q_heads, wl.head_dim))
            if len(chunks) == 1:
                calls = [rx.extend_attention_call(self.pool, layer, q, wl.num_q_heads, d_tab,
                                                  d_rows, d_prefix, d_qo, d_tiles, R, n_tiles,
                                                  self.scale, out, lse, self.stream)]
            else:
                calls = []
                for k, ch in enumerate(chunks):
                    cr, cp, cq, ct = d_extra[4 * k:4 * k + 4]
                    a = ch["q0"]
                    calls.append(rx.extend_attention_call(
                        self.pool, layer, q[a:], wl.num_q_heads, d_tab, cr, cp, cq, ct,
                        len(ch["rows"]), ch["n_tiles"], self.scale, out[a:], lse[a:],
                        self.stream))
            ev = self._event_start()
            for call in calls:
                call()
            self._event_end(ev, "extend", flops)
            self.gpu_launches += 1 + len(calls)
            outs[layer] = (out, lse)
        if self.on_extend is not None:
            self.on_extend(self.batch_no, [r.rid for r in reqs], prefix.copy(), qo, outs)

    def _decode_phase(self, wave, ctx0, prompt_nodes):
        """All decode steps of a wave.  Slot allocation and the decode plan
        depend only on the cache, not on kernel results, and the tree does not
        change while the wave decodes, so the host allocates every step's slots
        (one call), builds one plan valid for every step, uploads both with one
        copy, and the GPU then runs the steps back to back."""
        wl = self.wl
        B, T = len(wave), wl.decode_steps
        rows = np.arange(B, dtype=np.int32)
        if wl.page_size == 1:
            all_slots = self.cache.alloc_steps(B, T)                # [T, B]
        else:   # a token that starts a page takes a new one, others follow
            all_slots = self.cache.alloc_decode_steps(
                ctx0, self.h_table[np.arange(B), ctx0 - 1], T)
        all_pos = ctx0[None, :] + np.arange(T, dtype=np.int32)[:, None]
        self.h_table[rows[None, :], all_pos] = all_slots
        rids = np.array([r.rid for r in wave])
        self.trace.decode_steps.append(_DecodeRecord(rids, all_slots))
        if self.device is None:
            self.step_no += T
            return
        torch = self.torch
        self.plan_buf, info = self.cache.plan_decode(
            prompt_nodes, ctx0 + 1, rows, wl.num_q_heads, wl.num_kv_heads, wl.head_dim,
            self.plan_buf, n_steps=T)
        plan = self.plan_buf[:int(info.plan_words)]
        # the wave's prompt rows of the slot table (the extend kernels read
        # per-batch staged copies), then every step's decode slots
        width = int(ctx0.max())
        (tab,) = self.staging.upload([self.h_table[:B, :width].ravel()], as_tensors=True)
        self.d_table[:B, :width].copy_(tab.view(B, width))
        d_rows, d_pos, d_slots, d_plan = self.staging.upload(
            [np.tile(rows, T), all_pos.ravel().astype(np.int32), all_slots.ravel(), plan])
        rx.req_to_token_write(self.d_table, d_rows, d_pos, d_slots, self.stream)
        self.gpu_launches += 1
        need = int(info.workspace_bytes)
        if self.d_ws.numel() < need:
            self.d_ws = torch.empty(int(need * 1.25) + 256, dtype=torch.uint8, device=self.device)
        # every step's inputs and outputs, then one native call per layer
        inputs = self.inputs.decode_wave(self.step_no, wave, T)
        outs = {}
        tt = np.arange(T, dtype=np.uint64)
        for layer in self.layers:
            o, l = self._outputs(("dec", self.step_no, layer),
                                 (T, B, wl.num_q_heads, wl.head_dim))
            steps = np.zeros(T, dtype=rx.DECODE_STEP_DTYPE)
            for f, x in zip(("d_q", "d_k", "d_v"), inputs[layer]):
                steps[f] = x.data_ptr() + tt * np.uint64(x[0].numel() * x.element_size())
            steps["d_slots"] = d_slots.data_ptr() + tt * np.uint64(4 * B)
            steps["d_plan"] = d_plan.data_ptr()
            steps["info"] = ctypes.addressof(info)
            steps["d_out"] = o.data_ptr() + tt * np.uint64(o[0].numel() * 4)
            steps["d_lse"] = l.data_ptr() + tt * np.uint64(l[0].numel() * 4)
            steps["step"] = np.arange(T, dtype=np.int32)
            ev = self._event_start()
            rx.decode_steps(self.pool, layer, wl.num_q_heads, self.d_table, steps, B, self.scale,
                            self.d_ws, self.stream)
            self._event_end(ev, "decode", sum(self.decode_bytes(info, B, t * B)
                                              for t in range(T)) if self.timing else 0.0)
            self.gpu_launches += T * self._launches_per_decode([info])
            outs[layer] = (o, l)
        if self.on_decode is not None:
            for t in range(T):
                self.on_decode(self.step_no + t, t, list(rids), ctx0 + 1 + t,
                               {ly: (outs[ly][0][t], outs[ly][1][t]) for ly in self.layers},
                               info)
        if self.on_decode_wave is not None:
            self.on_decode_wave(self.step_no, list(rids), ctx0 + 1, outs, info)
        self.step_no += T

    def _outputs(self, key, shape):
        """fp32 output [..., Hq, d] and lse [..., Hq] tensors for one launch:
        fresh ones, or with reuse_outputs the ones this key got on an earlier
        run (same shapes every run)."""
        torch = self.torch
        if self.out_ring is not None:
            return self.out_ring.take(shape, self.stream)
        if self.reuse_outputs:
            bufs = self._out_bufs.get(key)
            if bufs is not None and tuple(bufs[0].shape) == tuple(shape):
                return bufs
        bufs = (torch.empty(shape, dtype=torch.float32, device=self.device),
                torch.empty(shape[:-1], dtype=torch.float32, device=self.device))
        if self.reuse_outputs:
            self._out_bufs[key] = bufs
        return bufs

    def _launches_per_decode(self, infos):
        """Kernels per decode step: kv_store (unless the decode kernel
        stores the new tokens itself), the decode kernel (one fused launch
        for tensor-core and warp-role items), merge."""
        i = infos[0]
        store = 0 if int(i.tails_private) == 1 else 1
        return store + int(int(i.n_work) > 0) + 1

    # ------------------------------------------------------------ timing
    def _event_start(self):
        if not self.timing:
            return None
        e = self.torch.cuda.Event(enable_timing=True)
        e.record(self.stream)
        return e

    def _event_end(self, start, kind, work):
        if start is None:
            return
        e = self.torch.cuda.Event(enable_timing=True)
        e.record(self.stream)
        self.kernel_events.append((kind, start, e, work))

    def _extend_flops(self, prefix, qo):
        """Algorithmic FLOPs of one extend launch: 4 * d * Hq per visible
        (query, key) pair; query i of a suffix of s over a prefix p sees
        p + i + 1 keys."""
        s = (qo[1:] - qo[:-1]).astype(np.int64)
        p = np.asarray(prefix, dtype=np.int64)
        pairs = int(np.sum(s * p + s * (s + 1) // 2))
        return 4.0 * self.wl.head_dim * self.wl.num_q_heads * pairs

    def decode_bytes(self, info, B, extra_tokens=0):
        """Algorithmic bytes of one decode launch: the distinct KV of the
        batch read once (K and V, bf16), its slot indices, Q (bf16) and the
        fp32 output and lse.  ``extra_tokens`` adds tokens beyond the plan's
        step-0 count (later steps of a multi-step plan)."""
        wl = self.wl
        kv = (info.distinct_kv_tokens + extra_tokens) * (2 * wl.num_kv_heads * wl.head_dim * 2 + 4)
        q = B * wl.num_q_heads * wl.head_dim * 2
        o = B * wl.num_q_heads * (wl.head_dim + 1) * 4
        return float(kv + q + o)
