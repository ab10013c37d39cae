"""ctypes binding of librx (include/rx.h): argument marshalling only.

Every computation happens in the native library: the radix cache in C++, the
attention and KV stores in sm_103a CUDA kernels.  Host arrays are numpy
arrays (int32 tokens/slots, int64 indptrs); device buffers are torch tensors
whose ``data_ptr()`` is passed through.  Importing this module loads
``lib/librx.so`` and raises ``ImportError`` if it has not been built: there is
no fallback path.
"""

import ctypes as C
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "librx.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"librx.so not found at {LIB_PATH}; build it first with "
        "`python -c 'import __graft_entry__ as g; g.build()'`")
_lib = C.CDLL(LIB_PATH)

RX_OK, RX_ERR_INVALID, RX_ERR_NO_SPACE, RX_ERR_STATE, RX_ERR_CUDA = range(5)
POLICIES = {"fcfs": 0, "lpm": 1, "dfs-weight": 2}     # RX_POLICY_* of rx.h
RX_WORK_WORDS = 8
RX_DECODE_STATIC_SCRATCH_BYTES = 16 << 20   # fixed scratch of rx_decode_attention_static


class RxError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"rx status {status}: {msg}")
        self.status = status


class NoSpace(RxError):
    pass


class StateError(RxError):
    pass


class rx_config(C.Structure):
    _fields_ = [("num_slots", C.c_int64), ("page_size", C.c_int32), ("reserved", C.c_int32),
                ("host_slots", C.c_int64)]


class rx_stats_t(C.Structure):
    _fields_ = [(n, C.c_int64) for n in (
        "cached_tokens", "evictable_tokens", "protected_tokens", "free_slots",
        "num_nodes", "evicted_nodes", "evicted_tokens", "clock", "host_cached_tokens",
        "host_free_slots", "host_evicted_nodes")]


class rx_evict_rec(C.Structure):
    _fields_ = [("node_id", C.c_int64), ("num_tokens", C.c_int64)]


class rx_decode_plan_info(C.Structure):
    _fields_ = [(n, C.c_int64) for n in (
        "plan_words", "n_work", "n_parts", "n_member_entries", "off_work",
        "off_members", "off_req_part_indptr", "off_req_parts",
        "n_shared_segments", "workspace_bytes", "distinct_kv_tokens", "n_work_tc", "tails_private")]


class rx_decode_step(C.Structure):
    _fields_ = [("d_q", C.c_void_p), ("d_k", C.c_void_p), ("d_v", C.c_void_p),
                ("d_slots", C.c_void_p), ("d_plan", C.c_void_p), ("info", C.c_void_p),
                ("d_out", C.c_void_p), ("d_lse", C.c_void_p), ("step", C.c_int32),
                ("reserved", C.c_int32)]


# the same layout as a numpy record, for filling many steps with array ops
DECODE_STEP_DTYPE = np.dtype([("d_q", np.uint64), ("d_k", np.uint64), ("d_v", np.uint64),
                              ("d_slots", np.uint64), ("d_plan", np.uint64),
                              ("info", np.uint64), ("d_out", np.uint64), ("d_lse", np.uint64),
                              ("step", np.int32), ("reserved", np.int32)])
assert DECODE_STEP_DTYPE.itemsize == C.sizeof(rx_decode_step)

# rx_extend_batch as a numpy record (pointers as uint64)
_EXT_PTRS = ("d_q", "d_k", "d_v", "d_new_slots", "d_req_to_token", "d_req_rows",
             "d_prefix_len", "d_qo_indptr", "d_tile_indptr", "d_out", "d_lse")
EXTEND_BATCH_DTYPE = np.dtype([(n, np.uint64) for n in _EXT_PTRS] +
                              [("n_new", np.int64), ("num_tiles", np.int64),
                               ("row_stride", np.int64), ("R", np.int32),
                               ("reserved", np.int32)])


class rx_extend_batch(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in _EXT_PTRS] + [
        ("n_new", C.c_int64), ("num_tiles", C.c_int64), ("row_stride", C.c_int64),
        ("R", C.c_int32), ("reserved", C.c_int32)]


assert EXTEND_BATCH_DTYPE.itemsize == C.sizeof(rx_extend_batch)


class rx_pool_desc(C.Structure):
    _fields_ = [("k_pool", C.c_void_p), ("v_pool", C.c_void_p), ("num_slots", C.c_int64),
                ("num_layers", C.c_int32), ("num_kv_heads", C.c_int32),
                ("head_dim", C.c_int32), ("reserved", C.c_int32)]


P = C.c_void_p
I32, I64, F32, SZ = C.c_int32, C.c_int64, C.c_float, C.c_size_t
_SIGS = {
    "rx_cache_create": [P, P],
    "rx_cache_destroy": [P],
    "rx_match_length": [P, P, I64, P],
    "rx_match_prefix": [P, P, I64, P, P, P],
    "rx_lock": [P, I64],
    "rx_unlock": [P, I64],
    "rx_alloc": [P, I64, P],
    "rx_evict": [P, I64, P],
    "rx_free": [P, P, I64],
    "rx_insert": [P, P, P, I64, P, P],
    "rx_stats": [P, P],
    "rx_eviction_log": [P, I64, P, I64, P],
    "rx_node_depth": [P, I64, P],
    "rx_extend_begin": [P, I32, P, P, P, I64, P, P, P, P],
    "rx_extend_end": [P, I32, P, P, P, I64, P, P, P, P],
    "rx_finish": [P, I32, P, P, P, I64, P, P, P, P],
    "rx_match_prefix_tiers": [P, P, I64, P, P, P, P, P],
    "rx_load_onboard": [P, I64, P, P, I64, P],
    "rx_write_through": [P, I64, P, P, I64, P, P],
    "rx_commit_write_through": [P, I64, I32],
    "rx_load_batch": [P, I32, P, P, P, P, I64, P, P],
    "rx_write_through_batch": [P, I32, P, P, P, I64, P, P],
    "rx_host_eviction_log": [P, I64, P, I64, P],
    "rx_debug_fail_alloc": [P, I64],
    "rx_host_alloc": [SZ, P],
    "rx_extend_wave": [P, I32, P, P, P, I64, P, P, P, P, P, P],
    "rx_host_free": [P],
    "rx_batch_conflict": [P, I64, I64, I32, P, P, P],
    "rx_batch_end": [P, P, P, I32, I32, P],
    "rx_plan_decode": [P, I32, P, P, P, I32, I32, I32, P, I64, P],
    "rx_plan_decode_steps": [P, I32, I32, P, P, P, I32, I32, I32, P, I64, P],
    "rx_alloc_steps": [P, I64, I32, P],
    "rx_alloc_decode_steps": [P, I32, I32, P, P, P],
    "rx_schedule": [P, I32, I32, P, P, P],
    "rx_verify_rows": [I32, P, P, I64, P, P, P, P, I64, P, P],
    "rx_verify_attention": [P, I32, P, I32, P, I64, P, P, I32, F32, P, P, P, SZ, P],
    "rx_kv_copy": [P, P, P, P, I64, P],
    "rx_kv_store": [P, I32, P, P, P, I64, P],
    "rx_req_to_token_write": [P, I64, I64, P, P, P, I64, P],
    "rx_extend_plan": [P, I32, I32, I32, I32, P, P],
    "rx_extend_attention": [P, I32, P, I32, P, I64, P, P, P, P, I32, I64, F32, P, P, P],
    "rx_decode_attention": [P, I32, P, I32, P, I64, P, P, I32, F32, P, P, P, SZ, P],
    "rx_decode_attention_static": [P, I32, P, I32, P, I64, P, P, I32, F32, P, P, P],
    "rx_decode_steps": [P, I32, I32, P, I64, P, I32, I32, F32, P, SZ, P],
    "rx_extend_batches": [P, I32, I32, P, I32, F32, P, P],
    "rx_events_create": [I32, P],
    "rx_events_destroy": [I32, P],
    "rx_event_elapsed_ms": [P, P, P],
    "rx_device_check": [P],
}
for _name, _args in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = C.c_int
_lib.rx_last_error.argtypes = [C.c_char_p, C.c_size_t]
_lib.rx_last_error.restype = C.c_size_t
_lib.rx_build_info.argtypes = []
_lib.rx_build_info.restype = C.c_char_p

EXPORTED = sorted(list(_SIGS) + ["rx_last_error", "rx_build_info"])


def last_error():
    buf = C.create_string_buffer(1024)
    _lib.rx_last_error(buf, 1024)
    return buf.value.decode()


def _check(st):
    if st == RX_OK:
        return
    msg = last_error()
    if st == RX_ERR_NO_SPACE:
        raise NoSpace(st, msg)
    if st == RX_ERR_STATE:
        raise StateError(st, msg)
    raise RxError(st, msg)


def _p(a):
    """Pointer of a contiguous numpy array (or None)."""
    if a is None:
        return None
    return a.ctypes.data


def _i32(x):
    return np.ascontiguousarray(x, dtype=np.int32)


def _i64(x):
    return np.ascontiguousarray(x, dtype=np.int64)


def build_info():
    return _lib.rx_build_info().decode()


# -------------------------------------------------------------- host cache
class RadixCache:
    """Owner of one native rx_cache (pages of `page_size` slots)."""

    def __init__(self, num_slots, page_size=1, host_slots=0):
        cfg = rx_config(int(num_slots), int(page_size), 0, int(host_slots))
        h = C.c_void_p()
        _check(_lib.rx_cache_create(C.byref(cfg), C.byref(h)))
        self._h = h
        self.num_slots = int(num_slots)
        self.page_size = int(page_size)
        self.host_slots = int(host_slots)
        self._i32 = C.c_int32()
        self._i64 = C.c_int64()

    def close(self):
        if self._h:
            _lib.rx_cache_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def batch_end(self, tokens, indptr, start):
        """End of the batch that starts at request `start` (rx_batch_end);
        tokens int32 (the wave's prompts concatenated), indptr int64."""
        out = C.c_int32()
        _check(_lib.rx_batch_end(self._h, _p(tokens), _p(indptr), int(start), len(indptr) - 1,
                                 C.byref(out)))
        return out.value

    # Pointer forms of the batch steps, for a caller that keeps its arrays
    # (the engine): every argument named *_p is the address of a contiguous
    # array of the C type the header gives, owned by the caller.  They skip
    # the per-call array handling of the forms above; offsets in an indptr
    # are relative to the tokens pointer passed with it.
    def batch_end_p(self, tokens_p, indptr_p, start, R):
        _check(_lib.rx_batch_end(self._h, tokens_p, indptr_p, int(start), int(R),
                                 C.byref(self._i32)))
        return self._i32.value

    def extend_begin_p(self, R, tokens_p, indptr_p, table_p, row_stride, prefix_p, nodes_p,
                       new_p):
        """rx_extend_begin; returns the number of new slots written at new_p."""
        _check(_lib.rx_extend_begin(self._h, int(R), tokens_p, indptr_p, table_p,
                                    int(row_stride), prefix_p, nodes_p, new_p,
                                    C.byref(self._i64)))
        return self._i64.value

    def extend_end_p(self, R, tokens_p, indptr_p, table_p, row_stride, prefix_p, nodes_p,
                     out_nodes_p):
        """rx_extend_end; returns the number of rows rewritten with tree slots."""
        _check(_lib.rx_extend_end(self._h, int(R), tokens_p, indptr_p, table_p,
                                  int(row_stride), prefix_p, nodes_p, out_nodes_p,
                                  C.byref(self._i64)))
        return self._i64.value

    def extend_wave_p(self, R, tokens_p, indptr_p, table_p, row_stride, ends, prefix, nodes,
                      new_slots, rewritten):
        """rx_extend_wave with the wave's arrays by address and caller-owned
        output arrays (numpy: int32 ends [R], int32 prefix [R], int64 nodes
        [R], int32 new_slots [total tokens], int64 rewritten [R]); returns
        the number of batches."""
        _check(_lib.rx_extend_wave(self._h, int(R), tokens_p, indptr_p, table_p, int(row_stride),
                                   _p(ends), C.byref(self._i32), _p(prefix), _p(nodes),
                                   _p(new_slots), _p(rewritten)))
        return self._i32.value

    # S1
    def match_length(self, tokens):
        t = _i32(tokens)
        out = C.c_int64()
        _check(_lib.rx_match_length(self._h, _p(t), len(t), C.byref(out)))
        return out.value

    def match_prefix(self, tokens):
        t = _i32(tokens)
        slots = np.empty(max(1, len(t)), dtype=np.int32)
        n = C.c_int64()
        node = C.c_int64()
        _check(_lib.rx_match_prefix(self._h, _p(t), len(t), _p(slots), C.byref(n),
                                    C.byref(node)))
        return slots[:n.value].copy(), node.value

    # S2
    def lock(self, node):
        _check(_lib.rx_lock(self._h, int(node)))

    def unlock(self, node):
        _check(_lib.rx_unlock(self._h, int(node)))

    # S3
    def alloc(self, k, out=None):
        if out is None:
            out = np.empty(max(1, k), dtype=np.int32)
        _check(_lib.rx_alloc(self._h, int(k), _p(out)))
        return out[:k]

    def alloc_steps(self, k, n_steps):
        """n_steps consecutive alloc(k); returns int32 [n_steps, k]."""
        out = np.empty((max(1, n_steps), max(1, k)), dtype=np.int32)
        _check(_lib.rx_alloc_steps(self._h, int(k), int(n_steps), _p(out)))
        return out[:n_steps, :k]

    def alloc_decode_steps(self, pos0, last_slot, n_steps):
        """Decode slots of n_steps steps for requests whose first decode
        token is at position pos0[b] after slot last_slot[b]; int32 [n_steps, B]."""
        p0, ls = _i32(pos0), _i32(last_slot)
        B = len(p0)
        out = np.empty((max(1, n_steps), max(1, B)), dtype=np.int32)
        _check(_lib.rx_alloc_decode_steps(self._h, B, int(n_steps), _p(p0), _p(ls), _p(out)))
        return out[:n_steps, :B]

    def schedule(self, policy, tokens, indptr):
        """Serving order of a waiting queue (rx_schedule): queue positions."""
        pol = POLICIES[policy] if isinstance(policy, str) else int(policy)
        t, ip = _i32(tokens), _i64(indptr)
        R = len(ip) - 1
        out = np.empty(max(1, R), dtype=np.int32)
        _check(_lib.rx_schedule(self._h, pol, R, _p(t), _p(ip), _p(out)))
        return out[:R]

    def evict(self, k):
        f = C.c_int64()
        _check(_lib.rx_evict(self._h, int(k), C.byref(f)))
        return f.value

    def free(self, slots):
        s = _i32(slots)
        _check(_lib.rx_free(self._h, _p(s), len(s)))

    # S10
    def insert(self, tokens, slots):
        t, s = _i32(tokens), _i32(slots)
        already = C.c_int64()
        node = C.c_int64()
        _check(_lib.rx_insert(self._h, _p(t), _p(s), len(t), C.byref(already), C.byref(node)))
        return already.value, node.value

    def stats(self):
        st = rx_stats_t()
        _check(_lib.rx_stats(self._h, C.byref(st)))
        return {n: getattr(st, n) for n, _ in rx_stats_t._fields_}

    def eviction_log(self):
        total = C.c_int64()
        _check(_lib.rx_eviction_log(self._h, 0, None, 0, C.byref(total)))
        n = total.value
        recs = (rx_evict_rec * max(1, n))()
        _check(_lib.rx_eviction_log(self._h, 0, recs, n, C.byref(total)))
        return [(recs[i].node_id, recs[i].num_tokens) for i in range(n)]

    def node_depth(self, node):
        d = C.c_int64()
        _check(_lib.rx_node_depth(self._h, int(node), C.byref(d)))
        return d.value

    # batch steps
    def extend_begin(self, tokens, tok_indptr, req_to_token):
        """req_to_token: int32 [R, row_stride] host array written in place."""
        R = len(tok_indptr) - 1
        prefix = np.empty(max(1, R), dtype=np.int32)
        nodes = np.empty(max(1, R), dtype=np.int64)
        new = np.empty(max(1, int(tok_indptr[-1])), dtype=np.int32)
        total = C.c_int64()
        _check(_lib.rx_extend_begin(self._h, R, _p(tokens), _p(tok_indptr), _p(req_to_token),
                                    req_to_token.shape[1], _p(prefix), _p(nodes), _p(new),
                                    C.byref(total)))
        return prefix[:R], nodes[:R], new[:total.value]

    def extend_end(self, tokens, tok_indptr, req_to_token, prefix, match_nodes):
        """Returns (prompt nodes, number of rows rewritten with tree slots)."""
        R = len(tok_indptr) - 1
        out = np.empty(max(1, R), dtype=np.int64)
        rew = C.c_int64()
        _check(_lib.rx_extend_end(self._h, R, _p(tokens), _p(tok_indptr), _p(req_to_token),
                                  req_to_token.shape[1], _p(prefix), _p(match_nodes), _p(out),
                                  C.byref(rew)))
        return out[:R], rew.value

    def finish(self, tokens, tok_indptr, req_to_token, prompt_len, prompt_nodes, nodes_out=None):
        """rx_finish; returns `already` per request (the nodes of the inserted
        sequences go to nodes_out, int64 [R], when given)."""
        R = len(tok_indptr) - 1
        already = np.empty(max(1, R), dtype=np.int64)
        _check(_lib.rx_finish(self._h, R, _p(tokens), _p(tok_indptr), _p(req_to_token),
                              req_to_token.shape[1], _p(prompt_len), _p(prompt_nodes),
                              _p(already), _p(nodes_out)))
        return already[:R]

    # two tiers
    def match_prefix_tiers(self, tokens):
        """(device slots, device node, host_len, host node)."""
        t = _i32(tokens)
        slots = np.empty(max(1, len(t)), dtype=np.int32)
        dl, hl, dn, hn = C.c_int64(), C.c_int64(), C.c_int64(), C.c_int64()
        _check(_lib.rx_match_prefix_tiers(self._h, _p(t), len(t), _p(slots), C.byref(dl),
                                          C.byref(hl), C.byref(dn), C.byref(hn)))
        return slots[:dl.value].copy(), dn.value, hl.value, hn.value

    def load_onboard(self, node, cap):
        """(host slots, device slots) of the copies to make."""
        h = np.empty(max(1, cap), dtype=np.int32)
        d = np.empty(max(1, cap), dtype=np.int32)
        n = C.c_int64()
        _check(_lib.rx_load_onboard(self._h, int(node), _p(h), _p(d), int(cap), C.byref(n)))
        return h[:n.value], d[:n.value]

    def write_through(self, node, cap):
        """(ticket, device slots, host slots)."""
        d = np.empty(max(1, cap), dtype=np.int32)
        h = np.empty(max(1, cap), dtype=np.int32)
        n, t = C.c_int64(), C.c_int64()
        _check(_lib.rx_write_through(self._h, int(node), _p(d), _p(h), int(cap), C.byref(n),
                                     C.byref(t)))
        return t.value, d[:n.value], h[:n.value]

    def commit_write_through(self, ticket, success):
        _check(_lib.rx_commit_write_through(self._h, int(ticket), 1 if success else 0))

    def load_batch(self, tokens, indptr, cap):
        """(host slots, device slots, per-request counts) of a batch's loads."""
        t, ip = _i32(tokens), _i64(indptr)
        R = len(ip) - 1
        h = np.empty(max(1, cap), dtype=np.int32)
        d = np.empty(max(1, cap), dtype=np.int32)
        cnt = np.empty(max(1, R), dtype=np.int64)
        n = C.c_int64()
        _check(_lib.rx_load_batch(self._h, R, _p(t), _p(ip), _p(h), _p(d), int(cap), C.byref(n),
                                  _p(cnt)))
        return h[:n.value], d[:n.value], cnt[:R]

    def load_batch_p(self, R, tokens_p, indptr_p, cap):
        """rx_load_batch with the prompts given by address (see the pointer
        forms of the batch steps)."""
        h = np.empty(max(1, cap), dtype=np.int32)
        d = np.empty(max(1, cap), dtype=np.int32)
        cnt = np.empty(max(1, R), dtype=np.int64)
        _check(_lib.rx_load_batch(self._h, int(R), tokens_p, indptr_p, _p(h), _p(d), int(cap),
                                  C.byref(self._i64), _p(cnt)))
        n = self._i64.value
        return h[:n], d[:n], cnt[:R]

    def write_through_batch(self, nodes, cap):
        """(device slots, host slots, per-node counts) of the backups."""
        nd = _i64(nodes)
        R = len(nd)
        d = np.empty(max(1, cap), dtype=np.int32)
        h = np.empty(max(1, cap), dtype=np.int32)
        cnt = np.empty(max(1, R), dtype=np.int64)
        n = C.c_int64()
        _check(_lib.rx_write_through_batch(self._h, R, _p(nd), _p(d), _p(h), int(cap),
                                           C.byref(n), _p(cnt)))
        return d[:n.value], h[:n.value], cnt[:R]

    def debug_fail_alloc(self, k):
        """Test hook: the k-th page allocation from now fails (0: off)."""
        _check(_lib.rx_debug_fail_alloc(self._h, int(k)))

    def host_eviction_log(self):
        total = C.c_int64()
        _check(_lib.rx_host_eviction_log(self._h, 0, None, 0, C.byref(total)))
        n = total.value
        recs = (rx_evict_rec * max(1, n))()
        _check(_lib.rx_host_eviction_log(self._h, 0, recs, n, C.byref(total)))
        return [(recs[i].node_id, recs[i].num_tokens) for i in range(n)]

    def plan_decode(self, prompt_nodes, ctx_len, req_rows, hq, hkv, d, plan=None, n_steps=None):
        """rx_plan_decode, or rx_plan_decode_steps when n_steps is given."""
        B = len(prompt_nodes)
        info = rx_decode_plan_info()
        pn, cl, rr = _i64(prompt_nodes), _i32(ctx_len), _i32(req_rows)

        def call(buf):
            cap = 0 if buf is None else len(buf)
            ptr = _p(buf) if buf is not None else None
            if n_steps is None:
                return _lib.rx_plan_decode(self._h, B, _p(pn), _p(cl), _p(rr), hq, hkv, d, ptr,
                                           cap, C.byref(info))
            return _lib.rx_plan_decode_steps(self._h, B, int(n_steps), _p(pn), _p(cl), _p(rr),
                                             hq, hkv, d, ptr, cap, C.byref(info))
        st = call(plan)
        if st != RX_OK and (plan is None or len(plan) < info.plan_words) and info.plan_words > 0:
            plan = np.empty(int(info.plan_words) * 2, dtype=np.int32)
            st = call(plan)
        _check(st)
        return plan, info


def batch_conflict(tokens, match_len, member_tokens, member_indptr):
    out = C.c_int32()
    t = _i32(tokens)
    R = len(member_indptr) - 1
    _check(_lib.rx_batch_conflict(_p(t), len(t), int(match_len), R, _p(member_tokens),
                                  _p(member_indptr), C.byref(out)))
    return bool(out.value)


def extend_plan(qo_indptr, hq, hkv, d):
    qo = _i32(qo_indptr)
    R = len(qo) - 1
    tiles = np.empty(R + 1, dtype=np.int32)
    n = C.c_int64()
    _check(_lib.rx_extend_plan(_p(qo), R, hq, hkv, d, _p(tiles), C.byref(n)))
    return tiles, n.value


# ------------------------------------------------------------- device ops
def pool_desc(k_pool, v_pool):
    """Descriptor of torch bf16 pools shaped [L, Hkv, N, d]."""
    L, hkv, n, d = k_pool.shape
    return rx_pool_desc(k_pool.data_ptr(), v_pool.data_ptr(), n, L, hkv, d, 0)


def _stream(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream)


def kv_store(pool, layer, d_slots, d_k, d_v, stream=None):
    _check(_lib.rx_kv_store(C.byref(pool), layer, d_slots.data_ptr(), d_k.data_ptr(),
                            d_v.data_ptr(), d_slots.numel(), _stream(stream)))


def req_to_token_write(d_table, d_rows, d_pos, d_slots, stream=None):
    _check(_lib.rx_req_to_token_write(d_table.data_ptr(), d_table.shape[0], d_table.shape[1],
                                      d_rows.data_ptr(), d_pos.data_ptr(), d_slots.data_ptr(),
                                      d_slots.numel(), _stream(stream)))


def extend_attention_call(pool, layer, d_q, hq, d_table, d_req_rows, d_prefix_len,
                          d_qo_indptr, d_tile_indptr, R, num_tiles, scale, d_out, d_lse,
                          stream=None):
    """rx_extend_attention with its arguments marshalled now; the returned
    callable makes the call (so a caller timing the launch with events
    brackets only the native call)."""
    args = (C.byref(pool), layer, d_q.data_ptr(), hq, d_table.data_ptr(), d_table.shape[1],
            d_req_rows.data_ptr(), d_prefix_len.data_ptr(), d_qo_indptr.data_ptr(),
            d_tile_indptr.data_ptr(), R, num_tiles, scale, d_out.data_ptr(), d_lse.data_ptr(),
            _stream(stream))
    fn = _lib.rx_extend_attention
    return lambda: _check(fn(*args))


def extend_attention(pool, layer, d_q, hq, d_table, d_req_rows, d_prefix_len, d_qo_indptr,
                     d_tile_indptr, R, num_tiles, scale, d_out, d_lse, stream=None):
    extend_attention_call(pool, layer, d_q, hq, d_table, d_req_rows, d_prefix_len, d_qo_indptr,
                          d_tile_indptr, R, num_tiles, scale, d_out, d_lse, stream)()


def decode_attention(pool, layer, d_q, hq, d_table, d_plan, info, B, scale, d_out, d_lse,
                     d_workspace, stream=None):
    _check(_lib.rx_decode_attention(C.byref(pool), layer, d_q.data_ptr(), hq, d_table.data_ptr(),
                                    d_table.shape[1], d_plan.data_ptr(), C.byref(info), B, scale,
                                    d_out.data_ptr(), d_lse.data_ptr(), d_workspace.data_ptr(),
                                    d_workspace.numel() * d_workspace.element_size(),
                                    _stream(stream)))


def extend_batches(pool, layer, hq, batches, scale, events=None, stream=None):
    """rx_extend_batches over a numpy array of EXTEND_BATCH_DTYPE records;
    ``events`` is None or a uint64 array of 4 event handles per batch."""
    assert batches.dtype == EXTEND_BATCH_DTYPE and batches.flags.c_contiguous
    ev = None
    if events is not None:
        assert events.dtype == np.uint64 and len(events) >= 4 * len(batches)
        ev = events.ctypes.data
    _check(_lib.rx_extend_batches(C.byref(pool), layer, hq, batches.ctypes.data, len(batches),
                                  scale, ev, _stream(stream)))


class EventPool:
    """Timing events made by the library (``rx_events_create``), handed out
    in blocks and never reused while the pool lives; ``close`` destroys
    them."""

    def __init__(self, block=1024):
        self.block = block
        self.blocks = []
        self.cur = None
        self.used = 0

    def take(self, n):
        """A uint64 array of n fresh event handles (consecutive)."""
        if self.cur is None or self.used + n > len(self.cur):
            blk = np.zeros(max(self.block, n), dtype=np.uint64)
            _check(_lib.rx_events_create(len(blk), blk.ctypes.data))
            self.blocks.append(blk)
            self.cur, self.used = blk, 0
        out = self.cur[self.used:self.used + n]
        self.used += n
        return out

    def close(self):
        for blk in self.blocks:
            _lib.rx_events_destroy(len(blk), blk.ctypes.data)
        self.blocks, self.cur, self.used = [], None, 0


class NativeEvent:
    """One library event; ``elapsed_time(end)`` in milliseconds, as a
    torch.cuda.Event gives it."""
    __slots__ = ("h",)

    def __init__(self, h):
        self.h = int(h)

    def elapsed_time(self, end):
        ms = C.c_float()
        _check(_lib.rx_event_elapsed_ms(C.c_void_p(self.h), C.c_void_p(end.h), C.byref(ms)))
        return ms.value


def decode_steps(pool, layer, hq, d_table, steps, B, scale, d_workspace, stream=None):
    """rx_decode_steps over a ctypes array of rx_decode_step or a numpy array
    of DECODE_STEP_DTYPE records."""
    if isinstance(steps, np.ndarray):
        assert steps.dtype == DECODE_STEP_DTYPE and steps.flags.c_contiguous
        ptr = steps.ctypes.data
    else:
        ptr = C.cast(steps, C.c_void_p)
    _check(_lib.rx_decode_steps(C.byref(pool), layer, hq, d_table.data_ptr(), d_table.shape[1],
                                ptr, len(steps), B, scale, d_workspace.data_ptr(),
                                d_workspace.numel() * d_workspace.element_size(), _stream(stream)))


def verify_rows(prefix_len, prefix_rows, draft_indptr, parents, draft_slots, out_stride):
    """rx_verify_rows: (rows int32 [N, out_stride], ctx_len [N], positions [N])."""
    pl, pr = _i32(prefix_len), _i32(prefix_rows)
    di, par, ds = _i64(draft_indptr), _i32(parents), _i32(draft_slots)
    R, N = len(pl), len(par)
    rows = np.zeros((max(1, N), out_stride), dtype=np.int32)
    ctx = np.empty(max(1, N), dtype=np.int32)
    pos = np.empty(max(1, N), dtype=np.int32)
    _check(_lib.rx_verify_rows(R, _p(pl), _p(pr), pr.shape[1] if pr.ndim == 2 else 0, _p(di),
                               _p(par), _p(ds), _p(rows), int(out_stride), _p(ctx), _p(pos)))
    return rows[:N], ctx[:N], pos[:N]


def verify_attention(pool, layer, d_q, hq, d_table, d_plan, info, N, scale, d_out, d_lse,
                     d_workspace, stream=None):
    _check(_lib.rx_verify_attention(C.byref(pool), layer, d_q.data_ptr(), hq, d_table.data_ptr(),
                                    d_table.shape[1], d_plan.data_ptr(), C.byref(info), N, scale,
                                    d_out.data_ptr(), d_lse.data_ptr(), d_workspace.data_ptr(),
                                    d_workspace.numel() * d_workspace.element_size(),
                                    _stream(stream)))


def kv_copy(src_pool, dst_pool, d_src_slots, d_dst_slots, stream=None):
    """rx_kv_copy between (or within) pools given as rx_pool_desc."""
    _check(_lib.rx_kv_copy(C.byref(src_pool), C.byref(dst_pool), d_src_slots.data_ptr(),
                           d_dst_slots.data_ptr(), d_src_slots.numel(), _stream(stream)))


def decode_attention_static(pool, layer, d_q, hq, d_table, d_plan, info, B, scale, d_out, d_lse,
                            stream=None):
    """rx_decode_attention_static: decode with the library's own fixed scratch."""
    _check(_lib.rx_decode_attention_static(C.byref(pool), layer, d_q.data_ptr(), hq,
                                           d_table.data_ptr(), d_table.shape[1], d_plan.data_ptr(),
                                           C.byref(info), B, scale, d_out.data_ptr(),
                                           d_lse.data_ptr(), _stream(stream)))


def host_alloc(nbytes):
    """rx_host_alloc: address of `nbytes` of page-locked, device-mapped host
    memory (free with host_free)."""
    out = C.c_void_p()
    _check(_lib.rx_host_alloc(int(nbytes), C.byref(out)))
    return out.value


def host_free(ptr):
    _check(_lib.rx_host_free(ptr))


def device_check():
    flags = C.c_int32()
    st = _lib.rx_device_check(C.byref(flags))
    if st != RX_OK:
        raise RxError(st, last_error() + f" (flags {flags.value})")
    return flags.value
