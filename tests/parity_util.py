"""Helpers of the GPU parity tests: run a workload through librx on the GPU,
collect sampled attention outputs, and compare them with the fp64 oracle
computed from the workload's token streams (never from the pool)."""

import numpy as np

from oracle import attention as oatt
from oracle.harness import run_bookkeeping

MAX_ABS = 1e-2    # attention tolerance vs fp64 (bf16 inputs, fp32 accumulation)
MEAN_ABS = 1e-3


class DeviceRun:
    def __init__(self, wl, layers=None, sample=None, extend_tokens=None, decode_steps=None,
                 check_bookkeeping=True, values_fn=None, policy="fcfs", chunk_tokens=None,
                 host_slots=0):
        import torch

        from radix_tree_prefix_gb300 import rx, workloads
        from radix_tree_prefix_gb300.engine import Engine, GatherInputs

        self.torch = torch
        self.wl = wl
        self.layers = list(range(wl.num_layers)) if layers is None else list(layers)
        self.sample = None if sample is None else set(sample)
        self.extend_tokens = extend_tokens
        self.decode_sel = None if decode_steps is None else set(decode_steps)
        self.dev = torch.device("cuda:0")
        self.vals = workloads.make_values(wl, self.dev, self.layers)
        if values_fn is not None:  # reshape the inputs (both sides read self.vals)
            values_fn(self.vals)
        self.ext = {}
        self.dec = {}
        self.rng = np.random.default_rng(123)
        eng = Engine(wl, device=self.dev, inputs=GatherInputs(wl, self.vals, self.layers),
                     layers=self.layers, on_extend=self._on_extend, on_decode=self._on_decode,
                     policy=policy, chunk_tokens=chunk_tokens, host_slots=host_slots)
        self.trace = eng.run()
        torch.cuda.synchronize()
        self.flags = rx.device_check()
        self.engine = eng
        if check_bookkeeping:
            want, _ = run_bookkeeping(wl.oracle_waves(), wl.num_slots, wl.decode_steps,
                                      page_size=wl.page_size, policy=policy,
                                      host_slots=host_slots)
            assert self.trace.as_tuple() == want.as_tuple(), "bookkeeping differs from oracle"

    def _pick_tokens(self, s):
        if self.extend_tokens is None or s <= self.extend_tokens:
            return np.arange(s)
        k = self.extend_tokens
        pick = set([0, s - 1, s // 2]) | set(self.rng.choice(s, size=k - 3, replace=False).tolist())
        return np.array(sorted(pick))

    def _on_extend(self, batch_no, rids, prefix, qo, outs):
        for i, rid in enumerate(rids):
            if self.sample is not None and rid not in self.sample:
                continue
            sel = self._pick_tokens(int(qo[i + 1] - qo[i]))
            idx = self.torch.from_numpy(qo[i] + sel).to(self.dev)
            for layer in self.layers:
                o, lse = outs[layer]
                self.ext[(rid, layer)] = (int(prefix[i]), sel,
                                          o.index_select(0, idx).double().cpu().numpy(),
                                          lse.index_select(0, idx).double().cpu().numpy())

    def _on_decode(self, step_no, t, rids, ctx, outs, info):
        if self.decode_sel is not None and t not in self.decode_sel:
            return
        for i, rid in enumerate(rids):
            if self.sample is not None and rid not in self.sample:
                continue
            for layer in self.layers:
                o, lse = outs[layer]
                self.dec[(rid, t, layer)] = (o[i].double().cpu().numpy(),
                                             lse[i].double().cpu().numpy())

    def _rows(self, kind, layer, idx):
        t = self.torch.from_numpy(np.asarray(idx, dtype=np.int64)).to(self.dev)
        return self.vals[kind][layer].index_select(0, t).double().cpu().numpy()

    def compare(self):
        """Returns (max abs error, mean abs error, number of rows compared)."""
        wl = self.wl
        errs = []
        n = 0
        self.worst = {}
        for (rid, layer), (m, sel, o, lse) in self.ext.items():
            r = wl.requests[rid]
            pidx = wl.prompt_store_index(r)
            q = self._rows("q", layer, pidx[m:][sel])
            k = self._rows("k", layer, pidx)
            v = self._rows("v", layer, pidx)
            want_o, want_l = oatt.softmax_attention(q, k, v, m + sel + 1)
            errs.append(np.abs(o - want_o).ravel())
            errs.append(np.abs(lse - want_l).ravel())
            self.worst[("extend", rid, layer)] = float(max(errs[-1].max(), errs[-2].max()))
            n += len(sel)
        for (rid, t, layer), (o, lse) in self.dec.items():
            r = wl.requests[rid]
            pidx = wl.prompt_store_index(r)
            oidx = wl.output_store_index(r)
            ctx = np.concatenate([pidx, oidx[:t + 1]])
            want_o, want_l = oatt.decode_attention(self._rows("q", layer, [oidx[t]])[0],
                                                   self._rows("k", layer, ctx),
                                                   self._rows("v", layer, ctx))
            errs.append(np.abs(o - want_o).ravel())
            errs.append(np.abs(lse - want_l).ravel())
            self.worst[("decode", rid, t, layer)] = float(max(errs[-1].max(), errs[-2].max()))
            n += 1
        e = np.concatenate(errs)
        return float(e.max()), float(e.mean()), n

    def assert_close(self):
        mx, mean, n = self.compare()
        assert n > 0
        assert self.flags == 0
        bad = sorted(((v, k) for k, v in self.worst.items() if v > MAX_ABS), reverse=True)
        assert mx <= MAX_ABS, f"max abs error {mx} over {n} rows; worst: {bad[:6]}"
        assert mean <= MEAN_ABS, f"mean abs error {mean} over {n} rows"
        return mx, mean, n
