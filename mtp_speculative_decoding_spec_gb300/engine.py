"""SpecVerifyEngine: owns the device buffers of one verify-step configuration and enqueues the
cycle -- k draft-head steps, the verify LM head, acceptance, commit -- on one CUDA stream.

PyTorch provides device memory and the stream; every step runs in libspec.so's kernels. No call
here reads a result back to the host except ``cycle_from_host``, which is the end-to-end path:
it copies one cycle's inputs from pinned host memory, runs the cycle and copies the 64-byte
results back, all asynchronously on the stream.

In adaptive mode with one request the cycle is, by default, a CUDA graph
(spec_width_graph_create): a select kernel reads the width the device chose and a switch runs
the body captured for that width -- its draft steps, a verify of width + 1 rows, acceptance,
commit and the next width -- so the host never learns the width and no idle draft step is
enqueued. With ``width_lag`` the host schedules the widths instead, one cycle late: the width
update also writes each choice through the device alias of pinned host memory
(spec_adapt_width_mirror), and the host enqueues cycle n at the width chosen after cycle n - 2,
read once that cycle's event has completed (the device is then running cycle n - 1). Each cycle
is then exactly its width's launches: no graph boundary, no select kernel, no copy of the
inputs into captured buffers, no idle draft step.
"""

import torch

from . import (ACCEPT_OUT_BYTES, COUNTERS_BYTES, ROWSTATS_BYTES, SPEC_F32,
               WIDTH_STATE_BYTES, spec_accept, spec_accept_exact, spec_accept_filtered,
               spec_adapt_width, spec_adapt_width_mirror, spec_host_alias,
               spec_commit_rollback, spec_draft_argmax, spec_graph_capture_begin,
               spec_graph_capture_end, spec_graph_destroy, spec_graph_instantiate,
               spec_graph_launch, spec_lmhead_verify, spec_verify_accept_greedy,
               spec_width_graph_create, spec_workspace_bytes)


class SpecVerifyEngine:
    def __init__(self, W, wdt, V, d, Vd, B, R, k_max, eos_id=-1, device="cuda:0",
                 want_q_logits=True, acceptance="ratio", adaptive_cost=None, alpha=0.1,
                 cycle_cost=None, width_graph=None, width_lag=False, fuse_greedy=False):
        """acceptance: "ratio" (u*q <= p with residual correction; spec_accept), "exact"
        (a draft counts only if it is the trunk's own sample; spec_accept_exact) or "filtered"
        (the top-k / top-p filtered target of set_requests(top_k=..., top_p=...), argmax drafts
        and one-hot q; spec_accept_filtered; the draft steps then run at temperature 0).
        adaptive_cost: None for fixed widths (set_requests(k=...)), or the prior relative cost
        of a cycle at widths 0..k_max: each cycle then ends with spec_adapt_width choosing every
        request's next width on the device.
        cycle_cost: in adaptive mode, a device tensor [B] of each cycle's measured cost for the
        cost fit (the caller keeps it current), or None to time the cycles on the device.
        width_graph: run adaptive cycles as a width graph (default: when B == 1); otherwise
        ``cycle`` enqueues k_max draft steps, of which those past every request's width return
        at once, and a verify of R rows.
        width_lag: run adaptive cycles of one request at host-scheduled widths, one cycle late
        (see the module doc); replaces the width graph.
        fuse_greedy: while every request is greedy (set_requests' temperatures <= 0) and the
        rule is the ratio rule, run a cycle's verify and acceptance as one launch
        (spec_verify_accept_greedy: the acceptance taken in the LM-head kernel's last block)."""
        if acceptance not in ("ratio", "exact", "filtered"):
            raise ValueError(
                f"acceptance must be 'ratio', 'exact' or 'filtered', not {acceptance!r}")
        self.acceptance = acceptance
        self.fuse_greedy = bool(fuse_greedy)
        self.all_greedy = False  # set_requests' temperatures, as the host gave them
        self.W, self.wdt, self.V, self.d, self.Vd = W, wdt, V, d, Vd
        self.B, self.R, self.k_max, self.eos_id = B, R, k_max, eos_id
        dev = torch.device(device)
        self.device = dev
        n = spec_workspace_bytes(V, B)
        self.ws = torch.zeros((n + 255) // 256 * 256, dtype=torch.uint8, device=dev)
        self.logits = torch.empty((B * R, V), dtype=torch.float32, device=dev)
        self.stats = torch.zeros(B * R * ROWSTATS_BYTES, dtype=torch.uint8, device=dev)
        kq = max(k_max, 1)
        self.q = torch.empty((kq * B, Vd), dtype=torch.float32, device=dev) if want_q_logits \
            else None
        self.qs = torch.zeros(kq * B * ROWSTATS_BYTES, dtype=torch.uint8, device=dev)
        self.drafts = torch.zeros((B, kq), dtype=torch.int32, device=dev)
        self.out = torch.zeros(B * ACCEPT_OUT_BYTES, dtype=torch.uint8, device=dev)
        self.counters = torch.zeros(B * COUNTERS_BYTES, dtype=torch.uint8, device=dev)
        self.temps = torch.zeros(B, dtype=torch.float32, device=dev)
        self.zero_temps = torch.zeros(B, dtype=torch.float32, device=dev)
        self.top_k = torch.full((B,), 20, dtype=torch.int32, device=dev)
        self.top_p = torch.full((B,), 0.95, dtype=torch.float32, device=dev)
        self.seeds = torch.zeros(B, dtype=torch.int64, device=dev)
        self.pos = torch.zeros(B, dtype=torch.int64, device=dev)
        self.k = torch.full((B,), k_max, dtype=torch.int32, device=dev)
        self.commit_status = torch.zeros(B, dtype=torch.int32, device=dev)
        self.state = None
        self.dtype_bytes = 4 if wdt == SPEC_F32 else 2  # bytes per hidden-row element
        self.adaptive = adaptive_cost is not None
        self.alpha = alpha
        if self.adaptive:
            if len(adaptive_cost) != k_max + 1:
                raise ValueError("adaptive_cost needs k_max + 1 entries")
            self.cost = torch.tensor(adaptive_cost, dtype=torch.float32, device=dev)
            self.width_state = torch.zeros(B * WIDTH_STATE_BYTES, dtype=torch.uint8, device=dev)
        self.cycle_cost = cycle_cost
        self.width_lag = bool(width_lag) and self.adaptive
        if width_lag and not self.adaptive:
            raise ValueError("width_lag schedules adaptive widths: give adaptive_cost")
        self.width_graph = self.adaptive and not self.width_lag and (
            B == 1 if width_graph is None else width_graph)
        if (self.width_graph or self.width_lag) and B != 1:
            raise ValueError("width graphs and host-scheduled widths run one request (the "
                             "verify rows of a width are contiguous only for one)")
        if self.width_lag:
            # slot n % 2: the widths of cycle n on the device, and their host-visible copy
            self.k_ring = torch.full((2, B), k_max, dtype=torch.int32, device=dev)
            if dev.type == "cuda":
                self.k_seen = torch.full((2, B), k_max, dtype=torch.int32).pin_memory()
                self.k_seen_dev = [spec_host_alias(self.k_seen[i]) for i in range(2)]
                self.lag_events = [torch.cuda.Event(), torch.cuda.Event()]
            else:  # the host-logic tests: no kernel runs, nothing to wait for
                self.k_seen = torch.full((2, B), k_max, dtype=torch.int32)
                self.k_seen_dev = [self.k_seen[i].data_ptr() for i in range(2)]
                self.lag_events = None
            self.n_cycles = 0
            self.last_width = None
        self.graph = self.graph_exec = None
        if self.width_graph:
            et = torch.float32 if wdt == SPEC_F32 else torch.int16
            self.H_in = torch.zeros((k_max + 1, d), dtype=et, device=dev)
            self.Hd_in = torch.zeros((max(k_max, 1), 1, d), dtype=et, device=dev)

    # ---------------------------------------------------------------- configuration
    def set_requests(self, temps=None, seeds=None, pos=None, k=None, top_k=None, top_p=None):
        if temps is not None:
            self.all_greedy = bool((torch.as_tensor(temps, dtype=torch.float32) <= 0).all())
        for dst, src in ((self.temps, temps), (self.seeds, seeds), (self.pos, pos),
                         (self.k, k), (self.top_k, top_k), (self.top_p, top_p)):
            if src is not None:
                dst.copy_(torch.as_tensor(src, dtype=dst.dtype), non_blocking=True)
        if k is not None and self.width_lag:  # the first two cycles run at these widths
            kk = torch.as_tensor(k, dtype=torch.int32)
            self.k_ring.copy_(kk.expand(2, self.B), non_blocking=True)
            self.k_seen.copy_(kk.expand(2, self.B))
            self.n_cycles = 0

    def attach_state(self, desc, mode):
        """A spec_state_desc (device pointers) committed after every acceptance."""
        self.state, self.state_mode = desc, mode

    # ---------------------------------------------------------------- the cycle
    def draft_step(self, i, h, gate=True, k_active=None):
        """Draft i (1-based) for every request from draft-head hidden rows h [B, d]; k_active:
        the widths that gate the step (default: the engine's widths when adaptive)."""
        B = self.B
        if k_active is None and self.adaptive and gate:
            k_active = self.k
        temps = self.zero_temps if self.acceptance == "filtered" else self.temps
        spec_draft_argmax(self.W, self.wdt, self.Vd, self.d, h, B, temps, self.seeds,
                          self.pos, i - 1, self.drafts[:, i - 1:], self.drafts.shape[1],
                          None if self.q is None else self.q[(i - 1) * B:], self.Vd,
                          self.qs[(i - 1) * B * ROWSTATS_BYTES:], k_active, self.ws)

    def verify(self, H, R=None):
        spec_lmhead_verify(self.W, self.wdt, self.V, self.d, H, self.B, R or self.R, self.temps,
                           self.logits, self.stats, self.ws)

    def accept(self, use_q=True, R=None, k=None):
        R = R or self.R
        k = self.k if k is None else k
        if self.acceptance == "filtered":
            spec_accept_filtered(self.B, self.k_max, k, self.drafts, self.logits, self.stats,
                                 self.V, R, self.temps, self.top_k, self.top_p, self.eos_id,
                                 self.seeds, self.pos, self.out, self.counters, self.ws)
            return
        if self.acceptance == "exact":
            spec_accept_exact(self.B, self.k_max, k, self.drafts, self.logits, self.stats,
                              self.V, R, self.temps, self.eos_id, self.seeds, self.pos,
                              self.out, self.counters, self.ws)
            return
        q = self.q if (use_q and self.q is not None) else None
        spec_accept(self.B, self.k_max, k, self.drafts, self.logits, self.stats, self.V,
                    R, q, self.qs if q is not None else None, self.Vd, self.Vd, self.temps,
                    self.eos_id, self.seeds, self.pos, self.out, self.counters, self.ws)

    def verify_accept(self, H, R=None, k=None, k_mirror=None):
        """Verify rows H and acceptance: one fused launch when greedy (see fuse_greedy). With
        k_mirror (adaptive, host-scheduled widths) the fused launch also takes the width update,
        into k and k_mirror; returns whether it did."""
        R = R or self.R
        k = self.k if k is None else k
        if self.fuse_greedy and self.all_greedy and self.acceptance == "ratio":
            adapt = k_mirror is not None and self.adaptive
            spec_verify_accept_greedy(self.W, self.wdt, self.V, self.d, H, self.B, R, self.temps,
                                      self.logits, self.stats, self.k_max, k, self.drafts,
                                      self.eos_id, self.out, self.counters, self.ws,
                                      cost=self.cost if adapt else None,
                                      cycle_cost=self.cycle_cost if adapt else None,
                                      alpha=self.alpha if adapt else 0.1,
                                      state=self.width_state if adapt else None,
                                      k_next=k if adapt else None,
                                      k_mirror=k_mirror if adapt else None)
            return adapt
        self.verify(H, R=R)
        self.accept(R=R, k=k)
        return False

    def commit(self, k=None):
        if self.state is not None:
            spec_commit_rollback(self.B, self.state, self.out, self.k if k is None else k,
                                 self.state_mode, self.commit_status)

    def adapt(self):
        if self.adaptive:
            spec_adapt_width(self.B, self.k_max, self.out, self.k, self.cost, self.cycle_cost,
                             self.alpha, self.width_state, self.k)

    def verify_cycle(self, H):
        """Verify + accept (+ commit, + the next width when adaptive): one verify cycle on
        device-resident inputs."""
        self.verify_accept(H)
        self.commit()
        self.adapt()

    def _cycle_lagged(self, H, Hd):
        """Cycle n at the width chosen after cycle n - 2 (the first two at set_requests' k)."""
        n = self.n_cycles
        s = n % 2
        if n >= 2 and self.lag_events is not None:
            self.lag_events[s].synchronize()  # cycle n - 2 (and its width update) has completed
        w = min(max(int(self.k_seen[s].max()), min(self.k_max, 1)), self.k_max)
        k_dev = self.k_ring[s]
        for i in range(1, w + 1):
            self.draft_step(i, Hd[i - 1], gate=False)
        # the choice after this cycle is cycle n + 2's width: slot s again, on both sides
        if self.state is None:
            # nothing to commit: the width update can share the fused verify's launch
            fused = self.verify_accept(H[:w + 1], R=w + 1, k=k_dev, k_mirror=self.k_seen_dev[s])
        else:
            # the commit reads this cycle's widths, which the update overwrites: it goes first
            self.verify_accept(H[:w + 1], R=w + 1, k=k_dev)
            self.commit(k=k_dev)
            fused = False
        if not fused:
            spec_adapt_width_mirror(self.B, self.k_max, self.out, k_dev, self.cost,
                                    self.cycle_cost, self.alpha, self.width_state, k_dev,
                                    self.k_seen_dev[s])
        if self.lag_events is not None:
            self.lag_events[s].record()
        self.n_cycles = n + 1
        self.last_width = w

    def _width_body(self, w):
        """The cycle at width w (w >= 1), on the current stream: what a width graph's body w
        holds (body 0, never chosen, runs width 1)."""
        w = max(w, 1)
        for i in range(1, w + 1):
            self.draft_step(i, self.Hd_in[i - 1], gate=False)
        self.verify_accept(self.H_in[:w + 1], R=w + 1)
        self.commit()
        self.adapt()

    def _build_width_graph(self):
        n = self.k_max + 1
        if self.device.type == "cuda":  # capture on a stream of its own
            torch.cuda.synchronize(self.device)
            stream = torch.cuda.Stream(self.device)
            stream.wait_stream(torch.cuda.current_stream(self.device))
            ctx = torch.cuda.stream(stream)
        else:  # the host-logic tests, whose library calls are recorded rather than run
            import contextlib
            stream, ctx = None, contextlib.nullcontext()
        self.graph, bodies = spec_width_graph_create(n, self.k, self.B)
        with ctx:
            for w in range(n):
                spec_graph_capture_begin(bodies[w], stream)
                try:
                    self._width_body(w)
                finally:
                    spec_graph_capture_end(stream)
        self.graph_exec = spec_graph_instantiate(self.graph)

    def close(self):
        """Release the width graph, if any (the engine's tensors are freed by PyTorch)."""
        if self.graph is not None:
            spec_graph_destroy(self.graph, self.graph_exec)
            self.graph = self.graph_exec = None

    def __del__(self):
        try:
            self.close()
        except Exception:  # interpreter shutdown: the library may be gone already
            pass

    def cycle(self, H, Hd, k):
        """Full cycle: k draft steps (Hd [k, B, d]), verify, accept, commit. Adaptive: the
        width chosen on the device; H holds k_max + 1 rows and Hd k_max rows, of which the
        width's first ones are used (a width graph), or k_max draft steps are enqueued, those
        past every request's width returning at once."""
        if self.width_lag:
            self._cycle_lagged(H, Hd)
            return
        if self.width_graph:
            if self.graph_exec is None:
                self._build_width_graph()
            self.H_in[:H.shape[0]].copy_(H.reshape(H.shape[0], -1))
            self.Hd_in[:Hd.shape[0]].copy_(Hd.reshape(Hd.shape[0], 1, -1))
            spec_graph_launch(self.graph_exec)
            return
        for i in range(1, (self.k_max if self.adaptive else k) + 1):
            self.draft_step(i, Hd[i - 1])
        self.verify_cycle(H)

    def cycle_from_host(self, H_host, Hd_host, k, out_host, H_dev, Hd_dev):
        """End-to-end cycle: pinned host inputs -> device, the cycle, results -> pinned host."""
        H_dev.copy_(H_host, non_blocking=True)
        if k > 0:
            Hd_dev[:k].copy_(Hd_host[:k], non_blocking=True)
        self.cycle(H_dev, Hd_dev, k)
        out_host.copy_(self.out, non_blocking=True)
