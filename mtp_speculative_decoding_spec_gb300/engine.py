"""SpecVerifyEngine: owns the device buffers of one verify-step configuration and enqueues the
cycle -- k draft-head steps, the verify LM head, acceptance, commit -- on one CUDA stream.

PyTorch provides device memory and the stream; every step runs in libspec.so's kernels. No call
here reads a result back to the host except ``cycle_from_host``, which is the end-to-end path:
it copies one cycle's inputs from pinned host memory, runs the cycle and copies the 64-byte
results back, all asynchronously on the stream.
"""

import torch

from . import (ACCEPT_OUT_BYTES, COUNTERS_BYTES, ROWSTATS_BYTES, SPEC_F32,
               WIDTH_STATE_BYTES, spec_accept, spec_accept_exact, spec_accept_filtered,
               spec_adapt_width,
               spec_commit_rollback, spec_draft_argmax, spec_lmhead_verify,
               spec_workspace_bytes)


class SpecVerifyEngine:
    def __init__(self, W, wdt, V, d, Vd, B, R, k_max, eos_id=-1, device="cuda:0",
                 want_q_logits=True, acceptance="ratio", adaptive_cost=None, alpha=0.1):
        """acceptance: "ratio" (u*q <= p with residual correction; spec_accept), "exact"
        (a draft counts only if it is the trunk's own sample; spec_accept_exact) or "filtered"
        (the top-k / top-p filtered target of set_requests(top_k=..., top_p=...), argmax drafts
        and one-hot q; spec_accept_filtered; the draft steps then run at temperature 0).
        adaptive_cost: None for fixed widths (set_requests(k=...)), or the relative cost of a
        cycle at widths 0..k_max: each cycle then ends with spec_adapt_width choosing every
        request's next width on the device, and ``cycle`` always enqueues k_max draft steps,
        of which those past every request's width return at once."""
        if acceptance not in ("ratio", "exact", "filtered"):
            raise ValueError(
                f"acceptance must be 'ratio', 'exact' or 'filtered', not {acceptance!r}")
        self.acceptance = acceptance
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

    # ---------------------------------------------------------------- configuration
    def set_requests(self, temps=None, seeds=None, pos=None, k=None, top_k=None, top_p=None):
        for dst, src in ((self.temps, temps), (self.seeds, seeds), (self.pos, pos),
                         (self.k, k), (self.top_k, top_k), (self.top_p, top_p)):
            if src is not None:
                dst.copy_(torch.as_tensor(src, dtype=dst.dtype), non_blocking=True)

    def attach_state(self, desc, mode):
        """A spec_state_desc (device pointers) committed after every acceptance."""
        self.state, self.state_mode = desc, mode

    # ---------------------------------------------------------------- the cycle
    def draft_step(self, i, h):
        """Draft i (1-based) for every request from draft-head hidden rows h [B, d]."""
        B = self.B
        temps = self.zero_temps if self.acceptance == "filtered" else self.temps
        spec_draft_argmax(self.W, self.wdt, self.Vd, self.d, h, B, temps, self.seeds,
                          self.pos, i - 1, self.drafts[:, i - 1:], self.drafts.shape[1],
                          None if self.q is None else self.q[(i - 1) * B:], self.Vd,
                          self.qs[(i - 1) * B * ROWSTATS_BYTES:],
                          self.k if self.adaptive else None, self.ws)

    def verify(self, H):
        spec_lmhead_verify(self.W, self.wdt, self.V, self.d, H, self.B, self.R, self.temps,
                           self.logits, self.stats, self.ws)

    def accept(self, use_q=True):
        if self.acceptance == "filtered":
            spec_accept_filtered(self.B, self.k_max, self.k, self.drafts, self.logits, self.stats,
                                 self.V, self.R, self.temps, self.top_k, self.top_p, self.eos_id,
                                 self.seeds, self.pos, self.out, self.counters, self.ws)
            return
        if self.acceptance == "exact":
            spec_accept_exact(self.B, self.k_max, self.k, self.drafts, self.logits, self.stats,
                              self.V, self.R, self.temps, self.eos_id, self.seeds, self.pos,
                              self.out, self.counters, self.ws)
            return
        q = self.q if (use_q and self.q is not None) else None
        spec_accept(self.B, self.k_max, self.k, self.drafts, self.logits, self.stats, self.V,
                    self.R, q, self.qs if q is not None else None, self.Vd, self.Vd, self.temps,
                    self.eos_id, self.seeds, self.pos, self.out, self.counters, self.ws)

    def commit(self):
        if self.state is not None:
            spec_commit_rollback(self.B, self.state, self.out, self.k, self.state_mode,
                                 self.commit_status)

    def adapt(self):
        if self.adaptive:
            spec_adapt_width(self.B, self.k_max, self.out, self.k, self.cost, self.alpha,
                             self.width_state, self.k)

    def verify_cycle(self, H):
        """Verify + accept (+ commit, + the next width when adaptive): one verify cycle on
        device-resident inputs."""
        self.verify(H)
        self.accept()
        self.commit()
        self.adapt()

    def cycle(self, H, Hd, k):
        """Full cycle: k draft steps (Hd [k, B, d]; k_max of them when adaptive), verify,
        accept, commit."""
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
