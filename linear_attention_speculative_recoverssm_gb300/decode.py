"""The deferred RecoverSSM of one layer across speculative decode steps.

A runner verifies a window per step, samples, and then must fold the
accepted tokens into each request's checkpoint.  The deferred form (page
"...cutedsl.kda.fused", module docstring; page "...recoverssm.kernels",
``_defer_commit_kernel`` and ``_prepare_flush_plan_kernel``) does not commit
after sampling: the accepted count becomes the request's pending replay, and
the next verify replays it in the same pass over the state.  This class only
sequences the library's entry points in that order; every step runs in the
library's kernels, on the given stream, with no host synchronisation, so a
sequence of steps can be captured in a CUDA graph.

* ``verify``: the fused replay + verify, or the stock verify (no replay) when
  the pending replays were just folded in by ``flush``;
* ``accept``: the accepted counts become the pending replays (defer); rows
  marked eager are committed at once from the records this step wrote;
* ``flush``: every pending replay is folded into its checkpoint in place
  (flush plan + commit); the next ``verify`` is then the stock one, because
  the plan leaves the pending counts as they are.
"""
from __future__ import annotations

from ._lib import (KDA_STATE_F32, kda_commit, kda_defer_commit, kda_flush_plan,
                   kda_replay_verify, kda_verify, layer_tables)


class DeferredRecoverSSM:
    """One layer's checkpoints, records and pending counts (device tensors,
    owned by the caller): state_pool FP32 [slots, H, 128, 128]; state_slots
    and record_rows int32 [B] (every live request needs a record row to be
    deferred); pending int32 [rows]; corr FP32 [rows, H, RQ, 128]; key_gate
    BF16 [rows, H, RQ, 256]; A_log FP32 [H]; dt_bias FP32 [H, 128]."""

    def __init__(self, state_pool, state_slots, record_rows, pending, corr, key_gate, A_log,
                 dt_bias, *, Q, lower_bound, q_scale, null_slot=0, split=0, status=None,
                 stream=None):
        import torch
        self.state_pool, self.state_slots, self.record_rows = state_pool, state_slots, record_rows
        self.pending, self.corr, self.key_gate = pending, corr, key_gate
        self.A_log, self.dt_bias = A_log, dt_bias
        self.Q, self.lower_bound, self.q_scale = Q, lower_bound, q_scale
        self.null_slot, self.split, self.status, self.stream = null_slot, split, status, stream
        self.B, self.H = state_slots.shape[0], A_log.shape[0]
        dev = state_pool.device
        # the commit's one-layer address tables and the flush plan's outputs,
        # made once so that no step allocates or copies from the host
        self._tables = layer_tables([state_pool], [corr], [key_gate], dev)
        self._plan = {name: torch.zeros(self.B, dtype=torch.int32, device=dev)
                      for name in ("commit_lens", "final_slots", "boundary_slots",
                                   "boundary_lens")}
        self.flushed = False

    def _commit(self, commit_lens, destinations, boundaries=None, boundary_lens=None):
        kda_commit(*self._tables, self.A_log, self.dt_bias, self.state_slots, commit_lens,
                   destinations, state_dtype=KDA_STATE_F32, lower_bound=self.lower_bound,
                   L=1, H=self.H, B=self.B, Q=self.corr.shape[2],
                   n_slots=self.state_pool.shape[0], n_rows=self.corr.shape[0],
                   boundaries=boundaries, boundary_lens=boundary_lens,
                   record_rows=self.record_rows, null_slot=self.null_slot, status=self.status,
                   stream=self.stream)

    def verify(self, q, k, v, raw_g, raw_beta, out, query_start_loc=None):
        """Verify this step's window (q, k, v, raw_g BF16 [T, H, 128],
        raw_beta BF16 [T, H]; T = B*Q, or packed windows of q_b <= Q tokens
        given by query_start_loc [B + 1]) into out BF16 [T, H, 128], writing
        the window's records.  With windows of different lengths the counts
        passed to ``accept`` must not exceed each request's q_b."""
        common = dict(Q=self.Q, lower_bound=self.lower_bound, q_scale=self.q_scale,
                      null_slot=self.null_slot, status=self.status, stream=self.stream,
                      query_start_loc=query_start_loc)
        if self.flushed:
            kda_verify(q, k, v, raw_g, raw_beta, self.A_log, self.dt_bias, self.state_pool,
                       self.state_slots, self.corr, self.key_gate, out,
                       record_rows=self.record_rows, **common)
        else:
            kda_replay_verify(q, k, v, raw_g, raw_beta, self.A_log, self.dt_bias,
                              self.state_pool, self.state_slots, self.record_rows,
                              self.pending, self.corr, self.key_gate, out, split=self.split,
                              **common)

    def accept(self, accepted, eager=None):
        """After sampling: ``accepted`` (int32 [B], overwritten: it ends as
        the commit plan, non-zero only on eager rows) becomes each request's
        pending replay; ``eager`` (uint8 [B] or None) marks rows committed
        now instead."""
        kda_defer_commit(self.state_slots, accepted, self.record_rows, self.pending,
                         eager=eager, null_slot=self.null_slot, status=self.status,
                         stream=self.stream)
        if eager is not None:
            self._commit(accepted, self.state_slots)
        self.flushed = False

    def flush(self):
        """Fold every pending replay into its checkpoint, in place."""
        p = self._plan
        kda_flush_plan(self.state_slots, self.record_rows, self.pending, p["commit_lens"],
                       p["final_slots"], p["boundary_slots"], p["boundary_lens"],
                       Q=self.Q, null_slot=self.null_slot, status=self.status,
                       stream=self.stream)
        self._commit(p["commit_lens"], p["final_slots"], p["boundary_slots"],
                     p["boundary_lens"])
        self.flushed = True
