"""Commit and rollback of the accepted prefix in KV cache and recurrent state (oracle; test
infrastructure only).

Sources (page titles and sections):

* lucebox-hub PR #15 "MTP speculative decoding", *Exactness*: "Rollback restores the
  KV/recurrent state bit-exactly"; every rollback case is cache- and logit-identical.
* DS4Server issue #98 "Add Qwen3.8 Flash Next native MTP speculation", *Implementation*:
  the recurrent state is snapshotted at every verify row, attention rows of rejected tokens are
  dropped, only the accepted prefix is kept, and re-running the ordinary forward is the
  fallback; nothing after an EOS is kept.
  *Completion requirements*: rejected rows leave every cache and recurrent component identical
  to ordinary decoding; capture-commit and fallback repair are both correct.
* llama.cpp PR #28104 "qwen4exp : port NextN/MTP speculative decoding to master", commits on
  full checkpoints, the replay livelock (replayed tokens are accepted, never re-verified) and
  on-device checkpoints.

Per request, one cycle fed k+1 verify rows (inputs x_0, d_1..d_k) at positions P..P+k. With
m = n_emit tokens emitted, the inputs that really belong to the sequence are x_0, t_1..t_{m-1}
(the last emitted token is next cycle's x_0, and an emitted EOS is never fed), so **the state
keeps exactly m rows**:

    KV:        rows [P, P+m) kept, rows [P+m, P+k+1) zero-filled, length P+m
               (reading: rows at or past the length are zero, so the whole buffer matches a
               run that never drafted)
    recurrent: snapshot commit  live <- slot[m]      (slot 0 = pre-cycle, slot r+1 = after row r)
               replay           live <- step^m(slot[0]) over rows 0..m-1
    conv rows: snapshot commit  conv <- conv_slot[m]
               replay           last C rows of concat(conv_slot[0], x_0..x_{m-1})

A request whose acceptance status is non-zero commits m = 0 (state restored to slot 0).

Index mode (this library's reading, not on the pages: a commit that moves no state). The live
state of a request is one of its slots, live_slot; the verify forward reads it there and writes
the state after verify row r into slot (live_slot + r + 1) mod n_slots, so the snapshot that
snapshot commit would copy (slot m above) already sits in slot (live_slot + m) mod n_slots, and
the commit makes that slot the live one. n_slots >= k + 2 keeps a cycle's k + 1 snapshots off
its own live slot.

The recurrent step is this project's synthetic stand-in for a gated linear-attention layer
(the real GDN update needs trained weights): per layer and head, with per-row inputs a (scalar
decay), b [dk], c [dv] and conv input x [W],

    S[i][j] <- fl32( fl32(a * S[i][j]) + fl32(b[i] * c[j]) )

every operation rounded separately to float32 (numpy float32 arithmetic, no fused
multiply-add), so snapshot commit and replay must agree byte for byte.

Pinned by: commit == the sequential no-draft run for every m and every EOS position, snapshot
commit == replay, index commit == snapshot commit for every live slot and m and over chained
cycles (each cycle's snapshots written relative to the previous commit's live slot), and closed
forms of the step (a = 1, b = 0 keeps S; S = 0 gives b (x) c;
small-integer inputs against exact integer arithmetic).
"""

import numpy as np


def synthetic_step(S, conv, a_t, b_t, c_t, x_t):
    """One recurrent step for all layers: S [L,H,dk,dv] f32, conv [L,C,W] f32, a_t [L,H],
    b_t [L,H,dk], c_t [L,H,dv], x_t [L,W]. Returns new (S, conv); inputs are not modified."""
    S = np.asarray(S, dtype=np.float32)
    a = np.asarray(a_t, dtype=np.float32)[:, :, None, None]
    outer = np.asarray(b_t, dtype=np.float32)[:, :, :, None] * \
        np.asarray(c_t, dtype=np.float32)[:, :, None, :]
    decayed = a * S
    S_new = decayed + outer
    conv = np.asarray(conv, dtype=np.float32)
    conv_new = np.concatenate([conv[:, 1:, :], np.asarray(x_t, dtype=np.float32)[:, None, :]],
                              axis=1)
    return S_new.astype(np.float32), conv_new.astype(np.float32)


def verify_snapshots(S0, conv0, a, b, c, x, n_rows):
    """What a verify forward captures: slot 0 = (S0, conv0), slot r+1 = after feeding row r."""
    slots_S = [np.array(S0, dtype=np.float32)]
    slots_conv = [np.array(conv0, dtype=np.float32)]
    for r in range(n_rows):
        S, cv = synthetic_step(slots_S[-1], slots_conv[-1], a[r], b[r], c[r], x[r])
        slots_S.append(S)
        slots_conv.append(cv)
    return np.stack(slots_S), np.stack(slots_conv)


def kept_rows(status, n_emit):
    """m: the number of verify rows the state keeps (0 when the cycle failed)."""
    return 0 if status != 0 else int(n_emit)


def kv_commit(kv, P, k, m):
    """KV trim: kv uint8 [layers, 2, capacity, row_bytes] holding rows [P, P+k] from the verify.
    Returns (new kv, new length). Rows [P+m, P+k+1) within capacity are zero-filled."""
    kv = np.array(kv, dtype=np.uint8, copy=True)
    cap = kv.shape[2]
    lo, hi = min(P + m, cap), min(P + k + 1, cap)
    kv[:, :, lo:hi, :] = 0
    return kv, P + m


def commit_snapshot(slots_S, slots_conv, m):
    """Snapshot commit: live <- slot[m] (copies)."""
    return np.array(slots_S[m], copy=True), np.array(slots_conv[m], copy=True)


def index_slot(live_slot, r, n_slots):
    """Index mode: the slot holding snapshot r of a cycle (r = 0 the pre-cycle state, r + 1
    the state after verify row r) whose live state is slot live_slot."""
    return (int(live_slot) + int(r)) % int(n_slots)


def commit_index(live_slot, m, n_slots):
    """Index commit: no state moves; the slot holding the state after the m kept rows becomes
    the live slot."""
    return index_slot(live_slot, m, n_slots)


def commit_replay(S0, conv0, a, b, c, x, m):
    """Restore the pre-cycle state and replay rows 0..m-1 with the synthetic step. The replayed
    rows are state updates only: they are never verified again (llama.cpp PR #28104, the
    fix for a replay that looped forever)."""
    S = np.array(S0, dtype=np.float32, copy=True)
    cv = np.array(conv0, dtype=np.float32, copy=True)
    for r in range(m):
        S, cv = synthetic_step(S, cv, a[r], b[r], c[r], x[r])
    return S, cv


def sequential_no_draft(kv_pre, P, kv_rows, S0, conv0, a, b, c, x, m):
    """Ordinary decoding of the m kept inputs one at a time: the reference the commit must
    reproduce byte for byte. kv_pre holds no rows at or past P; kv_rows [R, layers, 2,
    row_bytes] is what each input row writes at its position."""
    kv = np.array(kv_pre, dtype=np.uint8, copy=True)
    S = np.array(S0, dtype=np.float32, copy=True)
    cv = np.array(conv0, dtype=np.float32, copy=True)
    for r in range(m):
        kv[:, :, P + r, :] = kv_rows[r]
        S, cv = synthetic_step(S, cv, a[r], b[r], c[r], x[r])
    return kv, P + m, S, cv
