"""Drafting and acceptance for one request and one verify cycle (oracle; test infrastructure only).

Sources (page titles and sections):

* lucebox-hub PR #15 "MTP speculative decoding", *What*: the draft head chooses its token as
  the argmax over the first 64,000 vocabulary rows; one trunk pass over k+1 rows checks k
  drafts. *Exactness*: a greedy draft survives only when it is the trunk's own token, so the
  emitted bytes are those of decoding without drafts. *Speed*: 7.74 tokens per cycle at seven drafts implies
  k+1 tokens when every draft passes -- the bonus token from the last verify row.
* DS4Server issue #98 "Add Qwen3.8 Flash Next native MTP speculation", *Implementation* and the
  closing comment: a draft is kept when ``u*q <= p``, a rejection is replaced by a draw from
  ``max(0, p - q)``, zero and non-finite probabilities get defined outcomes, and an EOS among
  the drafts ends the block with nothing, token or state, kept past it.

The algorithm, per request (row r of the verify logits predicts the token after input r; draft
d_i is checked against verify row i-1; ``pos_base`` is the absolute position of the first
token this cycle emits):

T == 0 (greedy):
    for i = 1..k: t = argmax z[i-1]; if d_i == t: emit d_i (stop if EOS) else emit t, stop.
    all k accepted: emit argmax z[k] (bonus).
T > 0 (ratio rule), p_r = softmax(z[r]/T) over V, q_i = softmax(y[i]/T) over the draft rows and
0 beyond them (q_i = one-hot at d_i when no draft logits are given):
    for i = 1..k: u = U(pos_base+i-1, ACCEPT)
        if p_{i-1}(d_i) > 0 and u * q_i(d_i) <= p_{i-1}(d_i): emit d_i (stop if EOS)
        else: r = max(0, p_{i-1} - q_i); if sum r <= 0: r = p_{i-1}
              emit the inverse-CDF draw of r with U(pos_base+i-1, RESIDUAL); stop.
    all k accepted: emit the inverse-CDF draw of p_k with U(pos_base+k, BONUS).

Exact-match mode at T > 0 (``accept_request_exact``): the trunk's own token at each position is
the inverse-CDF draw of p_{i-1} with U(pos_base+i-1, BONUS); a draft is kept iff it equals that
token, the first mismatch emits the token, and all k kept emit the draw from p_k. The output is
then token-identical to decoding without drafts under the same seed (pinned against a sequential
sampler written independently in the tests).

Filtered sampling (``accept_request_filtered``; llama.cpp PR #28104, *Result*: the trunk samples
at temperature 1.0 with top-p 0.95 and top-k 20). The target becomes p'_r = the temperature-T
distribution of row r kept to its top_k tokens (largest logits, ties to the lower id), then to
the smallest prefix of those in descending probability whose mass over the top-k set reaches
top_p, renormalised. Drafts are the draft head's argmax picks and q is one-hot at the draft, so
the ratio rule keeps d_i when u <= p'_{i-1}(d_i), a rejection draws from p'_{i-1} without d_i,
and the bonus draws from p'_k: the emitted tokens follow the filtered target law exactly.

Draft set: lucebox-hub PR #15, *What*: the draft head covers 64,000 rows, the control and
special tokens plus the lowest ids. Read as two ranges, the lowest n_low ids and n_high rows
from hi_first (where a tokenizer keeps its special tokens): draft row r is vocabulary id r for
r < n_low, hi_first + r - n_low after. ``rows`` (the vocabulary ids of the draft rows, in
order) carries that map through ``draft_token``, ``draft_chain_tokens`` and ``accept_request``;
without it the draft rows are ids 0 .. Vd-1. q is zero at ids outside the set.

Inverse CDF: the smallest j (ascending token id) with cumsum(w)[j] > u * sum(w); if rounding
leaves none, the last j with w[j] > 0. Readings where the pages are silent are listed in the
design notes (draft rows checked against row i-1, lowest-index argmax ties, ``<=`` in the ratio
test, rejection when p(d) == 0 even at u == 0, fall back to p when the residual is empty, an
emitted EOS from a correction or bonus also ends the block).

Status codes (no decision is taken and nothing is emitted when status != 0):
    1 non-finite verify logits (NaN or +Inf anywhere in a row used, or a row of all -Inf),
      or non-finite draft logits at T > 0; 2 k outside [0, k_max]; 5 a draft id outside [0, V).

Every decision records a margin so the GPU comparison can set aside near-ties: ('gap', top-2
logit gap) for argmax decisions, ('ratio', |u*q - p|) for ratio tests and ('cdf', distance from
u*sum(w) to the nearest cumulative boundary) for inverse-CDF draws, both in probability units.

Pinned by: brute-force enumeration of the emitted-sequence law at V=8 (exact against the
chained target law within the 24-bit grid error), a chi-square test at V=4096, the T=0 identity
with sequential greedy decoding, and the special cases p == q (all accepted) and q one-hot on a
token with p == 0 (always rejected, residual == p).
"""

import numpy as np

from . import lmhead
from .philox import PURPOSE_ACCEPT, PURPOSE_BONUS, PURPOSE_DRAFT, PURPOSE_RESIDUAL

STATUS_OK = 0
STATUS_NONFINITE = 1
STATUS_BAD_K = 2
STATUS_BAD_TOKEN = 5


def inverse_cdf(w, u):
    """Inverse-CDF draw from non-negative weights ``w`` with uniform ``u`` in [0, 1).

    Returns (j, margin): j = the smallest index with cumsum(w)[j] > u * S where S = sum(w)
    (taken as the last cumulative value); if none (rounding), the last index with w[j] > 0.
    margin = distance from u*S to the nearer edge of bin j, in the units of w.
    """
    w = np.asarray(w, dtype=np.float64)
    c = np.cumsum(w)
    S = c[-1]
    t = u * S
    idx = np.flatnonzero(c > t)
    if idx.size:
        j = int(idx[0])
    else:
        j = int(np.flatnonzero(w > 0)[-1])
    lo = c[j - 1] if j > 0 else 0.0
    margin = min(abs(c[j] - t), abs(t - lo))
    return j, float(margin)


def draft_rows(n_low, hi_first, n_high):
    """Vocabulary ids of the draft rows: [0, n_low) then [hi_first, hi_first + n_high)."""
    return np.concatenate([np.arange(n_low), hi_first + np.arange(n_high)]).astype(np.int64)


def draft_token(y, T, u=None, rows=None):
    """The draft head's token from its logits row ``y`` (float64 [Vd]; row r is vocabulary id
    rows[r], or r without ``rows``).

    T == 0: argmax (lowest index on ties) -- lucebox-hub PR #15, *What*: the draft head "picks
    its token on the GPU". T > 0: inverse-CDF draw of softmax(y/T) with ``u`` =
    U(pos, DRAFT) (the reading that makes the ratio rule exact: drafts distributed as q).
    Returns (token, margin) with margin as in ``inverse_cdf`` (or the top-2 gap at T == 0).
    """
    st = lmhead.row_stats(y, T)
    if st["nonfinite"]:
        return -1, 0.0
    if T == 0:
        j, m = st["argmax"], st["gap"]
    else:
        j, m = inverse_cdf(lmhead.probs(y, T), u)
    return (int(rows[j]) if rows is not None else j), m


def accept_request(z, y, drafts, k, T, eos_id, uniform, pos_base, k_max=7, rows=None):
    """Acceptance for one request and one cycle.

    z:       float64 [>= k+1, V] verify logits; row r predicts position pos_base + r.
    y:       float64 [>= k, Vd] draft logits (row i-1 belongs to draft i) or None (one-hot q);
             column r is vocabulary id rows[r] (r without ``rows``), q is 0 elsewhere.
    drafts:  ints, drafts[i-1] = d_i.
    uniform: callable (pos, purpose) -> u in [0, 1) (the request's seeded Philox stream).
    Returns dict(status, n_accept, tokens, n_emit, eos_hit, sample_kind, sample_row, margins,
    ratio_terms) with sample_kind 0 none, 1 residual, 2 bonus draw; ratio_terms lists, per
    ratio test in order, the two sides (u * q(d_i), p(d_i)) that were compared.
    """
    res = dict(status=STATUS_OK, n_accept=0, tokens=[], n_emit=0, eos_hit=False,
               sample_kind=0, sample_row=-1, margins=[], ratio_terms=[])

    def fail(code):
        res.update(status=code, n_accept=0, tokens=[], n_emit=0, eos_hit=False,
                   sample_kind=0, sample_row=-1)
        return res

    if k < 0 or k > k_max:
        return fail(STATUS_BAD_K)
    z = np.asarray(z, dtype=np.float64)
    V = z.shape[1]
    d = [int(x) for x in drafts[:k]]
    if any(x < 0 or x >= V for x in d):
        return fail(STATUS_BAD_TOKEN)
    zst = [lmhead.row_stats(z[r], T) for r in range(k + 1)]
    if any(s["nonfinite"] for s in zst):
        return fail(STATUS_NONFINITE)
    if T > 0 and y is not None:
        y = np.asarray(y, dtype=np.float64)
        if any(lmhead.row_stats(y[i], T)["nonfinite"] for i in range(k)):
            return fail(STATUS_NONFINITE)

    tokens = res["tokens"]
    margins = res["margins"]

    def emit(tok):
        tokens.append(int(tok))
        if eos_id >= 0 and tok == eos_id:
            res["eos_hit"] = True
            return True
        return False

    if T == 0:
        for i in range(1, k + 1):
            t = zst[i - 1]["argmax"]
            margins.append(("gap", zst[i - 1]["gap"]))
            if d[i - 1] == t:
                res["n_accept"] += 1
                if emit(t):
                    break
            else:
                emit(t)
                break
        else:
            margins.append(("gap", zst[k]["gap"]))
            emit(zst[k]["argmax"])
    else:
        for i in range(1, k + 1):
            x = d[i - 1]
            p = lmhead.probs(z[i - 1], T)
            if y is None:
                q = np.zeros(V)
                q[x] = 1.0
            else:
                qd = lmhead.probs(y[i - 1], T)
                q = np.zeros(V)
                if rows is None:
                    q[: qd.shape[0]] = qd
                else:
                    q[np.asarray(rows)] = qd
            px, qx = float(p[x]), float(q[x])
            u = uniform(pos_base + i - 1, PURPOSE_ACCEPT)
            margins.append(("ratio", abs(u * qx - px)))
            res["ratio_terms"].append((u * qx, px))
            if px > 0.0 and u * qx <= px:
                res["n_accept"] += 1
                if emit(x):
                    break
            else:
                r = np.maximum(0.0, p - q)
                if not np.sum(r) > 0.0:
                    r = p
                u2 = uniform(pos_base + i - 1, PURPOSE_RESIDUAL)
                j, m = inverse_cdf(r, u2)
                margins.append(("cdf", m))
                res.update(sample_kind=1, sample_row=i - 1)
                emit(j)
                break
        else:
            p = lmhead.probs(z[k], T)
            u3 = uniform(pos_base + k, PURPOSE_BONUS)
            j, m = inverse_cdf(p, u3)
            margins.append(("cdf", m))
            res.update(sample_kind=2, sample_row=k)
            emit(j)
    res["n_emit"] = len(tokens)
    return res


def accept_request_exact(z, drafts, k, T, eos_id, uniform, pos_base, k_max=7):
    """Exact-match acceptance at temperature for one request and one cycle (lucebox-hub PR #15
    "MTP speculative decoding", *Exactness* and *Notes*: a draft is kept only if it is the
    token the trunk itself samples, so the emitted text is the same as decoding without drafts
    for the same seed).

    The trunk's own token at position pos is the inverse-CDF draw of p = softmax(z/T) with
    U(pos, BONUS) -- the draw decoding without drafts makes there. For i = 1..k:
    t_i = that draw from row i-1 at pos_base+i-1; if d_i == t_i, emit it (stop if EOS) and go
    on; otherwise emit t_i and stop. All k kept: emit the draw from row k at pos_base+k.
    T == 0: the draws are argmaxes and the result equals ``accept_request``.
    Same inputs, validation and result dict as ``accept_request`` (no draft logits needed);
    sample_kind 3 marks these draws, sample_row is the row of the last one.
    """
    if not T > 0:
        return accept_request(z, None, drafts, k, T, eos_id, uniform, pos_base, k_max)
    res = dict(status=STATUS_OK, n_accept=0, tokens=[], n_emit=0, eos_hit=False,
               sample_kind=0, sample_row=-1, margins=[])
    if k < 0 or k > k_max:
        res["status"] = STATUS_BAD_K
        return res
    z = np.asarray(z, dtype=np.float64)
    V = z.shape[1]
    d = [int(x) for x in drafts[:k]]
    if any(x < 0 or x >= V for x in d):
        res["status"] = STATUS_BAD_TOKEN
        return res
    if any(lmhead.row_stats(z[r], T)["nonfinite"] for r in range(k + 1)):
        res["status"] = STATUS_NONFINITE
        return res
    tokens, margins = res["tokens"], res["margins"]

    def trunk_token(r):
        j, m = inverse_cdf(lmhead.probs(z[r], T), uniform(pos_base + r, PURPOSE_BONUS))
        margins.append(("cdf", m))
        res.update(sample_kind=3, sample_row=r)
        return j

    def emit(tok):
        tokens.append(int(tok))
        if eos_id >= 0 and tok == eos_id:
            res["eos_hit"] = True
            return True
        return False

    for i in range(1, k + 1):
        t = trunk_token(i - 1)
        if d[i - 1] == t:
            res["n_accept"] += 1
            if emit(t):
                break
        else:
            emit(t)
            break
    else:
        emit(trunk_token(k))
    res["n_emit"] = len(tokens)
    return res


def draft_chain_tokens(y_rows, T, uniform, pos_base, rows=None):
    """Draft tokens for one request from precomputed draft logits rows (row i-1 -> draft i).

    Each draft is an independent call of ``draft_token`` with U(pos_base+i-1, DRAFT). Returns
    (tokens, margins).
    """
    toks, margins = [], []
    for i in range(1, len(y_rows) + 1):
        u = uniform(pos_base + i - 1, PURPOSE_DRAFT) if T > 0 else None
        t, m = draft_token(y_rows[i - 1], T, u, rows)
        toks.append(t)
        margins.append(("gap" if T == 0 else "cdf", m))
    return toks, margins


def filtered_probs(z, T, top_k, top_p):
    """p' for one logits row z (float64 [V]) at temperature T > 0 (see the module docstring).

    Returns (p' float64 [V], kept token ids in descending probability, margins) with margins
    ('gap', logit gap between the last kept and the first dropped token of the top-k cut;
    +inf when nothing is dropped) and ('cdf', |mass of the top-p prefix before its last token
    - top_p|, the distance of the top-p cut from flipping, in probability units).
    """
    z = np.asarray(z, dtype=np.float64)
    V = z.shape[0]
    order = np.lexsort((np.arange(V), -z))      # descending logit, ties to the lower id
    kk = min(int(top_k), V)
    top = order[:kk]
    gap = float(z[order[kk - 1]] - z[order[kk]]) if kk < V else float("inf")
    w = np.exp((z[top] - z[top[0]]) / T)
    pk = w / w.sum()
    before = np.concatenate(([0.0], np.cumsum(pk)[:-1]))  # mass ahead of each kept token
    n = int(np.sum(before < top_p))              # keep while the mass ahead is below top_p
    kept = top[:n]
    out = np.zeros(V)
    out[kept] = w[:n] / w[:n].sum()
    cut = min(abs(before[n - 1] - top_p), abs(before[n] - top_p) if n < kk else float("inf"))
    return out, kept, [("gap", gap), ("cdf", float(cut))]


def accept_request_filtered(z, drafts, k, T, top_k, top_p, eos_id, uniform, pos_base, k_max=7):
    """Acceptance against the top-k / top-p filtered target (module docstring) for one request
    and one cycle, with argmax drafts and q one-hot at each draft. T <= 0 is greedy acceptance
    (the filters keep the argmax). Same inputs, validation and result dict as
    ``accept_request``; margins also record each filter's cut."""
    if not T > 0:
        return accept_request(z, None, drafts, k, T, eos_id, uniform, pos_base, k_max)
    res = dict(status=STATUS_OK, n_accept=0, tokens=[], n_emit=0, eos_hit=False,
               sample_kind=0, sample_row=-1, margins=[])
    if k < 0 or k > k_max:
        res["status"] = STATUS_BAD_K
        return res
    z = np.asarray(z, dtype=np.float64)
    V = z.shape[1]
    d = [int(x) for x in drafts[:k]]
    if any(x < 0 or x >= V for x in d):
        res["status"] = STATUS_BAD_TOKEN
        return res
    if any(lmhead.row_stats(z[r], T)["nonfinite"] for r in range(k + 1)):
        res["status"] = STATUS_NONFINITE
        return res
    tokens, margins = res["tokens"], res["margins"]

    def emit(tok):
        tokens.append(int(tok))
        if eos_id >= 0 and tok == eos_id:
            res["eos_hit"] = True
            return True
        return False

    for i in range(1, k + 1):
        x = d[i - 1]
        p, _, m = filtered_probs(z[i - 1], T, top_k, top_p)
        margins.extend(m)
        u = uniform(pos_base + i - 1, PURPOSE_ACCEPT)
        margins.append(("ratio", abs(u - float(p[x]))))
        if p[x] > 0.0 and u <= p[x]:
            res["n_accept"] += 1
            if emit(x):
                break
        else:
            r = p.copy()
            r[x] = 0.0
            if not np.sum(r) > 0.0:
                r = p
            j, mc = inverse_cdf(r, uniform(pos_base + i - 1, PURPOSE_RESIDUAL))
            margins.append(("cdf", mc))
            res.update(sample_kind=1, sample_row=i - 1)
            emit(j)
            break
    else:
        p, _, m = filtered_probs(z[k], T, top_k, top_p)
        margins.extend(m)
        j, mc = inverse_cdf(p, uniform(pos_base + k, PURPOSE_BONUS))
        margins.append(("cdf", mc))
        res.update(sample_kind=2, sample_row=k)
        emit(j)
    res["n_emit"] = len(tokens)
    return res
