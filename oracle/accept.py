"""The accept step of one verify round, written out as the pages state it.

Greedy (T == 0).  mlx-dspark wiki page, "Architecture": the draft is compared
against the target's own logits and the longest accepted prefix is committed;
hysenlabs review, "The Problem": verification stops at the first mismatch.
[reading] The target's own token at the first mismatch (or the bonus token
after a fully accepted draft) is committed too: that is the only reading under
which every round makes progress and the output equals one-token-at-a-time
greedy decoding, as the PyPI page ("How it works") and the releases page
(v0.1.0) state.

Sampled (T > 0).  mlx-dspark releases page, v0.0.2 "Highlights": sample the
draft, accept it with probability min(1, p/q), resample from the residual on
rejection; the output is then an exact sample of the target at temperature T
(wiki page, "Architecture": the Leviathan/Chen rule).  Readings taken:

* p_i = softmax(z_i / T) of the target's fp32 logits, in fp64.  q_i is given
  as probabilities already at the draft's temperature and is never rescaled.
* Draft i (token d) is accepted iff u[i] < p_i[d] / q_i[d] (strict; u in
  [0, 1) makes the min(1, .) implicit).  q_i[d] == 0 gives an infinite ratio
  and the draft is accepted.
* Exactly m + 1 uniforms per round: u[0..m-1] are the accept tests, u[m]
  drives the single final draw.
* Final draw: the smallest k whose cumulative weight C_k (index order) exceeds
  u[m] * Z, Z the total weight.  If rounding leaves no such k, the last k with
  positive weight.  The weights are the residual max(0, p - q) of the first
  rejected row, or p_m when every draft was accepted; a residual with Z == 0
  falls back to p of that row.
"""

import numpy as np

from .qmm import row_stats, target_probs


def greedy_accept(logits, draft):
    """(out_len, tokens) for T == 0 from fp32 logits [m + 1, V] and draft [m]."""
    z = np.asarray(logits, dtype=np.float32)
    draft = [int(d) for d in draft]
    m = len(draft)
    if z.shape[0] != m + 1:
        raise ValueError("logits must have m + 1 rows")
    _, argmax, _ = row_stats(z, 0.0)
    tokens = []
    for i in range(m):
        if draft[i] != int(argmax[i]):
            tokens.append(int(argmax[i]))          # target token at the mismatch
            return len(tokens), tokens
        tokens.append(draft[i])                    # accepted draft
    tokens.append(int(argmax[m]))                  # bonus token
    return len(tokens), tokens


def inverse_cdf(weights, u):
    """Smallest k with cumsum(weights)[k] > u * sum(weights) (fp64, index order).

    Returns (k, threshold, cumsum).  Falls back to the last k with positive
    weight when rounding leaves the threshold at or above the final sum.
    """
    w = np.asarray(weights, dtype=np.float64)
    c = np.cumsum(w)
    z = c[-1]
    theta = float(u) * z
    above = np.nonzero(c > theta)[0]
    if above.size:
        k = int(above[0])
    else:
        k = int(np.nonzero(w > 0)[0][-1])
    return k, theta, c


def sampled_accept_detail(logits, q, draft, temperature, u):
    """Sampled accept with the intermediate quantities the parity tests need.

    Returns a dict with ``out_len``, ``tokens``, ``ratios`` (p/q for every
    examined draft), ``reject`` (index of the first rejected draft or -1),
    ``weights_kind`` ('residual', 'p_fallback' or 'bonus'), ``theta``, ``Z`` and
    ``cdf`` (the cumulative weights of the final draw).
    """
    if not temperature > 0:
        raise ValueError("sampled accept needs T > 0")
    z = np.asarray(logits, dtype=np.float32)
    qf = np.asarray(q, dtype=np.float32)
    draft = [int(d) for d in draft]
    u = np.asarray(u, dtype=np.float32)
    m = len(draft)
    if z.shape[0] != m + 1 or qf.shape[0] != m or u.shape[0] != m + 1:
        raise ValueError("shapes: logits [m+1, V], q [m, V], u [m+1]")
    tokens, ratios = [], []
    for i in range(m):
        p_i = target_probs(z[i], temperature)
        q_i = qf[i].astype(np.float64)
        d = draft[i]
        r = np.inf if q_i[d] == 0.0 else p_i[d] / q_i[d]
        ratios.append(r)
        if float(u[i]) < r:
            tokens.append(d)
            continue
        residual = np.maximum(0.0, p_i - q_i)
        kind = "residual"
        if residual.sum() == 0.0:
            residual, kind = p_i, "p_fallback"
        k, theta, c = inverse_cdf(residual, u[m])
        tokens.append(k)
        return dict(out_len=len(tokens), tokens=tokens, ratios=ratios, reject=i,
                    weights_kind=kind, theta=theta, Z=float(c[-1]), cdf=c)
    p_m = target_probs(z[m], temperature)
    k, theta, c = inverse_cdf(p_m, u[m])
    tokens.append(k)
    return dict(out_len=len(tokens), tokens=tokens, ratios=ratios, reject=-1,
                weights_kind="bonus", theta=theta, Z=float(c[-1]), cdf=c)


def sampled_accept(logits, q, draft, temperature, u):
    d = sampled_accept_detail(logits, q, draft, temperature, u)
    return d["out_len"], d["tokens"]


def spec_accept(logits, q, draft, temperature, u):
    """The accept step for either mode: (out_len, tokens)."""
    if temperature > 0:
        return sampled_accept(logits, q, draft, temperature, u)
    return greedy_accept(logits, draft)


def spec_accept_batched(logits, q, drafts, row_offsets, temperature, us):
    """B independent accept steps over stacked rows (continuous batching).

    PyPI page, "Concurrent throughput": B requests share one forward; each
    row set accepts and rolls back on its own.  Request b owns logits rows
    [row_offsets[b], row_offsets[b + 1]) (m_b + 1 of them), the matching m_b
    draft-probability rows of ``q`` (stacked in the same order, offset
    row_offsets[b] - b), its drafts ``drafts[b]`` and uniforms ``us[b]``.
    """
    out = []
    for b in range(len(row_offsets) - 1):
        r0, r1 = int(row_offsets[b]), int(row_offsets[b + 1])
        m_b = r1 - r0 - 1
        q_b = None if q is None else np.asarray(q)[r0 - b: r0 - b + m_b]
        out.append(spec_accept(np.asarray(logits)[r0:r1], q_b, drafts[b], temperature,
                               None if us is None else us[b]))
    return out


# ------------------------------------------------------------- truncation
# mlx-dspark releases page, v0.1.0 "Highlights": lossless top-p / top-k -
# nucleus / top-k truncation applied to both the draft and the target, so
# sampling stays an exact sample from the truncated target.  Readings taken:
#
# * The order is by the row's own values, largest first, ties to the lower
#   index: by the fp32 logit for the target (probabilities are monotone in it),
#   by the fp32 probability for a draft row.
# * top_k > 0 keeps the first top_k tokens in that order (0 = no limit).
# * top_p < 1 then keeps, among those, the shortest prefix whose probability
#   (renormalised over the top_k survivors) reaches top_p (1 = no limit).
# * The kept weights are renormalised; everything else gets probability 0.
# * The draft's truncation is the draft sampler's business (the library offers
#   the same rule for probability rows); the accept step truncates the target
#   and uses q as given, the distribution the drafts were drawn from.

def truncation_mask(keys, weights, top_k, top_p):
    """Boolean kept-mask of one row: order by keys (desc, ties to lower index),
    keep the first top_k, then the shortest prefix of those whose weight share
    reaches top_p."""
    keys = np.asarray(keys)
    w = np.asarray(weights, dtype=np.float64)
    V = keys.shape[0]
    order = np.lexsort((np.arange(V), -keys.astype(np.float64)))   # keys desc, then index asc
    n = V if top_k <= 0 else min(top_k, V)
    if top_p < 1.0:
        c = np.cumsum(w[order[:n]])
        total = c[-1]
        reach = np.nonzero(c >= top_p * total)[0]
        n = int(reach[0]) + 1 if reach.size else n
    mask = np.zeros(V, dtype=bool)
    mask[order[:n]] = True
    return mask


def truncated_target_probs(logits_row, temperature, top_k, top_p):
    """p' of one target row: softmax(z / T) restricted to the kept set, renormalised (fp64)."""
    z = np.asarray(logits_row, dtype=np.float32)
    e = np.exp((z.astype(np.float64) - float(z.max())) / float(temperature))
    keep = truncation_mask(z, e, top_k, top_p)
    e = np.where(keep, e, 0.0)
    return e / e.sum()


def truncate_probs(q_row, top_k, top_p):
    """The same rule on a probability row (fp32 in, fp64 out), for the draft side."""
    q = np.asarray(q_row, dtype=np.float32)
    w = q.astype(np.float64)
    keep = truncation_mask(q, w, top_k, top_p)
    w = np.where(keep, w, 0.0)
    return w / w.sum()


def sampled_accept_truncated_detail(logits, q, draft, temperature, u, top_k, top_p):
    """sampled_accept_detail with the target truncated (top_k / top_p) in every row."""
    if not temperature > 0:
        raise ValueError("sampled accept needs T > 0")
    z = np.asarray(logits, dtype=np.float32)
    qf = np.asarray(q, dtype=np.float32)
    draft = [int(d) for d in draft]
    u = np.asarray(u, dtype=np.float32)
    m = len(draft)
    tokens, ratios = [], []
    for i in range(m):
        p_i = truncated_target_probs(z[i], temperature, top_k, top_p)
        q_i = qf[i].astype(np.float64)
        d = draft[i]
        # a token the truncated target never emits is rejected whatever q says
        r = 0.0 if p_i[d] == 0.0 else (np.inf if q_i[d] == 0.0 else p_i[d] / q_i[d])
        ratios.append(r)
        if float(u[i]) < r:
            tokens.append(d)
            continue
        residual = np.maximum(0.0, p_i - q_i)
        kind = "residual"
        if residual.sum() == 0.0:
            residual, kind = p_i, "p_fallback"
        k, theta, c = inverse_cdf(residual, u[m])
        tokens.append(k)
        return dict(out_len=len(tokens), tokens=tokens, ratios=ratios, reject=i,
                    weights_kind=kind, theta=theta, Z=float(c[-1]), cdf=c)
    p_m = truncated_target_probs(z[m], temperature, top_k, top_p)
    k, theta, c = inverse_cdf(p_m, u[m])
    tokens.append(k)
    return dict(out_len=len(tokens), tokens=tokens, ratios=ratios, reject=-1,
                weights_kind="bonus", theta=theta, Z=float(c[-1]), cdf=c)


# ---------------------------------------------------------------- logprobs
# mlx-dspark releases page, v0.2.0 "Highlights": logprobs / top_logprobs, the
# chosen and the top-k target log-probabilities per token.  [reading] At
# temperature T (T = 1 when the round is greedy): log p_v = (z_v - max) / T -
# log sum_k exp((z_k - max) / T); the top list is ordered like truncation
# (logit desc, ties to the lower index).

def logprobs(logits_row, temperature, chosen, top_n):
    """(log p[chosen], top ids, top log-probabilities) of one row, fp64."""
    z = np.asarray(logits_row, dtype=np.float32)
    T = float(temperature) if temperature > 0 else 1.0
    d = (z.astype(np.float64) - float(z.max())) / T
    lse = np.log(np.exp(d).sum())
    lp = d - lse
    V = z.shape[0]
    order = np.lexsort((np.arange(V), -z.astype(np.float64)))[:top_n]
    return float(lp[int(chosen)]), order.astype(np.int64), lp[order]
