"""Float64 CPU oracle: attention KL divergence by materialise-then-reduce.

TEST INFRASTRUCTURE ONLY -- see the package docstring.  Plain numpy, float64,
one (batch, head) slice and one block of query rows at a time.  Nothing is
fused or reordered beyond the definitions below, so each line can be checked
by eye against the pages.

Sources (the pages this restates; no code was printed on them):
  [AGI] StreamKL article on agidaily.cc, sections "Why attention distillation
        matters" (problem definition), "Online formula" (the coupled online
        KL), "Forward" and "Backward" (recompute from LSE, the two gradient
        modes, the stable log-ratio).
  [ARX] "StreamKL: Fast and Memory-Efficient KL Divergence for Boosting
        Attention Distillation", arXiv 2606.20005 listing: abstract (row-wise
        KL between two attention distributions, tile-by-tile recompute).

Notation (the pages' own): S1 = s1*Q1 K1^T, S2 = s2*Q2 K2^T, P1 = softmax(S1),
P2 = softmax(S2) row-wise over the visible keys, KL_i = sum_j P1_ij
log(P1_ij / P2_ij), LSE_k = log sum_j exp(S_k,ij).

Readings taken where the pages are silent:
  * one softmax scale ``s`` multiplies both logit matrices by default; a
    second scale (``scale2``) may be given for the S2 side, e.g. a student
    with another head dimension (every function takes ``scale2=None``,
    meaning s2 = s1 = ``scale``);
  * the causal mask is bottom-right aligned: key j is visible to query i iff
    j <= i + (NK - NQ); causal with NQ > NK is rejected (every row keeps at
    least one key);
  * LSE is the natural-log log-sum-exp over the visible keys;
  * only KL is differentiated; the upstream gradient is dKL (one per row);
  * grouped key heads (GQA; MQA with one key head) are not on the pages and
    are taken in their usual sense: with H query heads and HK key heads (HK
    dividing H), query head h reads key head h // (H / HK) of its side, and a
    shared key head's gradient is the sum over the query heads that read it.

Arrays: q1 [NQ, d1], k1 [NK, d1], q2 [NQ, d2], k2 [NK, d2] per head; the
batched wrappers take [B, H, N, d].  Callers pass float64 copies of the exact
bf16 values the GPU sees.
"""

import functools

import numpy as np


def _quiet(fn):
    """Masked entries are -inf by construction and np.where discards the
    NaN/inf values computed there; silence the warnings they raise."""
    @functools.wraps(fn)
    def wrapped(*a, **k):
        with np.errstate(invalid="ignore", divide="ignore", over="ignore", under="ignore"):
            return fn(*a, **k)
    return wrapped


MODE_P2 = 0  # gradient into the P2 (student) side: standard distillation
MODE_P1 = 1  # gradient into the P1 side


def visible_mask(nq, nk, causal, rows=None):
    """Boolean [len(rows), NK] mask of visible (query, key) pairs.

    Causal reading: bottom-right alignment, j <= i + (NK - NQ), which is
    j <= i when NQ == NK (the pages state no alignment; [AGI] "Forward").
    """
    if rows is None:
        rows = np.arange(nq)
    rows = np.asarray(rows)
    if not causal:
        return np.ones((rows.shape[0], nk), dtype=bool)
    if nq > nk:
        raise ValueError("causal attention with NQ > NK leaves rows without keys")
    j = np.arange(nk)[None, :]
    return j <= rows[:, None] + (nk - nq)


def _logsumexp_rows(s, vis):
    """Row-wise log sum_j exp(s_ij) over visible j, with the max subtracted."""
    masked = np.where(vis, s, -np.inf)
    m = masked.max(axis=1)
    return m + np.log(np.sum(np.where(vis, np.exp(masked - m[:, None]), 0.0), axis=1))


@_quiet
def _head_rows(q1, k1, q2, k2, s1, s2, causal, rows):
    """Materialise S, log P and P for the given query rows of one head.

    [AGI] "Why attention distillation matters": the loss compares the two
    N_Q x N_K attention matrices P1 and P2 row by row; this is the
    materialise-then-reduce computation the method replaces.
    """
    nq, nk = q1.shape[0], k1.shape[0]
    vis = visible_mask(nq, nk, causal, rows)
    s1, s2 = s1 * (q1[rows] @ k1.T), s2 * (q2[rows] @ k2.T)
    lse1 = _logsumexp_rows(s1, vis)
    lse2 = _logsumexp_rows(s2, vis)
    # log-domain probabilities: P itself may underflow, log P never does
    logp1 = np.where(vis, s1 - lse1[:, None], -np.inf)
    logp2 = np.where(vis, s2 - lse2[:, None], -np.inf)
    p1 = np.where(vis, np.exp(logp1), 0.0)
    p2 = np.where(vis, np.exp(logp2), 0.0)
    # KL_i = sum_j P1 (log P1 - log P2), taken over visible keys only
    kl = np.sum(np.where(vis, p1 * (logp1 - logp2), 0.0), axis=1)
    return dict(vis=vis, s1=s1, s2=s2, lse1=lse1, lse2=lse2,
                logp1=logp1, logp2=logp2, p1=p1, p2=p2, kl=kl)


def _scales(scale, scale2):
    """(s1, s2): the S1-side and S2-side softmax scales."""
    return scale, (scale if scale2 is None else scale2)


def _row_blocks(n, block):
    for r0 in range(0, n, block):
        yield np.arange(r0, min(n, r0 + block))


def forward_head(q1, k1, q2, k2, scale, causal, row_block=256, scale2=None):
    """KL, LSE1, LSE2 for every query row of one head (float64 [NQ] each)."""
    s1, s2 = _scales(scale, scale2)
    nq = q1.shape[0]
    kl = np.empty(nq)
    lse1 = np.empty(nq)
    lse2 = np.empty(nq)
    for rows in _row_blocks(nq, row_block):
        r = _head_rows(q1, k1, q2, k2, s1, s2, causal, rows)
        kl[rows], lse1[rows], lse2[rows] = r["kl"], r["lse1"], r["lse2"]
    return kl, lse1, lse2


def _group(h_, k):
    """Query heads per key head for a [B, HK, N, d] key tensor."""
    hk = k.shape[1]
    if hk < 1 or h_ % hk:
        raise ValueError("the key head count must divide the query head count")
    return h_ // hk


def forward(q1, k1, q2, k2, scale, causal, row_block=256, scale2=None):
    """Batched forward over [B, H, N, d] inputs -> (kl, lse1, lse2) [B, H, NQ].
    k1, k2 may have fewer heads (grouped key heads, see the module notes)."""
    b_, h_, nq = q1.shape[:3]
    g1, g2 = _group(h_, k1), _group(h_, k2)
    out = [np.empty((b_, h_, nq)) for _ in range(3)]
    for b in range(b_):
        for h in range(h_):
            res = forward_head(q1[b, h], k1[b, h // g1], q2[b, h], k2[b, h // g2], scale, causal, row_block,
                               scale2)
            for o, v in zip(out, res):
                o[b, h] = v
    return tuple(out)


def forward_rows(q1, k1, q2, k2, scale, causal, rows, scale2=None):
    """Forward for selected query rows of one head (each row is independent)."""
    r = _head_rows(q1, k1, q2, k2, *_scales(scale, scale2), causal, np.asarray(rows))
    return r["kl"], r["lse1"], r["lse2"]


@_quiet
def forward_online(q1, k1, q2, k2, scale, causal, key_tile=64, row_block=256, scale2=None):
    """The pages' online coupled-KL recurrence, run in float64 ([AGI] "Online
    formula" and "Forward").

    Per query row, over key tiles: running maxima m1, m2; running sums
    l1 = sum e^(S1 - m1), l2 = sum e^(S2 - m2); coupled accumulator
    acc = sum e^(S1 - m1) (S1 - S2).  When m1 moves, l1 and acc are both
    multiplied by e^(m1_old - m1_new) (a B_Q-vector rescale); l2 follows m2.
    At the end LSE = m + log l and KL = acc / l1 + LSE2 - LSE1.
    Only the logit tiles of one key tile exist at a time.
    """
    sc1, sc2 = _scales(scale, scale2)
    nq, nk = q1.shape[0], k1.shape[0]
    kl = np.empty(nq)
    lse1 = np.empty(nq)
    lse2 = np.empty(nq)
    for rows in _row_blocks(nq, row_block):
        n = rows.shape[0]
        m1 = np.full(n, -np.inf)
        m2 = np.full(n, -np.inf)
        l1 = np.zeros(n)
        l2 = np.zeros(n)
        acc = np.zeros(n)
        for k0 in range(0, nk, key_tile):
            keys = np.arange(k0, min(nk, k0 + key_tile))
            vis = visible_mask(nq, nk, causal, rows)[:, keys]
            s1 = sc1 * (q1[rows] @ k1[keys].T)
            s2 = sc2 * (q2[rows] @ k2[keys].T)
            t1 = np.where(vis, s1, -np.inf).max(axis=1)
            t2 = np.where(vis, s2, -np.inf).max(axis=1)
            m1_new = np.maximum(m1, t1)
            m2_new = np.maximum(m2, t2)
            live1 = np.isfinite(m1_new)  # rows that have seen a visible key
            live2 = np.isfinite(m2_new)
            # correction factors; a row with no visible key yet keeps zeros
            a1 = np.where(np.isfinite(m1), np.exp(m1 - np.where(live1, m1_new, 0.0)), 0.0)
            a2 = np.where(np.isfinite(m2), np.exp(m2 - np.where(live2, m2_new, 0.0)), 0.0)
            e1 = np.where(vis, np.exp(s1 - np.where(live1, m1_new, 0.0)[:, None]), 0.0)
            e2 = np.where(vis, np.exp(s2 - np.where(live2, m2_new, 0.0)[:, None]), 0.0)
            l1 = a1 * l1 + e1.sum(axis=1)
            acc = a1 * acc + np.sum(np.where(vis, e1 * (s1 - s2), 0.0), axis=1)
            l2 = a2 * l2 + e2.sum(axis=1)
            m1, m2 = m1_new, m2_new
        lse1[rows] = m1 + np.log(l1)
        lse2[rows] = m2 + np.log(l2)
        kl[rows] = acc / l1 + lse2[rows] - lse1[rows]
    return kl, lse1, lse2


@_quiet
def forward_two_pass(q1, k1, q2, k2, scale, causal, key_tile=64, row_block=256, scale2=None):
    """The two-pass streaming alternative ([AGI] "Why FlashAttention does not
    carry over"): pass 1 streams keys for LSE1 and LSE2, pass 2 streams them
    again for sum_j P1 (S1 - S2); then KL = that sum - LSE1 + LSE2 (because
    log P1 - log P2 = S1 - S2 - LSE1 + LSE2 and P1 sums to one).
    """
    sc1, sc2 = _scales(scale, scale2)
    nq, nk = q1.shape[0], k1.shape[0]
    kl = np.empty(nq)
    lse1 = np.empty(nq)
    lse2 = np.empty(nq)
    tiles = [np.arange(k0, min(nk, k0 + key_tile)) for k0 in range(0, nk, key_tile)]
    for rows in _row_blocks(nq, row_block):
        vis_all = visible_mask(nq, nk, causal, rows)
        # pass 1: exact per-tile log-sum-exp, combined with np.logaddexp
        a = np.full(rows.shape[0], -np.inf)
        b = np.full(rows.shape[0], -np.inf)
        for keys in tiles:
            vis = vis_all[:, keys]
            s1 = np.where(vis, sc1 * (q1[rows] @ k1[keys].T), -np.inf)
            s2 = np.where(vis, sc2 * (q2[rows] @ k2[keys].T), -np.inf)
            for dst, s in ((0, s1), (1, s2)):
                t = s.max(axis=1)
                tt = np.where(np.isfinite(t), t, 0.0)
                part = np.where(np.isfinite(t),
                                tt + np.log(np.sum(np.exp(s - tt[:, None]), axis=1)), -np.inf)
                if dst == 0:
                    a = np.logaddexp(a, part)
                else:
                    b = np.logaddexp(b, part)
        # pass 2
        w = np.zeros(rows.shape[0])
        for keys in tiles:
            vis = vis_all[:, keys]
            s1 = sc1 * (q1[rows] @ k1[keys].T)
            s2 = sc2 * (q2[rows] @ k2[keys].T)
            p1 = np.where(vis, np.exp(np.where(vis, s1, 0.0) - a[:, None]), 0.0)
            w += np.sum(np.where(vis, p1 * (s1 - s2), 0.0), axis=1)
        lse1[rows], lse2[rows] = a, b
        kl[rows] = w - a + b
    return kl, lse1, lse2


@_quiet
def _grad_scores(r, dkl_rows, mode):
    """dL/dS on the gradient side for a block of rows.

    [AGI] "Backward": P is rebuilt as exp(S - LSE).  Mode P2 (standard
    distillation, gradient into the second distribution):
        dS2 = dKL_i (P2 - P1)
    Mode P1 (gradient into the first distribution) with the log-ratio taken
    from logits, log P1 - log P2 = (S1 - LSE1) - (S2 - LSE2), so nothing is
    computed as log of an underflowed probability:
        dS1 = dKL_i P1 (log P1 - log P2 - KL_i)
    Masked pairs get zero.
    """
    vis = r["vis"]
    if mode == MODE_P2:
        ds = dkl_rows[:, None] * (r["p2"] - r["p1"])
    elif mode == MODE_P1:
        ratio = np.where(vis, r["logp1"] - r["logp2"], 0.0)
        ds = dkl_rows[:, None] * r["p1"] * (ratio - r["kl"][:, None])
    else:
        raise ValueError("mode must be MODE_P2 or MODE_P1")
    return np.where(vis, ds, 0.0)


def backward_head(q1, k1, q2, k2, scale, causal, dkl, mode, row_block=256, scale2=None):
    """(dQ, dK) of L = sum_i dKL_i KL_i for one head, on the gradient side.

    Mode P2 returns (dQ2 [NQ, d2], dK2 [NK, d2]); mode P1 returns (dQ1, dK1).
    With S = s Q K^T on the gradient side: dQ = s dS K and dK = s dS^T Q.
    """
    s1, s2 = _scales(scale, scale2)
    nq, nk = q1.shape[0], k1.shape[0]
    qg, kg = (q2, k2) if mode == MODE_P2 else (q1, k1)
    sg = s2 if mode == MODE_P2 else s1
    dq = np.zeros((nq, qg.shape[1]))
    dk = np.zeros((nk, kg.shape[1]))
    for rows in _row_blocks(nq, row_block):
        r = _head_rows(q1, k1, q2, k2, s1, s2, causal, rows)
        ds = _grad_scores(r, dkl[rows], mode)
        dq[rows] = sg * (ds @ kg)
        dk += sg * (ds.T @ qg[rows])
    return dq, dk


def backward(q1, k1, q2, k2, scale, causal, dkl, mode, row_block=256, scale2=None):
    """Batched backward over [B, H, N, d] inputs; dkl is [B, H, NQ].  With
    grouped key heads dK has the gradient side's key head count: each query
    head's contribution is added into the key head it reads."""
    b_, h_, nq = q1.shape[:3]
    nk = k1.shape[2]
    g1, g2 = _group(h_, k1), _group(h_, k2)
    kg = k2 if mode == MODE_P2 else k1
    gg = g2 if mode == MODE_P2 else g1
    dg = kg.shape[3]
    dq = np.empty((b_, h_, nq, dg))
    dk = np.zeros((b_, kg.shape[1], nk, dg))
    for b in range(b_):
        for h in range(h_):
            dq[b, h], dk_h = backward_head(q1[b, h], k1[b, h // g1], q2[b, h], k2[b, h // g2],
                                           scale, causal, dkl[b, h], mode, row_block, scale2)
            dk[b, h // gg] += dk_h
    return dq, dk


def backward_dq_rows(q1, k1, q2, k2, scale, causal, dkl, mode, rows, scale2=None):
    """dQ for selected query rows of one head (a row's dS needs only that row)."""
    s1, s2 = _scales(scale, scale2)
    rows = np.asarray(rows)
    r = _head_rows(q1, k1, q2, k2, s1, s2, causal, rows)
    ds = _grad_scores(r, dkl[rows], mode)
    kg, sg = (k2, s2) if mode == MODE_P2 else (k1, s1)
    return sg * (ds @ kg)


def backward_dk_keys(q1, k1, q2, k2, scale, causal, dkl, mode, keys, row_block=256, first_row=0, scale2=None):
    """dK for selected keys of one head: dK_j = s sum_i dS_ij Q_i over all rows.

    ``first_row`` skips rows that see none of ``keys`` under the causal mask
    (their dS entries are exactly zero); it must not exceed min(keys) - (NK - NQ).
    """
    keys = np.asarray(keys)
    nq, nk = q1.shape[0], k1.shape[0]
    if first_row > 0 and (not causal or first_row > keys.min() - (nk - nq)):
        raise ValueError("first_row would skip rows that see the requested keys")
    s1, s2 = _scales(scale, scale2)
    qg, kg = (q2, k2) if mode == MODE_P2 else (q1, k1)
    sg = s2 if mode == MODE_P2 else s1
    dk = np.zeros((keys.shape[0], kg.shape[1]))
    for rows in _row_blocks(nq, row_block):
        rows = rows[rows >= first_row]
        if rows.shape[0] == 0:
            continue
        r = _head_rows(q1, k1, q2, k2, s1, s2, causal, rows)
        ds = _grad_scores(r, dkl[rows], mode)[:, keys]
        dk += sg * (ds.T @ qg[rows])
    return dk


def loss(q1, k1, q2, k2, scale, causal, dkl, scale2=None):
    """Scalar L = sum dKL * KL over all rows, for finite-difference checks."""
    kl, _, _ = forward(q1, k1, q2, k2, scale, causal, scale2=scale2)
    return float(np.sum(dkl * kl))
