"""Float64 CPU oracle for context-parallel chunk attention (dense and top-k sparse).

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  This module is the independent checker
that the CUDA path is compared against.  Only the test suite, the smoke check
of ``__graft_entry__`` and the ``cpu_baseline`` / ``--impl reference`` legs of
``bench.py`` may import or run it.  It shares no code, table or helper with the
CUDA library and imports nothing from it; inputs reach it as numpy arrays
(already rounded to the precision handed to the GPU, then widened to float64).

Every function cites the passage it follows, by page title and paragraph:

[CP]   "Context parallel attention: exchange keys and merge softmax globally"
       ¶1 each query sees every valid key of its sequence; causal means the
          permitted global prefix.
       ¶2 masks use global token positions; packed variable-length sequences
          must not attend across examples; GQA shares KV heads.
       ¶3 a chunk is summarised by its max score m, scaled exponential
          denominator l and scaled value numerator z; two summaries combine by
          rescaling both to the larger max and adding; divide only at the end.
       ¶4 an all-masked chunk needs a neutral summary (no -inf minus -inf);
          a query with no permitted key needs an explicit convention.
       ¶5 a zigzag layout changes ownership, not the attention relation; keep
          both the logical order and the physical chunk assignment.
[DSA-CP]  "[Feature-request] Context Parallel support for DSAttention",
          "Strategy: allgather CP mode": local Q against gathered global KV,
          causal diagonal shifted by cp_rank * local_seq (``causal_offset``),
          top-k indices in global sequence coordinates; step 7: a chunk run at
          an offset equals the matching slice of a full single-rank run.
[DSA-THD] "[1/2] Enable DSA CP, THD with absorbed MLA - #3674", sequence
          diagram (index mask + varlen bounds, then QK scores -> top-k ->
          sparse gather) and "Background" (absorbed MLA: attention runs on the
          latent; the key row is [latent | rope], the value is the latent).
[MoBA-CP] "Question on Implementing Context Parallelism with MoBA Efficient
          Attention": gating scores Q x K^T choose the top-k KV blocks.

Readings taken where the pages are silent:
  * neutral summary = (m=-inf, l=0, z=0); no permitted key -> O = 0, LSE = -inf;
  * LSE is a natural log of the scaled scores: LSE = m + ln(l);
  * GQA: query head h reads KV head h // (Hq // Hkv);
  * physical chunk c of a chunk map holds logical chunk map[c];
  * MoBA gate: mean of the block's keys, unscaled dot with the query, top-k
    among blocks that end at or before the start of the query's own block,
    ties to the lower block index, own block always added, output ascending
    and padded with -1.

Parity pins: every public function here is checked in tests/test_oracle_*.py
against brute force on tiny inputs (plain softmax without max subtraction and
math.fsum), against torch.nn.functional.scaled_dot_product_attention /
torch.logsumexp in float64, against a hand-derived closed-form worked example
(tests/golden/), and against the invariants the pages state.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

NEG_INF = -np.inf


# ---------------------------------------------------------------------------
# Positions and the permitted relation  ([CP] ¶1, ¶2, ¶5; [DSA-CP] allgather)
# ---------------------------------------------------------------------------

def logical_positions(n, offset=0, chunk_map=None, chunk_len=0):
    """Logical global position of each of ``n`` rows held in physical order.

    [CP] ¶5: a row's logical position is kept apart from where it is stored.
    With a chunk map, physical chunk c (rows c*chunk_len ...) holds logical
    chunk ``chunk_map[c]``.  [DSA-CP]: a local chunk is placed at
    ``causal_offset``; the offset is added to every position.
    """
    t = np.arange(n, dtype=np.int64)
    if chunk_map is not None:
        cmap = np.asarray(chunk_map, dtype=np.int64)
        t = cmap[t // chunk_len] * chunk_len + t % chunk_len
    return t + np.int64(offset)


def sequence_index(pos, cu_seqlens):
    """Index s of the packed sequence with cu[s] <= pos < cu[s+1], else -1.

    [CP] ¶2 packed variable-length boundaries.  ``cu_seqlens=None`` means one
    sequence that holds every position.
    """
    pos = np.asarray(pos, dtype=np.int64)
    if cu_seqlens is None:
        return np.zeros(pos.shape, dtype=np.int64)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    s = np.searchsorted(cu, pos, side="right") - 1
    s = np.where((pos < cu[0]) | (pos >= cu[-1]), -1, s)
    return s.astype(np.int64)


@dataclass
class Layout:
    """Logical positions and sequence ids of the query rows and KV rows."""

    qpos: np.ndarray
    kpos: np.ndarray
    qseq: np.ndarray
    kseq: np.ndarray
    causal: bool
    cu_seqlens: object = None

    def allowed(self, rows=None):
        """Boolean [len(rows), Tk]: may query row i attend to KV row j.

        allowed(i, j) = same packed sequence ([CP] ¶2) and, when causal,
        kpos_j <= qpos_i ([CP] ¶1, global positions per ¶2).
        """
        qp = self.qpos if rows is None else self.qpos[rows]
        qs = self.qseq if rows is None else self.qseq[rows]
        a = (qs[:, None] == self.kseq[None, :]) & (qs[:, None] >= 0)
        if self.causal:
            a &= self.kpos[None, :] <= qp[:, None]
        return a

    def allowed_logical(self, row, key_logical):
        """Permitted relation for one query row and keys given by logical position."""
        kl = np.asarray(key_logical, dtype=np.int64)
        ks = sequence_index(kl, self.cu_seqlens)
        a = (ks == self.qseq[row]) & (self.qseq[row] >= 0)
        if self.causal:
            a &= kl <= self.qpos[row]
        return a


def make_layout(Tq, Tk, causal=True, causal_offset=0, cu_seqlens=None,
                q_chunk_map=None, kv_chunk_map=None, chunk_len=0):
    """Build the layout of a local query chunk against the gathered KV.

    Query rows sit at ``causal_offset`` (+ chunk map), KV rows at their
    gathered logical positions ([DSA-CP] allgather mode, [CP] ¶5).
    """
    qpos = logical_positions(Tq, causal_offset, q_chunk_map, chunk_len)
    kpos = logical_positions(Tk, 0, kv_chunk_map, chunk_len)
    return Layout(qpos, kpos, sequence_index(qpos, cu_seqlens),
                  sequence_index(kpos, cu_seqlens), bool(causal), cu_seqlens)


def _kv_head(h, Hq, Hkv):
    """GQA sharing ([CP] ¶2): contiguous groups of Hq // Hkv query heads."""
    return h // (Hq // Hkv)


# ---------------------------------------------------------------------------
# Global softmax attention (the definition every chunked form must reach)
# ---------------------------------------------------------------------------

def dense_attention(q, k, v, scale, layout, rows=None, row_block=256):
    """Global-softmax attention of query rows over every permitted key.

    For each (i, h): P = {j : allowed(i, j)}; s_j = scale * <q_ih, k_jg>;
    m = max_P s; l = sum_P exp(s_j - m); O = sum_P exp(s_j - m) v_jg / l;
    LSE = m + ln l.  If P is empty: O = 0, LSE = -inf ([CP] ¶4 convention).
    Row blocking only bounds memory; each row is computed independently.

    q: [Tq, Hq, Dqk], k: [Tk, Hkv, Dqk], v: [Tk, Hkv, Dv] float64.
    Returns O [R, Hq, Dv], LSE [R, Hq] for R = len(rows) (all rows if None).
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    Tq, Hq, _ = q.shape
    Hkv = k.shape[1]
    rows = np.arange(Tq) if rows is None else np.asarray(rows, dtype=np.int64)
    O = np.zeros((len(rows), Hq, v.shape[2]))
    LSE = np.full((len(rows), Hq), NEG_INF)
    for r0 in range(0, len(rows), row_block):
        rr = rows[r0:r0 + row_block]
        A = layout.allowed(rr)
        nonempty = A.any(axis=1)
        for h in range(Hq):
            g = _kv_head(h, Hq, Hkv)
            S = scale * (q[rr, h, :] @ k[:, g, :].T)
            S = np.where(A, S, NEG_INF)
            m = S.max(axis=1) if S.shape[1] else np.full(len(rr), NEG_INF)
            shift = np.where(nonempty, m, 0.0)
            E = np.where(A, np.exp(S - shift[:, None]), 0.0)
            ell = E.sum(axis=1)
            Z = E @ v[:, g, :]
            safe = np.where(nonempty, ell, 1.0)
            O[r0:r0 + len(rr), h, :] = np.where(nonempty[:, None], Z / safe[:, None], 0.0)
            LSE[r0:r0 + len(rr), h] = np.where(nonempty, shift + np.log(safe), NEG_INF)
    return O, LSE


def dense_attention_backward(q, k, v, scale, layout, d_out):
    """Gradients of ``dense_attention`` with respect to q, k and v.

    [CP] ¶2: backward must return the contributions of a chunk's queries to
    the owners of K and V, so dk and dv cover every gathered KV row (what
    this chunk's queries add; summing over chunks is outside this function).
    [CP] ¶4: the backward rebuilds the probabilities from the forward's
    saved statistics; here they are the exact global-softmax weights.  With
    P[i, j] = softmax over the permitted keys of row i (0 elsewhere) and
    g = dO:
        dv[j]  = sum_i P[i, j] g[i]                      (per KV head, summed
        dP[i, j] = <g[i], v[j]>                           over its query heads)
        dS[i, j] = P[i, j] (dP[i, j] - sum_j' P[i, j'] dP[i, j'])
        dq[i]  = scale sum_j dS[i, j] k[j]
        dk[j]  = scale sum_i dS[i, j] q[i]
    A row with no permitted key contributes nothing.

    q: [Tq, Hq, Dqk], k: [Tk, Hkv, Dqk], v: [Tk, Hkv, Dv], d_out: [Tq, Hq, Dv].
    Returns dq [Tq, Hq, Dqk], dk [Tk, Hkv, Dqk], dv [Tk, Hkv, Dv] float64.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    g = np.asarray(d_out, np.float64)
    Tq, Hq, _ = q.shape
    Hkv = k.shape[1]
    A = layout.allowed()
    nonempty = A.any(axis=1)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for h in range(Hq):
        gh = _kv_head(h, Hq, Hkv)
        S = np.where(A, scale * (q[:, h, :] @ k[:, gh, :].T), NEG_INF)
        m = np.where(nonempty, S.max(axis=1) if S.shape[1] else 0.0, 0.0)
        E = np.where(A, np.exp(S - m[:, None]), 0.0)
        ell = np.where(nonempty, E.sum(axis=1), 1.0)
        P = E / ell[:, None]
        dv[:, gh, :] += P.T @ g[:, h, :]
        dP = g[:, h, :] @ v[:, gh, :].T
        dS = P * (dP - (P * dP).sum(axis=1, keepdims=True))
        dq[:, h, :] = scale * (dS @ k[:, gh, :])
        dk[:, gh, :] += scale * (dS.T @ q[:, h, :])
    return dq, dk, dv


# ---------------------------------------------------------------------------
# Chunk summaries and their merge  ([CP] ¶3, ¶4)
# ---------------------------------------------------------------------------

def neutral_summary(R, Dv):
    """The summary of a chunk with no permitted key: (m=-inf, l=0, z=0) ([CP] ¶4)."""
    return np.full(R, NEG_INF), np.zeros(R), np.zeros((R, Dv))


def chunk_summary(s, permitted, v):
    """(m, l, z) of one KV chunk for R query rows ([CP] ¶3).

    s: [R, n] scaled scores, permitted: [R, n] bool, v: [n, Dv].
    m = max over permitted s; l = sum exp(s - m); z = sum exp(s - m) v.
    A row with no permitted key gets the neutral summary ([CP] ¶4).
    """
    R = s.shape[0]
    Dv = v.shape[1]
    if s.shape[1] == 0:
        return neutral_summary(R, Dv)
    nonempty = permitted.any(axis=1)
    sm = np.where(permitted, s, NEG_INF)
    m = np.where(nonempty, sm.max(axis=1), NEG_INF)
    shift = np.where(nonempty, m, 0.0)
    e = np.where(permitted, np.exp(sm - shift[:, None]), 0.0)
    return m, e.sum(axis=1), e @ v


def merge_summaries(a, b):
    """Combine two chunk summaries by rescaling both to the larger max ([CP] ¶3).

    m = max(m_a, m_b); alpha_x = exp(m_x - m), taken as 0 when m_x = -inf so
    that -inf - (-inf) is never evaluated ([CP] ¶4); l and z add after the
    rescale.  Two neutral summaries merge to the neutral summary.
    """
    ma, la, za = a
    mb, lb, zb = b
    m = np.maximum(ma, mb)
    live = m > NEG_INF
    ref = np.where(live, m, 0.0)
    alpha_a = np.where(ma > NEG_INF, np.exp(np.where(ma > NEG_INF, ma, 0.0) - ref), 0.0)
    alpha_b = np.where(mb > NEG_INF, np.exp(np.where(mb > NEG_INF, mb, 0.0) - ref), 0.0)
    ell = alpha_a * la + alpha_b * lb
    z = alpha_a[:, None] * za + alpha_b[:, None] * zb
    return (np.where(live, m, NEG_INF), np.where(live, ell, 0.0),
            np.where(live[:, None], z, 0.0))


def finalise(summary):
    """Divide only at the end ([CP] ¶3): O = z / l, LSE = m + ln l.

    l = 0 (no permitted key anywhere) gives O = 0, LSE = -inf ([CP] ¶4).
    """
    m, ell, z = summary
    live = ell > 0
    safe = np.where(live, ell, 1.0)
    O = np.where(live[:, None], z / safe[:, None], 0.0)
    LSE = np.where(live, m + np.log(safe), NEG_INF)
    return O, LSE


def lse_merge(part_o, part_lse):
    """Merge finalised per-chunk results (O_c, LSE_c) into the global result.

    (O_c, LSE_c) carries the summary (m_c, l_c, z_c) up to a common factor:
    l_c = exp(LSE_c - m_c) and z_c = l_c O_c, so the [CP] ¶3 merge becomes
    L = max_c LSE_c, w_c = exp(LSE_c - L) (0 when LSE_c = -inf),
    LSE = L + ln sum w_c, O = sum w_c O_c / sum w_c.  All parts -inf gives
    (0, -inf) ([CP] ¶4).  part_o: [n, ..., Dv], part_lse: [n, ...].
    """
    po = np.asarray(part_o, np.float64)
    pl = np.asarray(part_lse, np.float64)
    L = pl.max(axis=0)
    live = L > NEG_INF
    ref = np.where(live, L, 0.0)
    w = np.where(pl > NEG_INF, np.exp(np.where(pl > NEG_INF, pl, 0.0) - ref), 0.0)
    W = w.sum(axis=0)
    safe = np.where(live, W, 1.0)
    O = np.where(live[..., None], (w[..., None] * po).sum(axis=0) / safe[..., None], 0.0)
    LSE = np.where(live, ref + np.log(safe), NEG_INF)
    return O, LSE


def summarised_attention(q, k, v, scale, layout, kv_chunk_len, rows=None):
    """Attention as per-KV-chunk summaries folded in chunk order ([CP] ¶3-4).

    KV chunk c holds the physical rows [c*kv_chunk_len, (c+1)*kv_chunk_len)
    (what one peer contributes).  Each chunk's (m, l, z) is computed over its
    permitted keys (neutral if none), the summaries are merged in ascending
    chunk order and the total is finalised once.  Also returns each chunk's
    finalised (O_c, LSE_c).

    Returns O [R, Hq, Dv], LSE [R, Hq], part_o [n, R, Hq, Dv], part_lse [n, R, Hq].
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    Tq, Hq, _ = q.shape
    Tk, Hkv, Dv = v.shape
    rows = np.arange(Tq) if rows is None else np.asarray(rows, dtype=np.int64)
    R = len(rows)
    n_chunks = -(-Tk // kv_chunk_len)
    A = layout.allowed(rows)
    O = np.zeros((R, Hq, Dv))
    LSE = np.full((R, Hq), NEG_INF)
    part_o = np.zeros((n_chunks, R, Hq, Dv))
    part_lse = np.full((n_chunks, R, Hq), NEG_INF)
    for h in range(Hq):
        g = _kv_head(h, Hq, Hkv)
        total = neutral_summary(R, Dv)
        for c in range(n_chunks):
            j0, j1 = c * kv_chunk_len, min((c + 1) * kv_chunk_len, Tk)
            s = scale * (q[rows, h, :] @ k[j0:j1, g, :].T)
            summ = chunk_summary(s, A[:, j0:j1], v[j0:j1, g, :])
            part_o[c, :, h, :], part_lse[c, :, h] = finalise(summ)
            total = merge_summaries(total, summ)
        O[:, h, :], LSE[:, h] = finalise(total)
    return O, LSE, part_o, part_lse


# ---------------------------------------------------------------------------
# Top-k sparse attention  ([DSA-CP] allgather mode, [DSA-THD] diagram, [MoBA-CP])
# ---------------------------------------------------------------------------

def _physical_row_of_logical(layout):
    """Inverse of the KV chunk map: logical position -> physical row (-1 if absent)."""
    Tk = len(layout.kpos)
    inv = np.full(Tk, -1, dtype=np.int64)
    ok = (layout.kpos >= 0) & (layout.kpos < Tk)
    inv[layout.kpos[ok]] = np.arange(Tk)[ok]
    return inv


def sparse_key_list(indices_row, Tk, block_size):
    """Logical key positions named by one row of indices, one entry per occurrence.

    block_size == 1: each index is a logical key position ([DSA-CP]: top-k
    indices in global coordinates).  block_size > 1: each index b names the
    logical keys [b*B, min((b+1)*B, Tk)) ([MoBA-CP] block selection).
    -1 marks an unused slot.  An index outside the key range (or below -1) is
    skipped and counted as bad.  Returns (keys int64 array, n_bad).
    """
    keys = []
    bad = 0
    for t in np.asarray(indices_row, dtype=np.int64).tolist():
        if t == -1:
            continue
        if t < -1 or t * block_size >= Tk:
            bad += 1
            continue
        if block_size == 1:
            keys.append(t)
        else:
            keys.extend(range(t * block_size, min((t + 1) * block_size, Tk)))
    return np.asarray(keys, dtype=np.int64), bad


def sparse_attention(q, k, v, scale, layout, indices, block_size=1, rows=None):
    """Attention of each query over the keys its indices select ([DSA-THD]).

    P(i, h) = {keys named by indices[i, h or 0, :]} intersected with the
    permitted relation (the index mask and varlen bounds are re-applied,
    [DSA-THD] diagram); softmax over P exactly as ``dense_attention``, each
    occurrence counted once.  Empty P -> O = 0, LSE = -inf.

    indices: [Tq, index_heads, topk], index_heads in {1, Hq}.
    Returns O [R, Hq, Dv], LSE [R, Hq], n_bad (bad index count over the rows).
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    Tq, Hq, _ = q.shape
    Tk, Hkv, Dv = v.shape
    indices = np.asarray(indices)
    index_heads = indices.shape[1]
    rows = np.arange(Tq) if rows is None else np.asarray(rows, dtype=np.int64)
    inv = _physical_row_of_logical(layout)
    O = np.zeros((len(rows), Hq, Dv))
    LSE = np.full((len(rows), Hq), NEG_INF)
    n_bad = 0
    for r, i in enumerate(rows.tolist()):
        for h in range(Hq):
            if index_heads == 1 and h > 0:
                keys, bad = keys0, 0
            else:
                keys, bad = sparse_key_list(indices[i, 0 if index_heads == 1 else h], Tk, block_size)
                keys0 = keys
            n_bad += bad
            if len(keys) == 0:
                continue
            keys = keys[layout.allowed_logical(i, keys)]
            phys = inv[keys]
            keys = keys[phys >= 0]
            phys = phys[phys >= 0]
            if len(keys) == 0:
                continue
            g = _kv_head(h, Hq, Hkv)
            s = scale * (k[phys, g, :] @ q[i, h, :])
            m = s.max()
            e = np.exp(s - m)
            ell = e.sum()
            O[r, h, :] = (e @ v[phys, g, :]) / ell
            LSE[r, h] = m + np.log(ell)
    return O, LSE, n_bad


# ---------------------------------------------------------------------------
# MoBA block gate  ([MoBA-CP]: gating scores Q x K^T choose top-k KV blocks)
# ---------------------------------------------------------------------------

def block_means(k, block_size, kpos=None):
    """Mean of the keys of every complete block, per KV head: [n_blocks, Hkv, D].

    Blocks are runs of LOGICAL key positions [b*B, (b+1)*B) ([MoBA-CP] blocks
    of the sequence; [CP] ¶5 a chunk map changes where a key is stored, not
    its position).  ``kpos`` gives the logical position of each stored KV row
    (None: stored in logical order); the rows are put back in logical order
    before pooling.
    """
    k = np.asarray(k, np.float64)
    if kpos is not None:
        order = np.argsort(np.asarray(kpos, dtype=np.int64), kind="stable")
        k = k[order]
    n_blocks = k.shape[0] // block_size
    kb = k[: n_blocks * block_size].reshape(n_blocks, block_size, k.shape[1], k.shape[2])
    return kb.sum(axis=1) / block_size


def moba_block_gate(q, k, qpos, block_size, topk, rows=None, kpos=None):
    """Block selection of every (query, head) pair.

    gate(i, h, b) = <q_ih, mean of block b's keys of KV head g(h)> (unscaled).
    Candidates are the complete blocks b with (b+1)*B <= own(i)*B, where
    own(i) = qpos_i // B is the query's own block.  The ``topk`` candidates
    with the largest gate are chosen, equal gates going to the lower block;
    fewer candidates -> all of them.  The own block is always added.  The
    row is returned in ascending block order, padded with -1 to topk + 1.
    Blocks are blocks of logical positions; ``kpos`` (logical position of
    each stored KV row, None = logical order) is passed to ``block_means``.

    Returns sel int32 [R, Hq, topk + 1].
    """
    q = np.asarray(q, np.float64)
    Tq, Hq, _ = q.shape
    Hkv = k.shape[1]
    mu = block_means(k, block_size, kpos)
    n_blocks = mu.shape[0]
    rows = np.arange(Tq) if rows is None else np.asarray(rows, dtype=np.int64)
    own = np.asarray(qpos, dtype=np.int64)[rows] // block_size
    n_cand = np.clip(own, 0, n_blocks)
    sel = np.full((len(rows), Hq, topk + 1), -1, dtype=np.int32)
    b = np.arange(n_blocks)
    for h in range(Hq):
        g = _kv_head(h, Hq, Hkv)
        G = q[rows, h, :] @ mu[:, g, :].T
        key = np.where(b[None, :] < n_cand[:, None], -G, np.inf)
        order = np.argsort(key, axis=1, kind="stable")
        for r in range(len(rows)):
            chosen = order[r, : min(topk, n_cand[r])].tolist()
            chosen.append(int(own[r]))
            chosen = sorted(chosen)
            sel[r, h, : len(chosen)] = chosen
    return sel


def moba_attention(q, k, v, scale, layout, sel, block_size, rows=None):
    """Attention over the selected blocks, causal within the own block."""
    O, LSE, _ = sparse_attention(q, k, v, scale, layout, sel, block_size, rows)
    return O, LSE


# ---------------------------------------------------------------------------
# DSA indexer: which keys a query attends to  ([DSA-THD] sequence diagram)
# ---------------------------------------------------------------------------

def dsa_indexer_topk(qI, kI, w, layout, topk, rows=None):
    """Key selection of the DSA indexer, per query row.

    [DSA-THD] sequence diagram: the index mask and the varlen bounds first,
    then the indexer's QK scores, then the top-k keys that the sparse
    attention gathers ([DSA-CP]: indices in global coordinates).  The score
    of key j for query i over the indexer heads h is

        score(i, j) = sum_h w_h * max(0, <qI[i, h], kI[j]>),

    taken over the keys the layout permits (same sequence, kpos_j <= qpos_i
    when causal), in float64 from the exact inputs.  Keys are named by their
    LOGICAL position ([DSA-CP]: global coordinates; [CP] ¶5: a chunk map
    changes where a key is stored, not its position): kI row j is stored at
    physical row j and sits at logical position layout.kpos[j].  The
    ``topk`` keys with the largest score are chosen, equal scores going to
    the lower logical position; a row with fewer permitted keys takes all of
    them.  Each row is returned as ascending logical positions padded with -1.

    qI: [Tq, H, D], kI: [Tk, D], w: [H].  Returns int32 [R, 1, topk].
    """
    qI = np.asarray(qI, np.float64)
    kI = np.asarray(kI, np.float64)
    w = np.asarray(w, np.float64)
    Tq, H, _ = qI.shape
    Tk = kI.shape[0]
    rows = np.arange(Tq) if rows is None else np.asarray(rows, dtype=np.int64)
    out = np.full((len(rows), 1, topk), -1, dtype=np.int32)
    j = np.arange(Tk)
    for r, i in enumerate(rows):
        A = layout.allowed(np.array([i]))[0]
        dots = qI[i] @ kI.T                               # [H, Tk]
        score = (w[:, None] * np.maximum(dots, 0.0)).sum(axis=0)
        phys = j[A]
        logical = layout.kpos[A]
        # descending score, ties to the lower logical position
        order = np.lexsort((logical, -score[phys]))
        chosen = np.sort(logical[order[:topk]])
        out[r, 0, :len(chosen)] = chosen
    return out
