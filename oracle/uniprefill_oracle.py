"""Plain fp64 CPU oracle of UniPrefill's per-layer drop step.

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import or run
this module.  The library's CUDA path never calls it and shares no code with
it (the two meet only in the seeded input generator package ``synth``).

Source: "UniPrefill: Universal Long-Context Prefill Acceleration via
Block-wise Dynamic Sparsification" (arXiv 2605.06221), cited below as
[UP §x, Eq. y].  Every function is the plain definition written out, slow
and unblocked; numpy's matmul, sort and cumsum are the only library steps.

Readings where the paper is silent or ambiguous (each is marked where used):

R1  scale: logits are q.k / sqrt(d_k) as in Eq. 2 (the S of Eq. 13 omits it).
R2  heads: Eq. 4 has no head index; the per-token score is the MEAN over the
    H_q query heads of Eq. 3, so that sum_g b_g = 1/G per request.
R3  GQA: query head h reads KV head floor(h / (H_q / H_kv)) (contiguous groups).
R4  the last block B_g may be short; Eq. 4 still divides by G, as written.
R5  every block is ranked (Eq. 5); the sink tokens i < A and the window
    tokens i >= N - n are added afterwards, at token granularity.
R6  ties in Eq. 5's sort: the packed key of Eq. 14 puts the block index in
    the low word, so among equal scores the HIGHER index ranks first.
R7  Eq. 14's phi is applied literally (comparison x >= 0); on the reachable
    domain (non-negative scores) it equals a sign-bit test.
R8  k* = min k with cum_k >= p * total, total = the sum of all block scores.
R9  n_eff = min(n, N): a request shorter than n uses all its tokens as the
    window; Eq. 3's 1/n becomes 1/n_eff.
R10 causal mask inside the window: the query at local position j sees the
    keys i <= j ("inline causal masking", UP §3.5).
R11 Eq. 17: a drop at layer l_k changes the KV length seen by layers l' > l_k
    (strictly); with no earlier drop the length is kv_len (= orig_len + delta).

Pins (tests/test_oracle_pins.py): sum_g b_g = 1/G; closed form at Q = 0;
equivalence with an explicit GQA head expansion; reduction to a textbook
softmax when n = N; brute-force subset enumeration for Eq. 5; Eq. 6's bound
on the dropped mass; hand-worked fixtures under tests/golden/ for Eq. 5/14
ties and thresholds and for Eqs. 16-17; Eq. 8 identities.  No function here
is "parity unpinned".
"""
from __future__ import annotations

import math

import numpy as np


# ----------------------------------------------------------------------------------------------
# helpers that a mutation test may swap out


def kv_head_of(h, group):
    """Query head h reads KV head floor(h / group) (reading R3)."""
    return h // group


def causal_visible(query_pos, key_pos):
    """Key i is visible to the query at local position j iff i <= j (reading R10)."""
    return key_pos[None, :] <= query_pos[:, None]


def softmax_rows(z):
    """Row softmax over the complete key axis (Eq. 2); -inf entries get weight 0."""
    m = z.max(axis=1, keepdims=True)
    e = np.exp(z - m)
    return e / e.sum(axis=1, keepdims=True)


# ----------------------------------------------------------------------------------------------
# score: Eqs. 2-4


def token_scores(Q, K, cu_seqlens, n):
    """Per-token importance s_i of Eq. 3, averaged over query heads (R2).

    [UP §3.2, Eqs. 2-3] s_i = (1/n) sum_{j in window} A_{j,i}, A = softmax_i(q_j K^T / sqrt(d_k))
    over the full sequence (causal inside the window, R10).  Q: [T, H_q, d_k],
    K: [T, H_kv, d_k], any float dtype (widened to fp64).  Returns fp64 [T].
    """
    Q = np.asarray(Q)
    K = np.asarray(K)
    T, Hq, dk = Q.shape
    Hkv = K.shape[1]
    group = Hq // Hkv
    cu = [int(c) for c in cu_seqlens]
    s = np.zeros(T, dtype=np.float64)
    for r in range(len(cu) - 1):
        a, b = cu[r], cu[r + 1]
        N = b - a
        if N <= 0:
            continue
        ne = min(n, N)                                       # R9
        qpos = np.arange(N - ne, N)
        vis = causal_visible(qpos, np.arange(N))
        acc = np.zeros(N, dtype=np.float64)
        for h in range(Hq):
            kh = kv_head_of(h, group)
            q = Q[b - ne:b, h, :].astype(np.float64)
            k = K[a:b, kh, :].astype(np.float64)
            z = (q @ k.T) / math.sqrt(dk)                       # R1
            z = np.where(vis, z, -np.inf)
            acc += softmax_rows(z).sum(axis=0)               # sum over the window rows j
        s[a:b] = acc / (ne * Hq)                             # Eq. 3's 1/n and the head mean (R2)
    return s


def cu_blocks_of(cu_seqlens, G):
    cu = [int(c) for c in cu_seqlens]
    out = [0]
    for r in range(len(cu) - 1):
        out.append(out[-1] + -(-(cu[r + 1] - cu[r]) // G))
    return np.asarray(out, dtype=np.int64)


def block_scores_from_tokens(s, cu_seqlens, G):
    """[UP §3.2, Eq. 4] b_g = (1/G) sum_{i in B_g} s_i, B_g = {gG, ..., min((g+1)G, N) - 1} (R4)."""
    cu = [int(c) for c in cu_seqlens]
    cb = cu_blocks_of(cu, G)
    out = np.zeros(int(cb[-1]), dtype=np.float64)
    for r in range(len(cu) - 1):
        a, b = cu[r], cu[r + 1]
        for g in range(int(cb[r + 1] - cb[r])):
            lo = a + g * G
            hi = min(b, lo + G)
            out[cb[r] + g] = s[lo:hi].sum() / G
    return out


def block_scores(Q, K, cu_seqlens, G, n):
    """Eqs. 2-4 end to end: fp64 block scores [sum_r ceil(N_r / G)]."""
    return block_scores_from_tokens(token_scores(Q, K, cu_seqlens, n), cu_seqlens, G)


# ----------------------------------------------------------------------------------------------
# select: Eqs. 5 and 14 plus the forced tokens of UP §3.3


def phi(x):
    """[UP §3.5, Eq. 14] monotone IEEE-754 map of an fp32 score to uint32 (applied literally, R7)."""
    x = np.asarray(x, dtype=np.float32)
    bits = x.view(np.uint32)
    return np.where(x >= 0, bits ^ np.uint32(0x80000000), bits ^ np.uint32(0xFFFFFFFF)).astype(np.uint32)


def pack_key(scores_f32, g):
    """[UP §3.5, Eq. 14] packed = (phi(b_g) << 32) | g, as an unsigned 64-bit word."""
    return (phi(scores_f32).astype(np.uint64) << np.uint64(32)) | np.asarray(g, dtype=np.uint64)


def rank_order(bbar):
    """Eq. 5's permutation pi: block scores descending, ties by higher index first (R6)."""
    bbar = np.asarray(bbar, dtype=np.float64)
    g = np.arange(len(bbar))
    return np.lexsort((-g, -bbar))


def topp_kstar(bbar, p):
    """[UP §3.3, Eq. 5] k* = min k with sum_{j<=k} b_pi(j) / sum_g b_g >= p (R8). Returns (order, k*)."""
    order = rank_order(bbar)
    if len(order) == 0:
        return order, 0
    cum = np.cumsum(np.asarray(bbar, dtype=np.float64)[order])
    thr = p * cum[-1]
    kstar = int(np.argmax(cum >= thr)) + 1
    return order, kstar


def select_request(bbar, N, G, n, A, p):
    """One request's keep decision: ranked blocks (Eq. 5) united with sinks and window (UP §3.3, R5)."""
    nb = -(-N // G)
    assert len(bbar) == nb
    assert np.all(np.isfinite(bbar)) and np.all(np.asarray(bbar) >= 0)
    order, kstar = topp_kstar(bbar, p)
    ranked = np.zeros(nb, dtype=bool)
    ranked[order[:kstar]] = True
    i = np.arange(N)
    token_keep = ranked[i // G] | (i < A) | (i >= N - n)
    block_keep = np.array([token_keep[g * G:min(N, (g + 1) * G)].any() for g in range(nb)], dtype=bool)
    return dict(order=order, kstar=kstar, ranked=ranked, token_keep=token_keep, block_keep=block_keep)


def select(block_sc, cu_seqlens, G, n, A, p):
    """All requests: token_keep u8 [T], block_keep u8 [sum nb], kstar [R], ranked blocks."""
    cu = [int(c) for c in cu_seqlens]
    cb = cu_blocks_of(cu, G)
    tk = np.zeros(cu[-1], dtype=np.uint8)
    bk = np.zeros(int(cb[-1]), dtype=np.uint8)
    ranked = np.zeros(int(cb[-1]), dtype=np.uint8)
    ks = np.zeros(len(cu) - 1, dtype=np.int64)
    for r in range(len(cu) - 1):
        N = cu[r + 1] - cu[r]
        if N == 0:
            continue
        d = select_request(np.asarray(block_sc[cb[r]:cb[r + 1]], dtype=np.float64), N, G, n, A, p)
        tk[cu[r]:cu[r + 1]] = d["token_keep"]
        bk[cb[r]:cb[r + 1]] = d["block_keep"]
        ranked[cb[r]:cb[r + 1]] = d["ranked"]
        ks[r] = d["kstar"]
    return dict(token_keep=tk, block_keep=bk, ranked=ranked, kstar=ks, cu_blocks=cb)


# ----------------------------------------------------------------------------------------------
# compact + metadata (UP §3.5 "vLLM scheduler integration"), Eq. 8, Eq. 16, Eq. 17


def compact(token_keep, cu_seqlens, hidden=None, positions=None, slots=None):
    """Stable gather of the kept tokens and the patched query_start_loc / seq_lens / num_actual_tokens."""
    keep = np.asarray(token_keep).astype(bool)
    cu = [int(c) for c in cu_seqlens]
    kept_index = np.flatnonzero(keep).astype(np.int64)       # ascending = stable
    seq_lens = np.array([int(keep[cu[r]:cu[r + 1]].sum()) for r in range(len(cu) - 1)], dtype=np.int64)
    new_cu = np.concatenate([[0], np.cumsum(seq_lens)]).astype(np.int64)
    out = dict(kept_index=kept_index, new_cu_seqlens=new_cu, seq_lens=seq_lens, num_actual_tokens=int(new_cu[-1]))
    if hidden is not None:
        out["hidden"] = np.asarray(hidden)[kept_index]
    if positions is not None:
        out["positions"] = np.asarray(positions)[kept_index]
    if slots is not None:
        out["slots"] = np.asarray(slots)[kept_index]
    return out


def carry_forward(H_block_in, H_kept_out, kept_index):
    """[UP §3.4, Eq. 8] H^(b+1,0)_i = H^(b,M_b+1)_i for kept i, H^(b,0)_i for dropped i."""
    H = np.array(H_block_in, copy=True)
    H[np.asarray(kept_index, dtype=np.int64)] = np.asarray(H_kept_out)
    return H


def slot_mapping(positions, cu_seqlens, block_table, B):
    """[UP §3.5, Eq. 16] slot_i = block_table[r_i, floor(p_i / B)] * B + (p_i mod B)."""
    cu = [int(c) for c in cu_seqlens]
    out = np.zeros(cu[-1], dtype=np.int64)
    for r in range(len(cu) - 1):
        for t in range(cu[r], cu[r + 1]):
            pi = int(positions[t])
            out[t] = int(block_table[r][pi // B]) * B + pi % B
    return out


def seqused(kept_len, drop_layer, layer, orig_len, kv_len):
    """[UP §3.5, Eq. 17] seqused_r = s_r^(l-) + (kv_len_r - orig_len_r), l- = last drop layer < layer (R11)."""
    R = len(orig_len)
    prev = [l for l in range(len(drop_layer)) if drop_layer[l] and l < layer]
    out = np.zeros(R, dtype=np.int64)
    for r in range(R):
        delta = int(kv_len[r]) - int(orig_len[r])
        base = int(kept_len[max(prev)][r]) if prev else int(orig_len[r])
        out[r] = base + delta
    return out


# ----------------------------------------------------------------------------------------------
# one whole drop step


def drop_step(Q, K, cu_seqlens, G, n, A, p, hidden=None, positions=None, slots=None):
    s = token_scores(Q, K, cu_seqlens, n)
    bs = block_scores_from_tokens(s, cu_seqlens, G)
    sel = select(bs, cu_seqlens, G, n, A, p)
    cmp_ = compact(sel["token_keep"], cu_seqlens, hidden, positions, slots)
    return dict(token_scores=s, block_scores=bs, **sel, compact=cmp_)
