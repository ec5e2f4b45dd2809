"""CPU oracle for the self-speculative verification step (test infrastructure).

This module is TEST INFRASTRUCTURE.  Only the test suite, the package smoke
check and the CPU-baseline leg of the benchmark may import or run it; the
product path never does.  It shares no code with the CUDA path.

It is a plain, slow, obviously-correct restatement, in float64 numpy, of
what one verification step computes:

  1. ``mask_build``       visibility of the speculative block's rows
  2. ``verify_attention`` masked softmax attention over
                          (committed prefix || soft prompt || block)
  3. ``vocab_reduce``     per judged row: argmax, log-sum-exp, proposal logit
  4. ``accept``           threshold longest prefix, or greedy tree walk;
     ``accept_soft``      soft matching (ratio test + residual draw)
     ``draft_tree``, ``prune_tree``, ``ss_block_vparent``: the next draft
     ``rotate_stream_values`` (SS Eq. 7), ``future_gather`` (ConFu hand-off)
  5. ``kv_commit``        append the accepted rows' K/V to the cache

Sources (page title, section / equation):

* "Lookahead Attention: Self-Speculative Verification via Parallel Token
  Proposals" (LA): sec. 2.1 diagram, sec. 2.2-2.4, sec. 3.1 mask M_LA,
  sec. 3.2 (lookahead KV discarded), sec. 3.3 (padding to one length).
* "ConFu: Contemplate the Future for Better Speculative Sampling" notes:
  key design 1 (soft prompt seen only by contemplate tokens, one contemplate
  token per draft node, 2T tokens verified in one pass).
* "Speculative Streaming: Fast LLM Inference without Auxiliary Models":
  Eq. 1 (main-stream MHA, softmax(QK^T/sqrt(d))V), Eq. 2 (stream j sees the
  main stream <= t and streams <= j at the same t), Eq. 4 and the text after
  it (tree nodes see their ancestors), the verification step (hard matching,
  beta accepted + 1 correction token).

Readings where the pages are garbled or silent (each is listed with its
reason in the design notes):

* LA prints M_LA with rows = keys and columns = queries; the masks here are
  query-major.  The diagram's top-left block is printed as the identity; the
  formula's M_causal (standard causal) is used.
* A lookahead row sees itself (diagonal) and no other lookahead row.
* The LA proposal of row i is judged by row i's own distribution, with
  p_i >= tau accepted ("exceeds" read as >=; tau = 0.3).
* SS Eq. 4 read together with the sentence after it: a node sees all of its
  ancestors and itself (not only its immediate parent).
* A stream row sees itself (Eq. 2, S_{t(<=j)} includes j).
* A ConFu contemplate token sees the prefix, its node's ancestors, its node,
  itself and the soft prompt; draft nodes never see the soft prompt.
* Tree root = node 0, always accepted; its K/V is committed first.
* Padding rows (vparent = -2) see nothing: O = 0, LSE = -inf.
* Paged cache: requests in ascending order take pages from the free list in
  order, after filling their partly used tail page.  A page stores, per KV
  head, the head dimension in blocks of ``blk`` elements, each block as
  page_size rows: pages[p][h][j // blk][slot][j % blk].
"""

from __future__ import annotations

import math

import numpy as np

VP_ROOT = -1
VP_PAD = -2

MODE_THRESH_CHAIN = 0
MODE_GREEDY_TREE = 1


# --------------------------------------------------------------------------
# 1. mask
# --------------------------------------------------------------------------

def la_prefill_mask(n: int, k: int) -> np.ndarray:
    """Full LA mask M_LA for n original and k lookahead positions.

    LA sec. 3.1, written query-major (row = query, column = key): original
    queries are causal over originals and never see lookahead keys; a
    lookahead query sees every original key and itself only.
    """
    L = n + k
    m = np.zeros((L, L), dtype=bool)
    for i in range(n):
        for j in range(i + 1):
            m[i, j] = True
    for i in range(n, L):
        for j in range(n):
            m[i, j] = True
        m[i, i] = True
    return m


def la_prefill_attention(q, k, v, n, scale=None):
    """Attention of all n + k positions under the full LA mask (LA sec. 3.1).

    q, k, v: [L][d] with L = n + k (n originals, then k lookahead rows);
    returns O [L][d] and LSE [L] (float64): softmax(q K^T * scale + M) V with
    M the additive 0 / -inf form of ``la_prefill_mask(n, L - n)``.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    L, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    mask = np.where(la_prefill_mask(n, L - n), 0.0, -np.inf)
    s = (q @ k.T) * scale + mask
    O = np.empty((L, d))
    LSE = np.empty(L)
    for i in range(L):
        m = s[i].max()
        LSE[i] = m + math.log(np.exp(s[i] - m).sum())
        O[i] = np.exp(s[i] - LSE[i]) @ v
    return O, LSE


def la_prefill_vparent(n: int, k: int) -> np.ndarray:
    """Parent pointers whose closure is M_LA (LA sec. 3.1): original i's
    parent is i - 1 (causal), every lookahead row's parent is the last
    original (it then sees all originals and itself)."""
    vp = np.empty(n + k, dtype=np.int64)
    vp[0] = VP_ROOT
    vp[1:n] = np.arange(n - 1)
    vp[n:] = n - 1 if n > 0 else VP_ROOT
    return vp


def mask_build(vparent: np.ndarray, soft_flags=None):
    """Visibility of the speculative block, per request.

    ``vparent[b][r]``: -1 -> row r sees only the prefix and itself (LA
    lookahead row, tree root); -2 -> padding row; p >= 0 -> row r sees what
    row p sees plus itself (tree ancestor closure, SS Eq. 2/4, ConFu).

    Returns (vis [B][R][R] bool: row r sees block column c,
             valid [B][R] bool, sees_soft [B][R] bool).
    Raises ValueError for a parent that is not an earlier valid row.
    """
    vparent = np.asarray(vparent)
    B, R = vparent.shape
    vis = np.zeros((B, R, R), dtype=bool)
    valid = np.zeros((B, R), dtype=bool)
    for b in range(B):
        for r in range(R):
            p = int(vparent[b, r])
            if p == VP_PAD:
                continue
            if p == VP_ROOT:
                pass
            elif p < 0 or p >= r or not valid[b, p]:
                raise ValueError(f"bad parent {p} for row {r} of request {b}")
            valid[b, r] = True
            # walk the parent chain: r, parent(r), parent(parent(r)), ...
            c = r
            while c >= 0:
                vis[b, r, c] = True
                c = int(vparent[b, c])
    if soft_flags is None:
        sees_soft = np.zeros((B, R), dtype=bool)
    else:
        sees_soft = (np.asarray(soft_flags) != 0) & valid
    return vis, valid, sees_soft


# --------------------------------------------------------------------------
# 2. attention
# --------------------------------------------------------------------------

def verify_attention(q, prefix_k, prefix_v, k_block, v_block, vis, valid,
                     sees_soft, soft_k=None, soft_v=None, scale=None,
                     requests=None, heads=None):
    """Masked attention of the speculative rows, in float64.

    q        [B][R][Hq][d]
    prefix_k list over requests of [Hkv][S_b][d] (committed prefix, logical
             order); prefix_v likewise
    k_block  [B][Hkv][R][d]  the block's own keys (v_block: values)
    soft_k   [Hkv][n_soft][d] or None
    vis, valid, sees_soft  from ``mask_build``

    For query head h the key/value head is h // (Hq / Hkv).  The columns of
    row r are [prefix 0..S_b) || [soft 0..n_soft) || [block 0..R), with the
    explicit additive mask 0 (visible) / -inf (hidden): every valid row sees
    the whole prefix, the soft columns iff sees_soft, block column c iff
    vis[r][c].  Scores s = (q . k) * scale with scale = 1/sqrt(d) (SS Eq. 1);
    LSE = ln sum_j exp(s_j); O = sum_j exp(s_j - LSE) v_j.

    ``requests`` / ``heads`` restrict the work (others left as NaN).
    Returns O [B][R][Hq][d] and LSE [B][Hq][R] (float64); rows that are not
    valid have O = 0 and LSE = -inf.
    """
    q = np.asarray(q, dtype=np.float64)
    B, R, Hq, d = q.shape
    Hkv = k_block.shape[1]
    G = Hq // Hkv
    if vis.shape != (B, R, R) or k_block.shape[:3] != (B, Hkv, R) or Hq % Hkv:
        raise ValueError("inconsistent shapes")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    n_soft = 0 if soft_k is None else soft_k.shape[1]
    O = np.full((B, R, Hq, d), np.nan)
    LSE = np.full((B, Hq, R), np.nan)
    reqs = range(B) if requests is None else requests
    hs = range(Hq) if heads is None else heads
    for b in reqs:
        S = prefix_k[b].shape[1]
        # explicit dense additive mask over the concatenated columns
        mask = np.full((R, S + n_soft + R), -np.inf)
        for r in range(R):
            if not valid[b, r]:
                continue
            mask[r, :S] = 0.0
            if sees_soft[b, r]:
                mask[r, S:S + n_soft] = 0.0
            for c in range(R):
                if vis[b, r, c]:
                    mask[r, S + n_soft + c] = 0.0
        for h in hs:
            kvh = h // G
            parts_k = [np.asarray(prefix_k[b][kvh], dtype=np.float64)]
            parts_v = [np.asarray(prefix_v[b][kvh], dtype=np.float64)]
            if n_soft:
                parts_k.append(np.asarray(soft_k[kvh], dtype=np.float64))
                parts_v.append(np.asarray(soft_v[kvh], dtype=np.float64))
            parts_k.append(np.asarray(k_block[b, kvh], dtype=np.float64))
            parts_v.append(np.asarray(v_block[b, kvh], dtype=np.float64))
            Kc = np.concatenate(parts_k, axis=0)
            Vc = np.concatenate(parts_v, axis=0)
            s = (q[b, :, h, :] @ Kc.T) * scale + mask       # [R][cols]
            for r in range(R):
                if not valid[b, r]:
                    O[b, r, h] = 0.0
                    LSE[b, h, r] = -np.inf
                    continue
                m = s[r].max()
                lse = m + math.log(np.exp(s[r] - m).sum())
                p = np.exp(s[r] - lse)
                O[b, r, h] = p @ Vc
                LSE[b, h, r] = lse
    return O, LSE


def gather_paged(pages, page_table, seq_len, page_size):
    """Logical per-request prefixes [Hkv][S_b][d] from a paged cache.

    pages [n_pages][Hkv][d // blk][page_size][blk]: element j of token t of
    request b, KV head h is pages[page_table[b][t // page_size]][h]
    [j // blk][t % page_size][j % blk].
    """
    out = []
    P, Hkv, nblk, ps, blk = pages.shape
    assert ps == page_size
    d = nblk * blk
    for b in range(len(seq_len)):
        S = int(seq_len[b])
        kk = np.empty((Hkv, S, d), dtype=pages.dtype)
        for t in range(S):
            p = int(page_table[b][t // page_size])
            for j in range(nblk):
                kk[:, t, j * blk:(j + 1) * blk] = pages[p, :, j, t % page_size]
        out.append(kk)
    return out


# --------------------------------------------------------------------------
# 3. vocab reduce
# --------------------------------------------------------------------------

def vocab_reduce(logits, proposal=None):
    """Per row of logits [n][V]: argmax (lowest index on ties), LSE, z[prop].

    LA sec. 2.4 needs the proposal's probability exp(z_prop - LSE); the
    greedy walk of SS ("verification step", hard matching) needs the argmax.
    """
    z = np.asarray(logits, dtype=np.float64)
    n = z.shape[0]
    amax = np.empty(n, dtype=np.int64)
    lse = np.empty(n)
    zprop = np.full(n, np.nan)
    for i in range(n):
        row = z[i]
        m = row.max()
        amax[i] = int(np.nonzero(row == m)[0][0])
        lse[i] = m + math.log(np.exp(row - m).sum())
        if proposal is not None:
            zprop[i] = row[int(proposal[i])]
    return amax, lse, zprop


# --------------------------------------------------------------------------
# 4. acceptance
# --------------------------------------------------------------------------

def accept_threshold_chain(zprop, lse, n_props, tau):
    """LA sec. 2.4: the longest prefix of proposals whose probabilities all
    reach tau.  Row i judges proposal i.  Returns L (number accepted)."""
    L = 0
    while L < n_props and math.exp(zprop[L] - lse[L]) >= tau:
        L += 1
    return L


def accept_greedy_tree(tokens, tree_parent, n_nodes, argmax_of_node):
    """SS verification step (hard matching), also ConFu's tree verify.

    From the root (node 0), repeatedly move to the child of the current node
    whose token equals the target's greedy token at the current node; stop
    when there is none.  Returns (path [root, ...], next_token) where
    next_token is the target's greedy token at the last accepted node (the
    correction token); beta = len(path) - 1 draft tokens are accepted.
    Siblings are expected to carry distinct tokens; otherwise the child with
    the lowest index is taken.
    """
    cur = 0
    path = [0]
    while True:
        want = int(argmax_of_node[cur])
        nxt = None
        for c in range(n_nodes):
            if int(tree_parent[c]) == cur and int(tokens[c]) == want:
                nxt = c
                break
        if nxt is None:
            return path, want
        cur = nxt
        path.append(cur)


def accept(mode, tau, tokens, tree_parent, n_nodes, argmax, lse, zprop,
           row_of=None):
    """Acceptance for every request.

    Chain mode (LA): proposal i of request b is judged by judge row i;
    acc_len = L, path = [0, 1, ..., L-1], next_token = argmax of row L when
    L < n_nodes else -1, last_node = L - 1.
    Tree mode: path as ``accept_greedy_tree``; acc_len = len(path) (root
    included), last_node = path[-1].
    ``row_of[b][node]`` gives the judge row of a node (identity if None).
    """
    B = tokens.shape[0]
    acc_len = np.zeros(B, dtype=np.int64)
    paths = []
    next_tok = np.zeros(B, dtype=np.int64)
    last = np.zeros(B, dtype=np.int64)
    for b in range(B):
        n = int(n_nodes[b])
        ro = (lambda j: j) if row_of is None else (lambda j, b=b: int(row_of[b][j]))
        if mode == MODE_THRESH_CHAIN:
            zp = [zprop[b][ro(i)] for i in range(n)]
            ls = [lse[b][ro(i)] for i in range(n)]
            L = accept_threshold_chain(zp, ls, n, tau)
            acc_len[b] = L
            paths.append(list(range(L)))
            next_tok[b] = int(argmax[b][ro(L)]) if L < n else -1
            last[b] = L - 1
        else:
            am = [int(argmax[b][ro(j)]) for j in range(n)]
            path, nt = accept_greedy_tree(tokens[b], tree_parent[b], n, am)
            acc_len[b] = len(path)
            paths.append(path)
            next_tok[b] = nt
            last[b] = path[-1]
    return acc_len, paths, next_tok, last


# --------------------------------------------------------------------------
# 4b. soft matching
# --------------------------------------------------------------------------
#
# "Speculative Streaming", verification step: soft matching accepts a drafted
# token x with probability min(1, p_target(x) / p_draft(x)) (the rejection
# sampling of Leviathan et al. that the page invokes), continues down the
# branch until a rejection, and samples one correction token at the
# rejection point from the main stream.  Readings: children of a node are
# tried in index order and the first accepted one is followed; each try is
# an independent test against the same p and q; the correction token is
# drawn from the normalised residual max(0, p - q) of the stop node (q = 0
# when the stop node has no drafted children, i.e. the bonus token is drawn
# from p); p and q are softmax(z / T).  The uniforms are inputs.

def softmax_t(z, temperature=1.0):
    """softmax(z / T) in float64."""
    z = np.asarray(z, dtype=np.float64) / float(temperature)
    m = z.max()
    e = np.exp(z - m)
    return e / e.sum()


def residual_sample(p, q, u):
    """Inverse-CDF draw from max(0, p - q) normalised (from p when q is None
    or the residual has no mass): the smallest v whose cumulative mass
    exceeds u times the total."""
    p = np.asarray(p, dtype=np.float64)
    r = p.copy() if q is None else np.maximum(0.0, p - np.asarray(q, dtype=np.float64))
    c = np.cumsum(r)
    if not c[-1] > 0.0:
        c = np.cumsum(p)
    v = int(np.searchsorted(c, float(u) * c[-1], side="right"))
    return min(v, len(c) - 1)


def accept_soft_tree(tokens, tree_parent, n_nodes, p_of, q_of, u_accept):
    """Soft-matching walk from the root (node 0).

    p_of(c): the target distribution at node c (over the token after c);
    q_of(c): the draft distribution c's children were drafted from, or None.
    Child x of the current node (index order) is accepted iff
    u_accept[x] * q(x) < p(x), i.e. u < p / q.  Returns the path.
    """
    cur = 0
    path = [0]
    while True:
        nxt = None
        p = None
        for c in range(n_nodes):
            if int(tree_parent[c]) != cur or c <= cur:
                continue
            if p is None:
                p = p_of(cur)
                q = q_of(cur)
            x = int(tokens[c])
            qx = 0.0 if q is None else float(q[x])
            if float(u_accept[c]) * qx < float(p[x]):
                nxt = c
                break
        if nxt is None:
            return path
        cur = nxt
        path.append(cur)


def accept_soft(logits, draft_logits, tokens, tree_parent, row_of, child_draft_row,
                n_nodes, u_accept, u_sample, temperature=1.0):
    """Soft-matching acceptance for every request.

    logits [B][Rj][V] (target), draft_logits [B][Rd][V]; row_of[b][c]: judge
    row of node c (identity if None); child_draft_row[b][c]: draft row of
    c's children (-1: none).  Returns (acc_len, paths, next_token,
    last_node) like ``accept`` in tree mode; next_token is the residual
    draw at the last node with u_sample[b].
    """
    B = len(tokens)
    acc_len = np.zeros(B, dtype=np.int64)
    paths, next_tok, last = [], np.zeros(B, dtype=np.int64), np.zeros(B, dtype=np.int64)
    for b in range(B):
        def row(c, b=b):
            return c if row_of is None else int(row_of[b][c])

        def p_of(c, b=b):
            return softmax_t(logits[b][row(c)], temperature)

        def q_of(c, b=b):
            dr = int(child_draft_row[b][c])
            return None if dr < 0 else softmax_t(draft_logits[b][dr], temperature)

        path = accept_soft_tree(tokens[b], tree_parent[b], int(n_nodes[b]), p_of, q_of,
                                u_accept[b])
        c = path[-1]
        acc_len[b] = len(path)
        paths.append(path)
        last[b] = c
        next_tok[b] = residual_sample(p_of(c), q_of(c), u_sample[b])
    return acc_len, paths, next_tok, last


# --------------------------------------------------------------------------
# 4c. tree draft construction and pruning
# --------------------------------------------------------------------------
#
# "Speculative Streaming", tree draft construction: the top-k tokens of
# each speculative stream's logits at the accepted position; stream-j
# tokens are the parents of stream-(j+1) tokens and stream-1 tokens the
# children of the root (the correction token); 1 + sum_g k^g nodes,
# flattened.  Parallel tree pruning: an edge (parent p, child c) survives
# iff softmax(early-exit logits at p)[token of c] reaches the threshold;
# a failing edge prunes the subtree under c.  Batching with streams: every
# surviving node carries gamma stream rows.  Readings: ties in top-k go to
# the lower token id; "falls below" prunes, so p >= threshold survives; the
# tree is flattened breadth-first (a node's children after all nodes of
# its level's predecessors, in parent order, then in top-k order), and
# pruning keeps that order.

def topk_tokens(z, k):
    """The k token ids of largest logit, largest first, ties to the lower id."""
    z = np.asarray(z, dtype=np.float64)
    order = np.lexsort((np.arange(len(z)), -z))
    return order[:k].astype(np.int64)


def draft_tree(stream_logits, k, root_token):
    """Full k-ary draft tree from gamma stream logit rows: (tokens, parent,
    depth) in breadth-first order; node 0 is the root."""
    gamma = len(stream_logits)
    top = [topk_tokens(stream_logits[j], k) for j in range(gamma)]
    tokens, parent, depth = [int(root_token)], [-1], [0]
    frontier = [0]
    for g in range(1, gamma + 1):
        nxt = []
        for p in frontier:
            for i in range(k):
                tokens.append(int(top[g - 1][i]))
                parent.append(p)
                depth.append(g)
                nxt.append(len(tokens) - 1)
        frontier = nxt
    return np.array(tokens), np.array(parent), np.array(depth)


def prune_tree(tokens, parent, early_logits, threshold):
    """Keep node c (> 0) iff its parent is kept and
    softmax(early_logits[parent[c]])[tokens[c]] >= threshold; the root is
    always kept.  Survivors keep their order.  Returns (tokens', parent'
    with new indices, keep_map: new index or -1 per old node)."""
    n = len(tokens)
    keep_map = np.full(n, -1, dtype=np.int64)
    new_tok, new_par = [], []
    probs = {}
    for c in range(n):
        p = int(parent[c])
        if c == 0:
            ok = True
        else:
            if p not in probs:
                probs[p] = softmax_t(early_logits[p])
            ok = keep_map[p] >= 0 and probs[p][int(tokens[c])] >= threshold
        if ok:
            keep_map[c] = len(new_tok)
            new_tok.append(int(tokens[c]))
            new_par.append(-1 if c == 0 else int(keep_map[p]))
    return np.array(new_tok), np.array(new_par), keep_map


def ss_block_vparent(parent, gamma, n_rows):
    """Parent pointers of the flattened SS block for a tree of n nodes: row j
    < n is node j (it sees its ancestors); row n + j*gamma + (s-1) is stream
    s of node j (stream 1 sees node j's view, stream s > 1 the view of
    stream s-1); rows past n(1 + gamma) up to n_rows are padding."""
    n = len(parent)
    vp = np.full(n_rows, VP_PAD, dtype=np.int64)
    for j in range(n):
        vp[j] = VP_ROOT if parent[j] < 0 else int(parent[j])
        for s in range(1, gamma + 1):
            r = n + j * gamma + (s - 1)
            vp[r] = j if s == 1 else r - 1
    return vp


# --------------------------------------------------------------------------
# 4d. stream value rotation and the ConFu future-token hand-off
# --------------------------------------------------------------------------

def rotate_stream_values(vb, n_nodes, gamma, eps):
    """"Speculative Streaming" Eq. 7 (value rotation): the value vector of
    stream s of node j is node j's value vector times e^{i eps s}.  Reading:
    consecutive pairs (v[2i], v[2i+1]) are the real and imaginary parts.
    vb [B][Hkv][R][d] (block values in the SS layout: rows 0..T_b-1 the
    nodes, row T_b + j*gamma + (s-1) stream s of node j); returns a float64
    copy with the stream rows rewritten."""
    out = np.array(vb, dtype=np.float64, copy=True)
    B = out.shape[0]
    for b in range(B):
        T = int(n_nodes[b])
        for j in range(T):
            for s in range(1, gamma + 1):
                r = T + j * gamma + (s - 1)
                c, sn = math.cos(eps * s), math.sin(eps * s)
                re, im = out[b, :, j, 0::2], out[b, :, j, 1::2]
                out[b, :, r, 0::2] = re * c - im * sn
                out[b, :, r, 1::2] = re * sn + im * c
    return out


def future_gather(o, last_node, row_offset):
    """"ConFu" key design 1: the future prediction handed to the next round
    is the output of the contemplate token attached to the last accepted
    node, block row row_offset + last_node (row_offset = T).  o
    [B][R][Hq][d] -> [B][Hq][d]."""
    o = np.asarray(o)
    return np.stack([o[b, row_offset + int(last_node[b])] for b in range(o.shape[0])])


# --------------------------------------------------------------------------
# 5. commit
# --------------------------------------------------------------------------

def kv_commit_contiguous(K, V, seq_len, k_block, v_block, paths):
    """Append accepted rows to a contiguous cache [B][Hkv][Smax][d].

    Row paths[b][i] of the block goes to position seq_len[b] + i; every
    other block row is dropped (LA sec. 3.2: speculative KV is not kept).
    Returns new (K, V, seq_len) copies.
    """
    K = K.copy()
    V = V.copy()
    seq = np.array(seq_len, dtype=np.int64).copy()
    for b, path in enumerate(paths):
        for i, row in enumerate(path):
            pos = int(seq[b]) + i
            if pos >= K.shape[2]:
                raise OverflowError("contiguous cache capacity exceeded")
            K[b, :, pos] = k_block[b, :, row]
            V[b, :, pos] = v_block[b, :, row]
        seq[b] += len(path)
    return K, V, seq


def kv_commit_paged(Kp, Vp, page_table, seq_len, free_pages, free_head,
                    k_block, v_block, paths, page_size):
    """Append accepted rows to a paged cache [n_pages][Hkv][d // blk][page][blk].

    Position t of request b lives in page page_table[b][t // page_size] at
    slot t % page_size (layout as ``gather_paged``).  Requests are served in ascending b; each first fills
    its partly used last page, then takes pages from
    free_pages[free_head], free_pages[free_head + 1], ... in order.
    Returns new (Kp, Vp, page_table, seq_len, free_head) copies.
    """
    Kp = Kp.copy()
    Vp = Vp.copy()
    pt = np.array(page_table).copy()
    seq = np.array(seq_len, dtype=np.int64).copy()
    head = int(free_head)
    for b, path in enumerate(paths):
        for i, row in enumerate(path):
            pos = int(seq[b]) + i
            j = pos // page_size
            if pos % page_size == 0:
                # a fresh page is needed for this position
                if j >= pt.shape[1]:
                    raise OverflowError("page table capacity exceeded")
                if head >= len(free_pages):
                    raise OverflowError("free page list exhausted")
                pt[b, j] = free_pages[head]
                head += 1
            p = int(pt[b, j])
            nblk, blk = Kp.shape[2], Kp.shape[4]
            for jj in range(nblk):
                Kp[p, :, jj, pos % page_size] = k_block[b, :, row, jj * blk:(jj + 1) * blk]
                Vp[p, :, jj, pos % page_size] = v_block[b, :, row, jj * blk:(jj + 1) * blk]
        seq[b] += len(path)
    return Kp, Vp, pt, seq, head
