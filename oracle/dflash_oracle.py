"""CPU oracle of the DFlash hot path -- TEST INFRASTRUCTURE, not product code.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this module. It shares no code with the CUDA path (it imports
nothing from the package) and takes plain numpy arrays; every floating-point
step runs in float64 from the exact values of the (bf16 or fp32) inputs.

Each function states the passage it follows. Page names:
  [DFlash]  "DFlash 块扩散解码" -- sections "KV 注入" (fusion, K/V injection and
            attention equations) and "验证流程" (verify steps).
  [SGLang]  "详解SGlang 最新DFlash投机解码算法的工程实现" -- section 3 (greedy
            accept rule and its tensor code), section 4.1 (KV materialisation:
            project, kv_proj, k_norm, k_rope, prefix-valid write), section 5.1
            (req_to_token position -> KV slot mapping).
  [SpecDec] "让大模型快 8 倍：从投机解码到 DDTree" -- section 3 (min(1, p/q) rule,
            residual distribution, 5-token worked example, identity
            min(p,q) + max(0, p-q) = p) and section 4 (cascade discard).
  [DLoop]   "DLoop 完全拆解" -- "机制一" (gate score c_s and the rule c_s >= g) and
            the looped verify of S concatenated blocks.

Readings where the pages are silent (each listed again in the design notes):
  * weights are stored [out, in] and applied as W @ x;
  * k_norm is RMSNorm over head_dim, x / sqrt(mean(x^2) + eps) * w;
  * k_rope is rotate-half RoPE, pair (i, i + D/2), angle pos * theta^(-2i/D);
  * softmax scale is 1/sqrt(D) unless given;
  * greedy argmax breaks ties by the lowest token index;
  * sampled accept is u < p(x)/q(x) (strict), one uniform per draft position and
    one per sequence for the resample; the inverse CDF walks the vocabulary in
    ascending index order and returns the smallest y with C(y) > u * Z;
  * a zero residual mass (reachable only through rounding) falls back to p;
  * uniforms within 1e-6 of a decision boundary are flagged, not trusted.
"""
from __future__ import annotations

import numpy as np

# flag bits of the sampled verify
FLAG_ACCEPT_BOUNDARY = 1   # |u - p/q| < 1e-6 at an evaluated accept test with p/q < 1
FLAG_CDF_BOUNDARY = 2      # u_final within 1e-6 of C(y-1)/Z or C(y)/Z
FLAG_DEGENERATE = 4        # residual mass Z == 0 at the rejection row
FLAG_INVALID = 8           # candidate had q(x) == 0 (not a draw from q)
FLAG_GATE_BOUNDARY = 1     # gate: |c - g| < 1e-4

BOUNDARY_EPS = 1e-6
GATE_EPS = 1e-4


def _f64(x):
    return np.asarray(x, dtype=np.float64)


# ---------------------------------------------------------------------------
# (a) target-context KV materialisation
# ---------------------------------------------------------------------------
def rms_norm(x, w, eps):
    """RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * w."""
    x = _f64(x)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * _f64(w)


def rope_rotate_half(x, pos, theta):
    """Rotate-half RoPE of vectors x[..., D] at absolute position ``pos``.

    Pair i (0 <= i < D/2) is (x[i], x[i + D/2]); it is turned by the angle
    pos * theta^(-2i/D).
    """
    x = _f64(x)
    D = x.shape[-1]
    half = D // 2
    i = np.arange(half, dtype=np.float64)
    ang = float(pos) * theta ** (-2.0 * i / D)
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def materialize_ctx_kv(hidden, commit_len, start_pos, W_f, b_f, W_kv, k_norm_w,
                       rms_eps, rope_theta, k_pools, v_pools, page_table, page_size):
    """Write the committed rows' context K/V into every draft layer's paged cache.

    [DFlash] KV 注入 step 2: h_ctx = W_f [h_l1; ...; h_lm] + b_f.
    [DFlash] KV 注入 step 3: K_ctx^(l) = h_ctx W_K^(l), V_ctx^(l) = h_ctx W_V^(l).
    [SGLang] 4.1: per layer kv_proj, then k_norm, then k_rope(positions), then a
      prefix-valid write: only rows j < commit_len[b] of sequence b are written.
    [SGLang] 5.1: logical position -> physical slot through the request's page
      table (page = table[b][pos // page], slot = pos % page).

    hidden [B, rows, m*d]; W_f [d, m*d]; b_f [d]; W_kv [L, 2, Hkv*D, d];
    k_norm_w [L, D] or None; pools: L arrays [num_pages, page, Hkv, D].
    Returns new float64 copies of the K and V pools; untouched rows keep their
    input values.
    """
    hidden = _f64(hidden)
    W_f, b_f, W_kv = _f64(W_f), _f64(b_f), _f64(W_kv)
    L = W_kv.shape[0]
    k_out = [_f64(p).copy() for p in k_pools]
    v_out = [_f64(p).copy() for p in v_pools]
    Hkv, D = k_out[0].shape[2], k_out[0].shape[3]
    B = hidden.shape[0]
    for b in range(B):
        n = int(commit_len[b])
        if n == 0:
            continue
        h_ctx = hidden[b, :n] @ W_f.T + b_f                    # [n, d]
        for layer in range(L):
            k = (h_ctx @ W_kv[layer, 0].T).reshape(n, Hkv, D)
            v = (h_ctx @ W_kv[layer, 1].T).reshape(n, Hkv, D)
            if k_norm_w is not None:
                k = rms_norm(k, _f64(k_norm_w)[layer], rms_eps)
            for j in range(n):
                pos = int(start_pos[b]) + j
                kj = k[j]
                if rope_theta > 0:
                    kj = rope_rotate_half(kj, pos, rope_theta)
                page = int(page_table[b, pos // page_size])
                slot = pos % page_size
                k_out[layer][page, slot] = kj
                v_out[layer][page, slot] = v[j]
    return k_out, v_out


# ---------------------------------------------------------------------------
# (b) draft block attention
# ---------------------------------------------------------------------------
def gather_ctx(pool, page_table_row, ctx_len, page_size):
    """Rows 0..ctx_len-1 of one sequence from a paged pool: [ctx_len, Hkv, D]."""
    pos = np.arange(int(ctx_len))
    pages = np.asarray(page_table_row)[pos // page_size]
    return _f64(pool)[pages, pos % page_size]


def block_attn(q, k_blk, v_blk, k_pool, v_pool, page_table, ctx_len, page_size, scale=None, causal=False):
    """Attention(Q_draft, [K_draft; K_ctx], [V_draft; V_ctx]) with no mask.

    [DFlash] 块扩散 (draft uses bidirectional, non-causal attention inside the
    block) and KV 注入 step 3 (queries of the draft tokens attend to the block's
    own K/V and to the injected context K/V). Grouped-query attention: q-head h
    reads kv-head h // (Hq / Hkv).

    causal=True is the in-block causal variant of [DFlash] 块扩散的双向注意力问题
    (JetSpec: block position i sees positions 0 .. i): query i, at block row
    i + n_kv - n_q, keeps every context key and the block keys up to its own
    row. Requires n_kv >= n_q.

    q [B, n_q, Hq, D]; k_blk, v_blk [B, n_kv, Hkv, D]; pools [pages, page, Hkv, D].
    Returns out [B, n_q, Hq, D] in float64.
    """
    q, k_blk, v_blk = _f64(q), _f64(k_blk), _f64(v_blk)
    B, n_q, Hq, D = q.shape
    Hkv = k_blk.shape[2]
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    out = np.zeros((B, n_q, Hq, D))
    for b in range(B):
        Kc = gather_ctx(k_pool, page_table[b], ctx_len[b], page_size)
        Vc = gather_ctx(v_pool, page_table[b], ctx_len[b], page_size)
        K = np.concatenate([Kc, k_blk[b]], axis=0)            # [keys, Hkv, D]
        V = np.concatenate([Vc, v_blk[b]], axis=0)
        C = Kc.shape[0]
        n_kv = k_blk.shape[1]
        for h in range(Hq):
            g = h // G
            s = scale * (q[b, :, h, :] @ K[:, g, :].T)         # [n_q, keys]
            if causal:
                assert n_kv >= n_q, "causal block attention needs n_kv >= n_q"
                for i in range(n_q):
                    s[i, C + i + n_kv - n_q + 1:] = -np.inf
            s = s - s.max(axis=1, keepdims=True)
            w = np.exp(s)
            w = w / w.sum(axis=1, keepdims=True)
            out[b, :, h, :] = w @ V[:, g, :]
    return out


# ---------------------------------------------------------------------------
# (c) verify: greedy rule
# ---------------------------------------------------------------------------
def verify_greedy(target_logits, cand, n_draft=None):
    """Greedy accept rule.

    [SGLang] 3: target_predict[i] = argmax of target row i; matches[i] =
    (cand[i+1] == target_predict[i]); accept_len = number of leading matches
    (cumulative product, then sum); bonus = target_predict[accept_len];
    commit_len = accept_len + 1 (at least one token is always committed).
    [SpecDec] 4: after the first mismatch every later draft is discarded.

    target_logits [B, n_max+1, V]; cand [B, n_max+1] (cand[:, 0] is the anchor);
    n_draft [B] drafts to check per sequence (rows beyond are ignored).
    Returns dict: accept_len, bonus, commit_len, out_tokens [B, n_max+1] (the
    accepted drafts then the bonus, padded with -1), target_pred [B, n_max+1]
    (argmax of each checked row, -1 beyond).
    """
    z = _f64(target_logits)
    cand = np.asarray(cand, dtype=np.int64)
    B, R, V = z.shape
    n_max = R - 1
    if n_draft is None:
        n_draft = np.full(B, n_max)
    acc = np.zeros(B, dtype=np.int32)
    bonus = np.zeros(B, dtype=np.int64)
    out_tokens = np.full((B, R), -1, dtype=np.int64)
    target_pred = np.full((B, R), -1, dtype=np.int64)
    for b in range(B):
        n = int(n_draft[b])
        for r in range(n + 1):
            target_pred[b, r] = int(np.argmax(z[b, r]))      # first index among ties
        a = 0
        while a < n and cand[b, a + 1] == target_pred[b, a]:
            a += 1
        acc[b] = a
        bonus[b] = target_pred[b, a]
        out_tokens[b, :a] = cand[b, 1:a + 1]
        out_tokens[b, a] = bonus[b]
    return {"accept_len": acc, "bonus": bonus, "commit_len": acc + 1,
            "out_tokens": out_tokens, "target_pred": target_pred}


# ---------------------------------------------------------------------------
# (c) verify: sampled rule
# ---------------------------------------------------------------------------
def softmax(z, temperature=1.0):
    """softmax(z / T) over the last axis, float64."""
    s = _f64(z) / temperature
    s = s - s.max(axis=-1, keepdims=True)
    e = np.exp(s)
    return e / e.sum(axis=-1, keepdims=True)


def inverse_cdf(weights, u):
    """Smallest index y with C(y) > u * Z, C the running sum of ``weights`` in
    ascending index order and Z its total. Also returns whether u lies within
    1e-6 of C(y-1)/Z or C(y)/Z."""
    w = _f64(weights)
    C = np.cumsum(w)
    Z = C[-1]
    y = int(np.argmax(C > u * Z))
    lo = C[y - 1] / Z if y > 0 else 0.0
    hi = C[y] / Z
    near = abs(lo - u) < BOUNDARY_EPS or abs(hi - u) < BOUNDARY_EPS
    return y, near


def verify_sample(target_logits, draft_logits, cand, n_draft, u_acc, u_final, temperature=1.0):
    """Sampled (rejection-sampling) accept rule.

    [SpecDec] 3: a drafted token x is accepted with probability min(1, p(x)/q(x)),
    realised as u < p(x)/q(x) with the supplied uniform u. On rejection the token
    is redrawn from the residual p'(y) = max(0, p(y) - q(y)) / (1 - beta), with
    beta = sum_y min(p(y), q(y)); the mass 1 - beta is computed directly as
    Z = sum_y max(0, p(y) - q(y)).
    [SpecDec] 4: after the first rejection every later draft is discarded.
    [DFlash] 验证流程 / pseudocode: if every draft is accepted, the bonus is drawn
    from the target's last row p_n.
    [DLoop] looped verify: S blocks concatenated into one candidate list are
    checked by the same sequential rule.

    target_logits [B, n_max+1, V]: p_r = softmax(row r / T);
    draft_logits [B, n_max, V]: q_r = softmax(row r / T) is the law cand[r+1]
    was drawn from; u_acc [B, n_max]; u_final [B].
    Returns dict like verify_greedy plus flags [B] and, per sequence, the
    debug values p_x, q_x (per checked position), Z, one_minus_beta, and the
    final distribution the bonus was drawn from.
    """
    zt, zd = _f64(target_logits), _f64(draft_logits)
    cand = np.asarray(cand, dtype=np.int64)
    B, R, V = zt.shape
    acc = np.zeros(B, dtype=np.int32)
    bonus = np.zeros(B, dtype=np.int64)
    flags = np.zeros(B, dtype=np.uint8)
    out_tokens = np.full((B, R), -1, dtype=np.int64)
    debug = []
    for b in range(B):
        n = int(n_draft[b])
        p = softmax(zt[b, :n + 1], temperature)               # [n+1, V]
        q = softmax(zd[b, :n], temperature) if n > 0 else np.zeros((0, V))
        a = 0
        rejected = False
        p_x, q_x = [], []
        for i in range(1, n + 1):
            x = int(cand[b, i])
            px, qx = p[i - 1, x], q[i - 1, x]
            p_x.append(px)
            q_x.append(qx)
            if qx == 0.0:
                flags[b] |= FLAG_INVALID
                ratio = np.inf
            else:
                ratio = px / qx
            if ratio < 1.0 and abs(float(u_acc[b, i - 1]) - ratio) < BOUNDARY_EPS:
                flags[b] |= FLAG_ACCEPT_BOUNDARY
            if float(u_acc[b, i - 1]) < ratio:
                a += 1
            else:
                rejected = True
                break
        Z = one_minus_beta = None
        if rejected:
            row_p, row_q = p[a], q[a]
            resid = np.maximum(0.0, row_p - row_q)
            Z = resid.sum()
            one_minus_beta = 1.0 - np.minimum(row_p, row_q).sum()
            if Z == 0.0:
                flags[b] |= FLAG_DEGENERATE
                dist = row_p
            else:
                dist = resid
        else:
            dist = p[n]
        y, near = inverse_cdf(dist, float(u_final[b]))
        if near:
            flags[b] |= FLAG_CDF_BOUNDARY
        acc[b] = a
        bonus[b] = y
        out_tokens[b, :a] = cand[b, 1:a + 1]
        out_tokens[b, a] = y
        debug.append({"p_x": np.array(p_x), "q_x": np.array(q_x), "Z": Z,
                      "one_minus_beta": one_minus_beta,
                      "final_dist": dist / dist.sum()})
    return {"accept_len": acc, "bonus": bonus, "commit_len": acc + 1,
            "out_tokens": out_tokens, "flags": flags, "debug": debug}


# ---------------------------------------------------------------------------
# Draft-side token choice over the MASK positions
# ---------------------------------------------------------------------------
def draft_select(draft_logits, anchor, n_draft=None, u_draft=None, temperature=0.0):
    """Candidates of one round from the draft's MASK-position logits.

    [DFlash] 推理流程 step 4 and its decode listing: the block is [anchor, MASK,
    ..., MASK]; the logits of MASK position i give draft token i, taken as the
    argmax (draft_tokens = argmax(logits[i]) for i = 1 .. k-1). [SpecDec] DFlash
    section: a token is sampled from each position's distribution instead; the
    candidates are [anchor] + draft tokens. [SGLang] 3 decode listing: the same
    [last_bonus] + draft_tokens candidate layout.

    draft_logits [B, n_max, V] (row i <-> draft position i + 1); anchor [B];
    n_draft [B] (rows i >= n_b are not drafted); u_draft [B, n_max] uniforms.
    temperature == 0: argmax with the lowest index on ties; q_x = 1 (the greedy
    draft is a point mass); row_lse = LSE(z).
    temperature > 0: x ~ softmax(z / T) by inverse CDF in ascending token order
    (smallest y with C(y) > u * Z); q_x = softmax(z / T)[x]; row_lse =
    LSE(z / T); flags FLAG_CDF_BOUNDARY when u is within 1e-6 of C(y-1)/Z or
    C(y)/Z.
    Returns cand [B, n_max+1] int64 (cand[:, 0] = anchor, -1 past n_b), q_x and
    row_lse [B, n_max] float64 (0 past n_b), flags [B, n_max] uint8.
    """
    z = _f64(draft_logits)
    B, n_max, V = z.shape
    n_draft = np.full(B, n_max) if n_draft is None else np.asarray(n_draft)
    cand = np.full((B, n_max + 1), -1, dtype=np.int64)
    cand[:, 0] = np.asarray(anchor, dtype=np.int64)
    q_x = np.zeros((B, n_max))
    row_lse = np.zeros((B, n_max))
    flags = np.zeros((B, n_max), dtype=np.uint8)
    T = temperature if temperature > 0 else 1.0
    for b in range(B):
        for i in range(int(n_draft[b])):
            row = z[b, i]
            s = row / T
            mx = s.max()
            row_lse[b, i] = mx + np.log(np.exp(s - mx).sum())
            if temperature > 0:
                y, near = inverse_cdf(np.exp(s - mx), float(u_draft[b, i]))
                cand[b, i + 1] = y
                q_x[b, i] = np.exp(s[y] - row_lse[b, i])
                flags[b, i] = FLAG_CDF_BOUNDARY if near else 0
            else:
                cand[b, i + 1] = int(np.argmax(row))    # first maximum: lowest index
                q_x[b, i] = 1.0
    return dict(cand=cand, q_x=q_x, row_lse=row_lse, flags=flags)


# ---------------------------------------------------------------------------
# DLoop block gate
# ---------------------------------------------------------------------------
def log_softmax_at(z, x, temperature=1.0):
    """log softmax(z / T)[x] for one row: z[x]/T - LSE_v(z[v]/T)."""
    s = _f64(z) / temperature
    mx = s.max()
    return s[int(x)] - (mx + np.log(np.exp(s - mx).sum()))


def gate(draft_logits, tokens, active, temperature, g):
    """[DLoop] 机制一: c_s = sum over the block's drafted tokens of
    log p_draft(x_i); draft another stage iff c_s >= g.

    draft_logits [B, k, V]; tokens [B, k]; active [B] (inactive sequences get
    c = 0, cont = 0). Returns c [B], cont [B] uint8, row_lse [B, k] (LSE of
    row / T), flags [B] (|c - g| < 1e-4).
    """
    z = _f64(draft_logits)
    B, k, V = z.shape
    c = np.zeros(B)
    cont = np.zeros(B, dtype=np.uint8)
    flags = np.zeros(B, dtype=np.uint8)
    row_lse = np.zeros((B, k))
    for b in range(B):
        for i in range(k):
            s = z[b, i] / temperature
            mx = s.max()
            row_lse[b, i] = mx + np.log(np.exp(s - mx).sum())
        if active is not None and not active[b]:
            continue
        c[b] = sum(log_softmax_at(z[b, i], tokens[b, i], temperature) for i in range(k))
        cont[b] = 1 if c[b] >= g else 0
        if abs(c[b] - g) < GATE_EPS:
            flags[b] |= FLAG_GATE_BOUNDARY
    return {"c": c, "cont": cont, "row_lse": row_lse, "flags": flags}


def dloop_stage_count(conts):
    """[DLoop] 机制一: stages drafted before verify. ``conts`` is [S, B] of gate
    decisions; stage s+1 is drafted only while every earlier gate said continue,
    and the stage whose gate said stop is still verified. Returns S_b in 1..S."""
    conts = np.asarray(conts)
    S, B = conts.shape
    out = np.full(B, S, dtype=np.int32)
    for b in range(B):
        for s in range(S):
            if conts[s, b] == 0:
                out[b] = s + 1
                break
    return out


# ---------------------------------------------------------------------------
# DDTree: draft tree from the per-position marginals, greedy tree walk
# ([SpecDec] section 6: 6.1 tree shape, 6.2 node budget, 6.3 best-first heap,
# 6.5 greedy walk)
# ---------------------------------------------------------------------------
FLAG_TREE_TIE = 1     # two candidates within 1e-5 in log-probability decided a pop


def ddtree_topk(draft_logits, K, temperature=1.0):
    """[SpecDec] 6.1: the K most probable tokens of every drafted position.

    draft_logits [B, n, V] (row i <-> position i + 1). Returns tok [B, n, K]
    int64 sorted by probability (ties: lower token index first) and logp
    [B, n, K] = log softmax(z / T) at those tokens, float64.
    """
    z = _f64(draft_logits) / temperature
    B, n, V = z.shape
    mx = z.max(axis=2, keepdims=True)
    lse = mx + np.log(np.exp(z - mx).sum(axis=2, keepdims=True))
    tok = np.zeros((B, n, K), dtype=np.int64)
    logp = np.zeros((B, n, K))
    for b in range(B):
        for i in range(n):
            order = np.lexsort((np.arange(V), -z[b, i]))[:K]   # value desc, then index asc
            tok[b, i] = order
            logp[b, i] = z[b, i, order] - lse[b, i, 0]
    return tok, logp


def ddtree_build(tok, logp, budget):
    """[SpecDec] 6.3 best-first heap, taken step by step: the root's candidate
    children (the position-1 top-K) go on a heap ordered by path probability;
    each step pops the most probable candidate into the tree and pushes its
    children (the next position's top-K, path log-probability = parent's +
    the child's); stop when the tree holds ``budget`` nodes (the root, the
    already verified anchor, takes no slot) or the heap is empty. A path's
    probability is the product of the per-position marginals (6.3).

    Ties (reading; the pages do not order equal probabilities): the candidate
    with the smaller depth, then the earlier-popped parent (the root first),
    then the lower rank among its siblings pops first. A pop that a distinct
    candidate trails by less than 1e-5 in log-probability flags the sequence
    (exact ties are decided by the order and are not flagged).

    tok [B, n, K], logp [B, n, K]. Returns node_token, node_parent (index of
    the parent node, -1 = root), node_depth (1-based position), node_rank
    [B, budget] int (-1 past n_nodes), node_logp [B, budget] float64, n_nodes
    [B], flags [B]. Nodes are in pop order, so every parent precedes its
    children.
    """
    import heapq
    tok = np.asarray(tok)
    logp = _f64(logp)
    B, n, K = tok.shape
    node_token = np.full((B, budget), -1, dtype=np.int64)
    node_parent = np.full((B, budget), -1, dtype=np.int32)
    node_depth = np.full((B, budget), -1, dtype=np.int32)
    node_rank = np.full((B, budget), -1, dtype=np.int32)
    node_logp = np.zeros((B, budget))
    n_nodes = np.zeros(B, dtype=np.int32)
    flags = np.zeros(B, dtype=np.uint8)
    for b in range(B):
        # entry: (-path logp, depth, parent pop index (-1 = root), rank)
        heap = [(-logp[b, 0, r], 1, -1, r) for r in range(K)] if n > 0 else []
        heapq.heapify(heap)
        cnt = 0
        while heap and cnt < budget:
            neg, d, par, r = heapq.heappop(heap)
            # exact ties are decided by the order above; a distinct candidate
            # closer than 1e-5 could swap places under another rounding
            others = [h[0] for h in heap if h[0] != neg]
            if others and min(others) - neg < 1e-5:
                flags[b] = FLAG_TREE_TIE
            node_token[b, cnt] = tok[b, d - 1, r]
            node_parent[b, cnt] = par
            node_depth[b, cnt] = d
            node_rank[b, cnt] = r
            node_logp[b, cnt] = -neg
            if d < n:
                for rc in range(K):
                    heapq.heappush(heap, (neg - logp[b, d, rc], d + 1, cnt, rc))
            cnt += 1
        n_nodes[b] = cnt
    return dict(node_token=node_token, node_parent=node_parent, node_depth=node_depth, node_rank=node_rank,
                node_logp=node_logp, n_nodes=n_nodes, flags=flags)


def ddtree_walk_greedy(target_logits, node_token, node_parent, n_nodes):
    """[SpecDec] 6.5 greedy tree walk with the greedy accept rule ([SGLang] 3):
    start at the root; at the current node (row 0 for the root, row 1 + j for
    node j: the target's distribution after the path to that node) the target
    predicts argmax of that row (lowest index on ties); the child holding that
    token is accepted and becomes the current node (siblings hold distinct
    tokens, so there is at most one); stop when no child holds it. The bonus is
    the prediction at the last accepted node.

    target_logits [B, 1 + budget, V]; node_token, node_parent [B, budget];
    n_nodes [B]. Returns accept_len [B] (accepted nodes), commit_len =
    accept_len + 1, bonus [B], path [B, n_path_max] node indices (-1 padded),
    out_tokens [B, budget + 1] (accepted tokens then the bonus, -1 padded).
    """
    z = _f64(target_logits)
    B, R, V = z.shape
    budget = R - 1
    acc = np.zeros(B, dtype=np.int32)
    bonus = np.zeros(B, dtype=np.int64)
    path = np.full((B, budget), -1, dtype=np.int32)
    out_tokens = np.full((B, budget + 1), -1, dtype=np.int64)
    for b in range(B):
        cur = -1            # the root
        a = 0
        while True:
            row = 0 if cur < 0 else 1 + cur
            tp = int(np.argmax(z[b, row]))
            nxt = -1
            for j in range(int(n_nodes[b])):
                if node_parent[b, j] == cur and node_token[b, j] == tp:
                    nxt = j
                    break
            if nxt < 0:
                bonus[b] = tp
                break
            path[b, a] = nxt
            out_tokens[b, a] = tp
            a += 1
            cur = nxt
        acc[b] = a
        out_tokens[b, a] = bonus[b]
    return dict(accept_len=acc, commit_len=acc + 1, bonus=bonus, path=path, out_tokens=out_tokens)
