"""Plain CPU oracle of the expert-parallel MoE layer forward pass.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import or call this
module; only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use it.  It shares no code with the CUDA library: it takes plain
numpy arrays (bf16 values as their uint16 bit patterns, fp32 logits) and
computes in float64, one obvious step at a time.

What it computes, and where each step is defined:

* route -- "Expert Coupling" (arXiv 2610.09372), Appendix A-A1, Table II
  (router: FP32 linear gate, top-k of E, gate weights are the selected
  probabilities) and FarSkip-Collective (arXiv 2511.11505), Sec. 2.1, the MoE
  definition MoE(A) = sum_j G(A)_j MLP^j(A) with G a sparse top-k selection.
  Reading: the k largest logits, ties to the lower expert index, weights a
  softmax over the selected k only (they sum to one).
* dispatch layout -- "Kernel fusion for expert parallelism" (brunomaga.github.io),
  section "Expert parallelism: dispatch and combine" (E_loc = E/W experts per
  rank) and "Expert Coupling" Sec. V-A (deduplicating dispatcher: one row per
  unique (token, destination rank); correlated placement: a per-layer
  permutation of expert IDs) and Appendix A-A2 (the receiver expands rows into
  expert-major order).
* expert FFN -- FarSkip-Collective Sec. 2.1 (gated MLP) and the kernel-fusion
  page, section "Fusing the layer into one kernel", stages 4-6 (gate/up MatMul,
  SwiGLU, down MatMul).  Reading: h = SiLU(x Wg^T) * (x Wu^T), y = h Wd^T.
* combine -- kernel-fusion page, section "Expert parallelism: dispatch and
  combine" (the owner sums the k weighted contributions; Sigma_t is the sum of
  the per-rank partials sigma^y_t), stage 7 "reduce" (scale by the routing
  weight, accumulate into the rank's partial), and "Expert Coupling" Sec. V-A
  (one partial output per (token, rank) pair); the residual add follows
  FarSkip-Collective Sec. 3 (o_{k+1} = o_k + f_{k+1}(.)).
* dense_forward -- the AllGather-ReduceScatter form of the kernel-fusion page:
  every expert evaluated on every token, zero weight where not routed.

Every function here is pinned by the CPU tests in ``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import numpy as np


# ----------------------------------------------------------------------------- helpers

def widen_bf16(a):
    """bf16 bit patterns (uint16) -> exact float64 values."""
    a = np.asarray(a, dtype=np.uint16)
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def slot_of_expert(placement, E):
    """Inverse of the placement permutation: slot[e] = p such that placement[p] == e.

    The placement lists, slot by slot, the global expert held there ("Expert
    Coupling" Sec. V-A: the placement is a permutation of global expert IDs).
    """
    placement = np.asarray(placement, dtype=np.int64)
    if placement.shape != (E,) or sorted(placement.tolist()) != list(range(E)):
        raise ValueError("placement is not a permutation of range(E)")
    slot = np.empty(E, dtype=np.int64)
    slot[placement] = np.arange(E)
    return slot


def rank_of_expert(placement, E, W):
    """rank(e) = slot(e) // (E / W): each rank holds E/W consecutive slots
    (kernel-fusion page, E_loc = E/W; "Expert Coupling" Sec. V-A, E/EP experts
    per GPU).  Identity placement gives rank(e) = e // (E/W)."""
    if E % W != 0:
        raise ValueError("E must be a multiple of W")
    return slot_of_expert(placement, E) // (E // W)


# ----------------------------------------------------------------------------- route

def route(logits, k, renormalize=True):
    """Top-k routing over fp32 logits.

    For every token t the pairs (-L[t,e], e) are sorted lexicographically and
    the first k kept: the k largest logits, in descending order, ties to the
    lower expert index.  The weights are a softmax over the k kept logits,
    w_j = exp(L_j - L_max) / sum_j' exp(L_j' - L_max), here in float64.
    renormalize=False keeps instead the full-softmax probabilities of the kept
    experts ("Expert Coupling" Table II read literally): the denominator sums
    over all E logits.

    Returns topk_ids int32 [N, k] and topk_w float64 [N, k].
    """
    L = np.asarray(logits, dtype=np.float32)
    N, E = L.shape
    if not (1 <= k <= E):
        raise ValueError("need 1 <= k <= E")
    if not np.all(np.isfinite(L)):
        raise ValueError("logits must be finite")
    expert = np.broadcast_to(np.arange(E), L.shape)
    order = np.lexsort((expert, -L.astype(np.float64)), axis=-1)  # last key is primary
    ids = order[:, :k]
    sel = np.take_along_axis(L, ids, axis=1).astype(np.float64)
    z = np.exp(sel - sel.max(axis=1, keepdims=True))
    if renormalize:
        w = z / z.sum(axis=1, keepdims=True)
    else:
        Lf = L.astype(np.float64)
        w = z / np.exp(Lf - sel.max(axis=1, keepdims=True)).sum(axis=1, keepdims=True)
    return ids.astype(np.int32), w


def route_sigmoid_bias(logits, bias, k):
    """The auxiliary-loss-free sigmoid router ("Expert Coupling" Appendix A-B:
    sigmoid scores with a per-expert bias; the DeepSeek-V3 router).  Reading:
    s_e = sigmoid(L_e) evaluated in float64 and rounded once to fp32; the k
    largest fp32 sums s_e + bias_e are selected (descending, ties to the lower
    expert index); the weights are s_e / sum of the selected s_e, in float64.
    The selection is a floating-point decision, so it is taken on the same
    fp32 values the kernel compares."""
    L = np.asarray(logits, dtype=np.float32)
    b = np.asarray(bias, dtype=np.float32)
    N, E = L.shape
    if not (1 <= k <= E):
        raise ValueError("need 1 <= k <= E")
    s = (1.0 / (1.0 + np.exp(-L.astype(np.float64)))).astype(np.float32)
    key = (s + b[None, :]).astype(np.float32)
    expert = np.broadcast_to(np.arange(E), L.shape)
    order = np.lexsort((expert, -key.astype(np.float64)), axis=-1)
    ids = order[:, :k]
    sel = np.take_along_axis(s, ids, axis=1).astype(np.float64)
    return ids.astype(np.int32), sel / sel.sum(axis=1, keepdims=True)


# ----------------------------------------------------------------------------- layout

def dispatch_layout(topk_ids, placement, E, W):
    """Dispatch layout: the row tables of the plain and the deduplicated dispatch.

    Plain: one row per (token, expert) pair.  Rows are grouped by expert in slot
    order (slot p holds expert placement[p]), and inside an expert's segment the
    tokens ascend.  This is a stable counting sort of the flat pairs (t, j) by
    slot(topk_ids[t, j]).

    Dedup: one row per distinct (token, rank) pair, rank-major, tokens ascending
    inside a rank.  expand_src maps each plain (expert-major) row to the dedup
    row it is copied from on the receiving rank.
    """
    ids = np.asarray(topk_ids, dtype=np.int64)
    N, k = ids.shape
    if np.any(ids < 0) or np.any(ids >= E):
        raise ValueError("expert id out of range")
    slot = slot_of_expert(placement, E)
    rank = rank_of_expert(placement, E, W)
    R = N * k

    # plain rows: counting sort by slot, stable in the flat pair index t*k + j
    key = slot[ids].reshape(-1)
    counts_by_slot = np.bincount(key, minlength=E)
    start_by_slot = np.concatenate([[0], np.cumsum(counts_by_slot)])
    order = np.argsort(key, kind="stable")          # flat pair index of each row
    row_token = (order // k).astype(np.int32)
    pair_row = np.empty(R, dtype=np.int64)
    pair_row[order] = np.arange(R)
    pair_row = pair_row.reshape(N, k).astype(np.int32)

    expert_counts = counts_by_slot[slot].astype(np.int32)             # by expert id
    expert_offsets = np.append(start_by_slot[slot], R).astype(np.int32)
    rank_offsets = start_by_slot[np.arange(W + 1) * (E // W)].astype(np.int32)

    # dedup rows: the distinct (token, rank) pairs
    member = np.zeros((N, W), dtype=bool)
    member[np.repeat(np.arange(N), k), rank[ids].reshape(-1)] = True
    r_of_row, t_of_row = np.nonzero(member.T)        # rank-major, tokens ascending
    R_d = len(t_of_row)
    dedup_counts = member.sum(axis=0).astype(np.int32)
    dedup_offsets = np.concatenate([[0], np.cumsum(dedup_counts)]).astype(np.int32)
    dedup_row_of = -np.ones((N, W), dtype=np.int64)
    dedup_row_of[t_of_row, r_of_row] = np.arange(R_d)
    pair_dedup_row = dedup_row_of[np.arange(N)[:, None], rank[ids]].astype(np.int32)
    expand_src = np.empty(R, dtype=np.int32)
    expand_src[pair_row.reshape(-1)] = pair_dedup_row.reshape(-1)

    return dict(
        expert_counts=expert_counts,
        expert_offsets=expert_offsets,
        rank_offsets=rank_offsets,
        row_token=row_token,
        pair_row=pair_row,
        dedup_counts=dedup_counts,
        dedup_offsets=dedup_offsets,
        dedup_row_token=t_of_row.astype(np.int32),
        pair_dedup_row=pair_dedup_row,
        expand_src=expand_src,
        n_dedup_rows=int(R_d),
        rank_member=member,
    )


def layout_stats(layout, N, k, W):
    """The per-layer counters of "Expert Coupling" Table I: rows dispatched,
    distinct ranks per token, rows removed by deduplication, and the share of
    tokens whose experts all sit on one rank."""
    member = layout["rank_member"]
    distinct = member.sum(axis=1)
    R, R_d = N * k, layout["n_dedup_rows"]
    return dict(
        rows=R,
        dedup_rows=R_d,
        dedup_reduction=1.0 - R_d / R,
        ranks_per_token=float(distinct.mean()),
        same_rank_share=float(np.mean(distinct == 1)),
        max_over_mean_load=float(layout["expert_counts"].max() / (R / len(layout["expert_counts"]))),
    )


# ----------------------------------------------------------------------------- dispatch

def dispatch(x, row_token):
    """Plain dispatch: xd[i] = x[row_token[i]] (a copy of bf16 rows)."""
    return np.asarray(x)[np.asarray(row_token, dtype=np.int64)]


def dispatch_dedup(x, dedup_row_token):
    """Dedup dispatch: one copy of each token per destination rank."""
    return np.asarray(x)[np.asarray(dedup_row_token, dtype=np.int64)]


def expand(xd_dedup, expand_src):
    """Receiver-side expansion of dedup rows into expert-major order."""
    return np.asarray(xd_dedup)[np.asarray(expand_src, dtype=np.int64)]


# ----------------------------------------------------------------------------- expert FFN

def silu(v):
    """SiLU(v) = v / (1 + exp(-v))."""
    return v / (1.0 + np.exp(-v))


def swiglu_mlp(X, wg, wu, wd):
    """One SwiGLU expert on rows X (float64 [n, H]); weights in nn.Linear layout
    wg, wu [I, H], wd [H, I] (float64).  h = SiLU(X wg^T) * (X wu^T), y = h wd^T."""
    g = X @ wg.T
    u = X @ wu.T
    h = silu(g) * u
    return h, h @ wd.T


def expert_ffn(xd, expert_offsets, expert_counts, wg, wu, wd):
    """Grouped expert FFN over the expert-major rows xd (bf16 bits [R, H]).

    Expert e owns rows [expert_offsets[e], expert_offsets[e] + expert_counts[e]).
    Returns h [R, I] and y [R, H] in float64 (no intermediate rounding).
    """
    X = widen_bf16(xd)
    E, I, H = np.shape(wg)
    R = X.shape[0]
    h = np.zeros((R, I))
    y = np.zeros((R, H))
    for e in range(E):
        a, n = int(expert_offsets[e]), int(expert_counts[e])
        if n == 0:
            continue
        h[a:a + n], y[a:a + n] = swiglu_mlp(X[a:a + n], widen_bf16(wg[e]), widen_bf16(wu[e]),
                                           widen_bf16(wd[e]))
    return h, y


# ----------------------------------------------------------------------------- combine

def combine(y, topk_w, pair_row, residual=None):
    """out[t] = residual[t] + sum_j w[t, j] * y[pair_row[t, j]], summed in j order."""
    N, k = np.shape(topk_w)
    out = np.zeros((N, y.shape[1])) if residual is None else widen_bf16(residual).copy()
    for j in range(k):
        out += np.asarray(topk_w)[:, j:j + 1] * y[np.asarray(pair_row)[:, j]]
    return out


def combine_dedup(y, topk_w, pair_row, pair_dedup_row, n_dedup_rows, residual=None):
    """Two-level combine of the deduplicating dispatcher.

    The rank that holds the experts forms one partial per (token, rank):
    partial[d] = sum over the token's j with pair_dedup_row[t, j] == d of
    w[t, j] * y[pair_row[t, j]] (j order).  The owner of the token then sums its
    partials in ascending rank order (dedup rows are rank-major, so ascending d)
    and adds the residual.
    """
    N, k = np.shape(topk_w)
    w = np.asarray(topk_w)
    partial = np.zeros((n_dedup_rows, y.shape[1]))
    for t in range(N):
        for j in range(k):
            partial[pair_dedup_row[t, j]] += w[t, j] * y[pair_row[t, j]]
    out = np.zeros((N, y.shape[1])) if residual is None else widen_bf16(residual).copy()
    for t in range(N):
        for d in sorted(set(int(v) for v in pair_dedup_row[t])):
            out[t] += partial[d]
    return partial, out


# ----------------------------------------------------------------------------- whole layer

def shared_expert(x, shared):
    """Shared expert (FarSkip-Collective Sec. 2.1: an MLP run on every token in
    addition to the routed experts): the SwiGLU MLP of (wg_s, wu_s, wd_s),
    bf16 weights [I_s, H], [I_s, H], [H, I_s], over all rows of x."""
    wg_s, wu_s, wd_s = shared
    return swiglu_mlp(widen_bf16(x), widen_bf16(wg_s), widen_bf16(wu_s), widen_bf16(wd_s))


def layer_forward(logits, x, wg, wu, wd, k, W, placement=None, residual=None, dedup=False,
                  shared=None):
    """The whole forward pass: route -> layout -> dispatch -> FFN -> combine,
    plus, if given, the shared expert's output added to every token."""
    N, E = np.shape(logits)
    placement = np.arange(E) if placement is None else placement
    ids, w = route(logits, k)
    lay = dispatch_layout(ids, placement, E, W)
    if dedup:
        xd_dedup = dispatch_dedup(x, lay["dedup_row_token"])
        xe = expand(xd_dedup, lay["expand_src"])
    else:
        xd_dedup = None
        xe = dispatch(x, lay["row_token"])
    h, y = expert_ffn(xe, lay["expert_offsets"], lay["expert_counts"], wg, wu, wd)
    if dedup:
        partial, out = combine_dedup(y, w, lay["pair_row"], lay["pair_dedup_row"],
                                     lay["n_dedup_rows"], residual)
    else:
        partial, out = None, combine(y, w, lay["pair_row"], residual)
    h_s = y_s = None
    if shared is not None:
        h_s, y_s = shared_expert(x, shared)
        out = out + y_s
    return dict(topk_ids=ids, topk_w=w, layout=lay, xd=xe, xd_dedup=xd_dedup, h=h, y=y,
                partial=partial, out=out, h_shared=h_s, y_shared=y_s)


def token_outputs(x_rows, ids_rows, w_rows, expert_weights, residual_rows=None):
    """Layer output for a few tokens, straight from the MoE definition
    out[t] = residual[t] + sum_j w[t, j] * MLP^{ids[t, j]}(x[t]).

    ``expert_weights(e)`` returns bf16 (wg[e], wu[e], wd[e]).  Used to check
    sampled tokens of full-size workloads one by one.
    """
    X = widen_bf16(x_rows)
    n = X.shape[0]
    out = np.zeros_like(X) if residual_rows is None else widen_bf16(residual_rows).copy()
    y_rows = np.zeros((n, ids_rows.shape[1], X.shape[1]))
    by_expert = {}
    for t in range(n):
        for j in range(ids_rows.shape[1]):
            by_expert.setdefault(int(ids_rows[t, j]), []).append((t, j))
    for e, pairs in sorted(by_expert.items()):
        wg, wu, wd = (widen_bf16(m) for m in expert_weights(e))
        ts = [t for t, _ in pairs]
        _, ye = swiglu_mlp(X[ts], wg, wu, wd)
        for (t, j), row in zip(pairs, ye):
            y_rows[t, j] = row
    for j in range(ids_rows.shape[1]):
        out += np.asarray(w_rows)[:, j:j + 1] * y_rows[:, j]
    return out, y_rows


def dense_forward(logits, x, wg, wu, wd, k, residual=None):
    """Brute-force dense form (the AllGather-ReduceScatter semantics): every
    expert runs on every token; G[t, e] is the routing weight where e is
    selected and zero elsewhere; out = residual + sum_e G[:, e] * MLP^e(x)."""
    N, E = np.shape(logits)
    ids, w = route(logits, k)
    G = np.zeros((N, E))
    np.put_along_axis(G, ids.astype(np.int64), w, axis=1)
    X = widen_bf16(x)
    out = np.zeros_like(X) if residual is None else widen_bf16(residual).copy()
    for e in range(E):
        _, ye = swiglu_mlp(X, widen_bf16(wg[e]), widen_bf16(wu[e]), widen_bf16(wd[e]))
        out += G[:, e:e + 1] * ye
    return out


# ----------------------------------------------------------------------------- placement search

def coselection(topk_ids, E):
    """Co-selection counts of "Expert Coupling" Sec. V-A and Appendix A-D
    (Algorithm 1): W[e, e'] = number of tokens whose selected set contains both
    e and e'.  Symmetric; the diagonal W[e, e] counts the tokens that select e."""
    ids = np.asarray(topk_ids, dtype=np.int64)
    W = np.zeros((E, E), dtype=np.int64)
    for j in range(ids.shape[1]):
        for j2 in range(ids.shape[1]):
            np.add.at(W, (ids[:, j], ids[:, j2]), 1)
    return W


def swap_gain(W, group, a, b):
    """Change of the within-group co-selection total when experts a and b
    (in different groups) trade places."""
    A, B = group[a], group[b]
    in_A = (group == A)
    in_B = (group == B)
    in_A[a] = False
    in_B[b] = False
    return int(W[a, in_B].sum() + W[b, in_A].sum() - W[a, in_A].sum() - W[b, in_B].sum())


def partition(W, G, max_swaps):
    """Balanced partition ("Expert Coupling" Appendix A-D, procedure Partition):
    start from G contiguous groups of E/G experts; repeatedly apply the swap of
    two experts from different groups with the largest gain in within-group
    co-selection, until no swap has a positive gain or max_swaps swaps were
    made.  Reading of "the swap with the largest gain" when several tie: the
    pair (a, b), a < b, that comes first in lexicographic order.
    Returns (group of each expert, number of swaps made)."""
    W = np.asarray(W, dtype=np.int64)
    E = W.shape[0]
    if E % G != 0:
        raise ValueError("E must be a multiple of the number of groups")
    group = np.arange(E) // (E // G)
    swaps = 0
    for _ in range(max_swaps):
        best, pair = 0, None
        for a in range(E):
            for b in range(a + 1, E):
                if group[a] == group[b]:
                    continue
                g = swap_gain(W, group, a, b)
                if g > best:
                    best, pair = g, (a, b)
        if pair is None:
            break
        a, b = pair
        group[a], group[b] = group[b], group[a]
        swaps += 1
    return group, swaps


def correlated_placement(W, ranks, nodes=1, max_swaps=10_000):
    """Algorithm 1 of "Expert Coupling": one node -> Partition(W, P); several
    nodes -> Partition across nodes first, then each node's experts (in
    ascending id order) across its P/N ranks; rank(e) = n * P/N + rho_n(e).
    Returned as a placement permutation: slot p holds placement[p], ranks take
    E/P consecutive slots, experts of a rank in ascending id order."""
    W = np.asarray(W, dtype=np.int64)
    E = W.shape[0]
    if ranks % nodes != 0 or E % ranks != 0:
        raise ValueError("need nodes | ranks | E")
    rank = np.empty(E, dtype=np.int64)
    swaps = 0
    if nodes == 1:
        rank, swaps = partition(W, ranks, max_swaps)
    else:
        node, s = partition(W, nodes, max_swaps)
        swaps += s
        per = ranks // nodes
        for n in range(nodes):
            members = np.nonzero(node == n)[0]
            rho, s = partition(W[np.ix_(members, members)], per, max_swaps)
            swaps += s
            rank[members] = n * per + rho
    placement = np.concatenate([np.nonzero(rank == r)[0] for r in range(ranks)])
    return placement.astype(np.int32), swaps


def within_rank_coselection(W, placement, ranks):
    """Total co-selection of expert pairs that share a rank (the objective)."""
    E = len(placement)
    rank = np.empty(E, dtype=np.int64)
    rank[np.asarray(placement)] = np.arange(E) // (E // ranks)
    total = 0
    for a in range(E):
        for b in range(a + 1, E):
            if rank[a] == rank[b]:
                total += int(W[a, b])
    return total
