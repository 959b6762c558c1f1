"""Plain fp64 CPU oracle of the dropless (MegaBlocks-style) MoE block.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / reference leg of ``bench.py`` may import this
module.  The CUDA library never calls it and shares no code with it.

Source of every definition: George Lin's blog post on MoE training systems
(MegaBlocks / FlexMoE / fused communication-computation), section 1
"MegaBlocks: MoE as block-sparse matrix multiplication":

* 1.1  each token is sent to experts by a gate network; dropless means no
       expert has a capacity, so no token is ever dropped.
* 1.2  expert i computes Output_i = Input_i @ W_i^1 with W_i^1 in R^{d x F};
       all experts together are one block-sparse product: SDD (layer 1),
       an activation, then DSD (layer 2, which uses the weight "in transposed
       form"); the weight gradient is DSTD (section 1.3).
* 1.3  block size 128x128; token counts are padded to a multiple of 128
       (at most 127 pad rows per expert); the hybrid BCSR-COO format keeps
       BCSR row offsets and column indices and also materialises each
       nonzero block's row index; the transpose index lists every nonzero
       block in transposed (column-major) order without copying data.
* 1.4  one kernel reorders tokens from batch order into expert-grouped
       order and pads each group; one kernel builds the topology and its
       transpose metadata.

Everything is computed in float64 from the bf16 / fp32 inputs, without
intermediate rounding, with the plainest loops that state each definition.
Matrix products use ``numpy.matmul`` as a library step.  Readings taken where
the page is silent:

* router: softmax over all E experts; the k largest are taken on the fp32
  logits themselves (softmax is monotone, so this is the same choice, made
  without any rounding), ties to the lower expert id; weights are the
  softmax probabilities, renormalised over the chosen k on request.
* order inside an expert group: ascending assignment index a = t*k + j.
* pad rows of the permuted input and of the permuted output gradient are 0.
* transpose order: column ascending, then row ascending.
* GELU is the exact erf form; SwiGLU is silu(x W1) * (x W3).
"""

from __future__ import annotations

import numpy as np
from scipy.special import erf as _erf

BLOCK = 128
SQRT1_2 = np.sqrt(0.5)
INV_SQRT_2PI = 1.0 / np.sqrt(2.0 * np.pi)


# ----------------------------------------------------------------------------
# encodings
# ----------------------------------------------------------------------------

def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Decode bf16 bit patterns (uint16) to float64 exactly."""
    u = np.asarray(bits).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        return u.view(np.float32).astype(np.float64)


def as_f64(a) -> np.ndarray:
    """Accept bf16 bits (uint16) or any float array; return float64."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return bf16_to_f64(a)
    return a.astype(np.float64)


# ----------------------------------------------------------------------------
# activations (section 1.2: SDD -> activation -> DSD)
# ----------------------------------------------------------------------------

def gelu(x):
    """x * Phi(x), Phi the standard normal CDF (exact erf form)."""
    return x * 0.5 * (1.0 + _erf(x * SQRT1_2))


def gelu_grad(x):
    """d/dx [x Phi(x)] = Phi(x) + x phi(x)."""
    return 0.5 * (1.0 + _erf(x * SQRT1_2)) + x * INV_SQRT_2PI * np.exp(-0.5 * x * x)


def sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def silu(x):
    return x * sigmoid(x)


def silu_grad(x):
    s = sigmoid(x)
    return s * (1.0 + x * (1.0 - s))


# ----------------------------------------------------------------------------
# a1: router (section 1.1: a gate network assigns each token to experts)
# ----------------------------------------------------------------------------

def softmax_rows(logits) -> np.ndarray:
    z = as_f64(logits)
    z = z - z.max(axis=1, keepdims=True)
    ez = np.exp(z)
    return ez / ez.sum(axis=1, keepdims=True)


def route_topk(logits, k: int, renormalize: bool):
    """Top-k routing.

    Returns ``expert_idx`` (int32 [T, k], best first) and ``gate_w``
    (float64 [T, k]).  The choice is made on the fp32 logits: larger logit
    first, equal logits by lower expert id.
    """
    logits = np.asarray(logits, dtype=np.float32)
    T, E = logits.shape
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    p = softmax_rows(logits)
    ids = np.broadcast_to(np.arange(E), (T, E))
    # lexsort: last key is the primary key -> by -logit, then by expert id
    order = np.lexsort((ids, -logits), axis=1)
    expert_idx = order[:, :k].astype(np.int32)
    gate_w = np.take_along_axis(p, expert_idx.astype(np.int64), axis=1)
    if renormalize:
        gate_w = gate_w / gate_w.sum(axis=1, keepdims=True)
    return expert_idx, gate_w


def route_topk_backward(logits, expert_idx, d_gate, renormalize: bool):
    """Gradient of the gate weights of ``route_topk`` with respect to the logits.

    The chosen set is piecewise constant in the logits, so only the weights
    carry gradient.  Chain rule through the definitions, token by token:
    w_j = p[s_j] (or p[s_j] / sum_i p[s_i] with renormalisation), p the fp64
    softmax; d logits[e] = sum_j d_gate[j] * d w_j / d logits[e], with the
    Jacobian of the softmax d p_a / d z_e = p_a (delta_ae - p_e).
    Returns float64 [T, E].
    """
    logits = np.asarray(logits, dtype=np.float32)
    T, E = logits.shape
    ei = np.asarray(expert_idx, dtype=np.int64)
    k = ei.shape[1]
    g = np.asarray(d_gate, dtype=np.float64).reshape(T, k)
    p = softmax_rows(logits)
    out = np.zeros((T, E))
    for t in range(T):
        jac_p = np.diag(p[t]) - np.outer(p[t], p[t])  # d p_a / d z_e
        sel = ei[t]
        dp_sel = jac_p[sel]                            # [k, E]
        if renormalize:
            z = p[t, sel].sum()
            dz = dp_sel.sum(axis=0)                    # d Z / d z_e
            jac_w = dp_sel / z - np.outer(p[t, sel], dz) / (z * z)
        else:
            jac_w = dp_sel
        out[t] = g[t] @ jac_w
    return out


def gate_logits(x, w_gate):
    """Router logits of a linear gate network (section 1.1: a gate network
    assigns each token to experts): logits[t, e] = <x[t, :], w_gate[e, :]>,
    with one d-vector per expert in the rows of ``w_gate`` [E, d].  fp64 from
    the bf16 inputs; the routing decision is then route_topk on the fp32
    logits the GPU produced (the same values for both sides)."""
    return as_f64(x) @ as_f64(w_gate).T


# ----------------------------------------------------------------------------
# a2: permute + pad (sections 1.3 "block size" and 1.4)
# ----------------------------------------------------------------------------

def permute_pad(expert_idx, E: int, x=None, block: int = BLOCK):
    """Group assignments by expert and pad every group to a multiple of the
    block size (128, the page's choice; 64 and 256 for its ablation).

    Assignment a = t*k + j carries token t to expert expert_idx[t, j].
    Returns a dict with
      tokens_per_expert int64 [E]      T_e
      padded_offsets    int64 [E+1]    exclusive scan of ceil(T_e/B)*B
      P                 int            padded_offsets[E]
      dest_row          int64 [A]      row of assignment a in expert order
      src_of_row        int64 [P]      assignment held by each row, -1 = pad
      x_perm            float64 [P, d] (when x is given) permuted rows, pads 0
    """
    ei = np.asarray(expert_idx, dtype=np.int64)
    T, k = ei.shape
    flat = ei.reshape(-1)
    A = flat.size
    if A and (flat.min() < 0 or flat.max() >= E):
        raise ValueError("expert id out of range")
    tokens_per_expert = np.zeros(E, dtype=np.int64)
    for e in flat:
        tokens_per_expert[e] += 1
    padded = -(-tokens_per_expert // block) * block
    padded_offsets = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        padded_offsets[e + 1] = padded_offsets[e] + padded[e]
    P = int(padded_offsets[E])

    dest_row = np.full(A, -1, dtype=np.int64)
    src_of_row = np.full(P, -1, dtype=np.int64)
    for e in range(E):
        members = np.nonzero(flat == e)[0]  # ascending assignment index
        rows = padded_offsets[e] + np.arange(members.size)
        dest_row[members] = rows
        src_of_row[rows] = members
    out = dict(tokens_per_expert=tokens_per_expert, padded_offsets=padded_offsets,
               P=P, dest_row=dest_row, src_of_row=src_of_row)
    if x is not None:
        xf = as_f64(x)
        x_perm = np.zeros((P, xf.shape[1]), dtype=np.float64)
        for p in range(P):
            a = src_of_row[p]
            if a >= 0:
                x_perm[p] = xf[a // k]
        out["x_perm"] = x_perm
    return out


# ----------------------------------------------------------------------------
# a3: hybrid BCSR-COO topology + transpose index (section 1.3)
# ----------------------------------------------------------------------------

def build_topology(padded_offsets, F: int, tokens_per_expert=None, block: int = BLOCK):
    """Block topology of the sparse [P x E*F] matrix of all experts.

    Row block r belongs to the expert whose padded group contains rows
    r*128 .. r*128+127; it holds that expert's F/128 column blocks.
    BCSR: row_offsets [P/128+1], column_indices [nnz]; COO view:
    row_indices [nnz].  Transpose index: the nonzero blocks re-listed by
    (column, row) ascending -- column_offsets_t [E*F/128+1],
    row_indices_t [nnz], and block_offsets_t [nnz] = BCSR position of each.
    With ``tokens_per_expert``: row_fill [P/128], the rows of each row block
    that hold tokens (the rest of a block is padding, section 1.3), counted
    by walking the expert's tokens through its blocks.
    """
    B = int(block)
    po = np.asarray(padded_offsets, dtype=np.int64)
    E = po.size - 1
    if F % B:
        raise ValueError("F must be a multiple of the block size")
    nb = F // B
    R = int(po[E]) // B

    row_offsets = [0]
    column_indices = []
    row_indices = []
    for r in range(R):
        e = None
        for ee in range(E):
            if po[ee] <= r * B < po[ee + 1]:
                e = ee
                break
        for j in range(nb):
            column_indices.append(e * nb + j)
            row_indices.append(r)
        row_offsets.append(len(column_indices))
    nnz = len(column_indices)

    # transposed view: every block as (column, row, position), sorted
    entries = sorted((column_indices[q], row_indices[q], q) for q in range(nnz))
    ncols = E * nb
    column_offsets_t = np.zeros(ncols + 1, dtype=np.int64)
    for c, _, _ in entries:
        column_offsets_t[c + 1] += 1
    column_offsets_t = np.cumsum(column_offsets_t)
    out_fill = {}
    if tokens_per_expert is not None:
        tpe = np.asarray(tokens_per_expert, dtype=np.int64)
        fill = np.zeros(R, dtype=np.int64)
        for e in range(E):
            left = int(tpe[e])
            for r in range(int(po[e]) // B, int(po[e + 1]) // B):
                fill[r] = min(B, left)
                left -= fill[r]
            assert left == 0, "tokens_per_expert does not fit the padded offsets"
        out_fill["row_fill"] = fill
    return dict(
        nnz=nnz, R=R, nb=nb, E=E, F=F, block=B, **out_fill,
        row_offsets=np.asarray(row_offsets, dtype=np.int64),
        column_indices=np.asarray(column_indices, dtype=np.int64),
        row_indices=np.asarray(row_indices, dtype=np.int64),
        column_offsets_t=column_offsets_t.astype(np.int64),
        row_indices_t=np.asarray([r for _, r, _ in entries], dtype=np.int64),
        block_offsets_t=np.asarray([q for _, _, q in entries], dtype=np.int64),
    )


def _rows(r, B=BLOCK):
    return slice(r * B, (r + 1) * B)


# ----------------------------------------------------------------------------
# a4/a8: SDD -- sampled dense x dense -> block-sparse (section 1.2)
# ----------------------------------------------------------------------------

def sdd(Xd, W, topo, b_trans: bool = False):
    """blocks[q] = Xd[rows of r] @ Wn[:, cols of c] for each nonzero (r, c).

    ``W`` is [K, E*F] (b_trans False) or [E*F, K] (b_trans True, used as its
    transpose).  Returns float64 [nnz, B, B] (B = the topology's block size).
    """
    B = topo.get("block", BLOCK)
    X = as_f64(Xd)
    Wf = as_f64(W)
    Wn = Wf.T if b_trans else Wf
    out = np.zeros((topo["nnz"], B, B))
    for q in range(topo["nnz"]):
        r = topo["row_indices"][q]
        c = topo["column_indices"][q]
        out[q] = X[_rows(r, B)] @ Wn[:, _rows(c, B)]
    return out


# ----------------------------------------------------------------------------
# a5/a10: DSD -- block-sparse x dense -> dense (section 1.2, 1.3 "BCSR")
# ----------------------------------------------------------------------------

def dsd(blocks, W, topo, P: int, w_trans: bool = False, blocks2=None, W2=None):
    """C[P, N] = S @ Wn (+ S2 @ Wn2), S given by its nonzero blocks.

    Walks each row block's nonzero blocks in BCSR order.  ``W`` is
    [E*F, N]; with ``w_trans`` it is [N, E*F] and used transposed (this is
    DSD with the transposed dense operand, the backward data gradient
    through layer 1).
    """
    B = topo.get("block", BLOCK)
    S = as_f64(blocks)
    Wf = as_f64(W)
    Wn = Wf.T if w_trans else Wf
    C = np.zeros((P, Wn.shape[1]))
    ro = topo["row_offsets"]
    for r in range(topo["R"]):
        for q in range(ro[r], ro[r + 1]):
            c = topo["column_indices"][q]
            C[_rows(r, B)] += S[q] @ Wn[_rows(c, B)]
    if blocks2 is not None:
        C += dsd(blocks2, W2, topo, P, w_trans=w_trans)
    return C


# ----------------------------------------------------------------------------
# a9: DSTD -- (block-sparse)^T x dense -> dense, via the transpose index
# ----------------------------------------------------------------------------

def dstd(blocks, D, topo, c_trans: bool = False):
    """C = S^T @ D, S [P, E*F] given by blocks, D [P, N].

    Walks the transpose index: column block c of S (row block c of S^T)
    visits blocks block_offsets_t[column_offsets_t[c] : column_offsets_t[c+1]].
    Returns [E*F, N], or its transpose [N, E*F] when ``c_trans``.
    """
    B = topo.get("block", BLOCK)
    S = as_f64(blocks)
    Df = as_f64(D)
    ncols = topo["E"] * topo["nb"]
    C = np.zeros((ncols * B, Df.shape[1]))
    cot = topo["column_offsets_t"]
    for c in range(ncols):
        for j in range(cot[c], cot[c + 1]):
            q = topo["block_offsets_t"][j]
            r = topo["row_indices_t"][j]
            C[_rows(c, B)] += S[q].T @ Df[_rows(r, B)]
    return C.T.copy() if c_trans else C


# ----------------------------------------------------------------------------
# a6/a7/a11: un-permute + top-k weighted combine, and its backward
# ----------------------------------------------------------------------------

def unpermute_combine(y_perm, dest_row, gate_w, T: int, k: int):
    """y[t] = sum_j w[t, j] * y_perm[dest_row[t*k + j]] (w = 1 when None)."""
    Y = as_f64(y_perm)
    y = np.zeros((T, Y.shape[1]))
    for t in range(T):
        for j in range(k):
            a = t * k + j
            w = 1.0 if gate_w is None else float(np.asarray(gate_w).reshape(-1)[a])
            y[t] += w * Y[dest_row[a]]
    return y


def combine_backward(dy, y_perm, src_of_row, gate_w, k: int):
    """Gradient of unpermute_combine.

    dy_perm[p] = w[a] * dy[a // k] for the row holding assignment a,
    0 for pad rows; d_gate[a] = <dy[a // k], y_perm[p]>.
    """
    dyf = as_f64(dy)
    Y = as_f64(y_perm)
    src = np.asarray(src_of_row)
    P = src.size
    T = dyf.shape[0]
    w = np.asarray(gate_w, dtype=np.float64).reshape(-1)
    dy_perm = np.zeros((P, dyf.shape[1]))
    d_gate = np.zeros(T * k)
    for p in range(P):
        a = src[p]
        if a < 0:
            continue
        t = a // k
        dy_perm[p] = w[a] * dyf[t]
        d_gate[a] = float(dyf[t] @ Y[p])
    return dy_perm, d_gate.reshape(T, k)


# ----------------------------------------------------------------------------
# the whole layer as the block-sparse chain (sections 1.2 - 1.4)
# ----------------------------------------------------------------------------

def layer_blocksparse(x, logits, w1, w2, dy, k: int, act: str, renormalize: bool, w3=None,
                      backward: bool = True, block: int = BLOCK):
    """Route -> permute/pad -> topology -> SDD -> act -> DSD -> combine, and back.

    Every intermediate of the GPU chain is returned (float64), so single
    steps can be compared as well as the final outputs.  ``block``: the
    block size of the format (section 1.3 compares 64, 128 and 256).
    """
    logits = np.asarray(logits, dtype=np.float32)
    T, E = logits.shape
    W1 = as_f64(w1)
    W2 = as_f64(w2)
    F = W1.shape[1] // E
    expert_idx, gate_w = route_topk(logits, k, renormalize)
    pp = permute_pad(expert_idx, E, x, block=block)
    topo = build_topology(pp["padded_offsets"], F, pp["tokens_per_expert"], block=block)
    P = pp["P"]
    out = dict(expert_idx=expert_idx, gate_w=gate_w, topo=topo, **pp)

    Xp = pp["x_perm"]
    if act == "gelu":
        H = sdd(Xp, W1, topo)
        A = gelu(H)
        out.update(H=H, A=A)
    elif act == "swiglu":
        W3 = as_f64(w3)
        H1 = sdd(Xp, W1, topo)
        H3 = sdd(Xp, W3, topo)
        A = silu(H1) * H3
        out.update(H1=H1, H3=H3, A=A)
    else:
        raise ValueError(act)
    y_perm = dsd(A, W2, topo, P)
    y = unpermute_combine(y_perm, pp["dest_row"], gate_w, T, k)
    out.update(y_perm=y_perm, y=y)
    if not backward:
        return out

    dy_perm, d_gate = combine_backward(dy, y_perm, pp["src_of_row"], gate_w, k)
    dA = sdd(dy_perm, W2, topo, b_trans=True)
    dW2 = dstd(A, dy_perm, topo)
    if act == "gelu":
        dH = dA * gelu_grad(out["H"])
        dx_perm = dsd(dH, W1, topo, P, w_trans=True)
        dW1 = dstd(dH, Xp, topo, c_trans=True)
        out.update(dH=dH)
    else:
        H1, H3 = out["H1"], out["H3"]
        dH1 = dA * H3 * silu_grad(H1)
        dH3 = dA * silu(H1)
        dx_perm = dsd(dH1, W1, topo, P, w_trans=True, blocks2=dH3, W2=W3)
        dW1 = dstd(dH1, Xp, topo, c_trans=True)
        out["dW3"] = dstd(dH3, Xp, topo, c_trans=True)
        out.update(dH1=dH1, dH3=dH3)
    dx = unpermute_combine(dx_perm, pp["dest_row"], None, T, k)
    out.update(dy_perm=dy_perm, d_gate=d_gate, dA=dA, dW2=dW2, dW1=dW1, dx_perm=dx_perm, dx=dx,
               d_logits=route_topk_backward(logits, expert_idx, d_gate, renormalize))
    return out


# ----------------------------------------------------------------------------
# the whole layer as E separate dense expert MLPs (section 1.2, the batched
# per-expert formulation the block-sparse product replaces)
# ----------------------------------------------------------------------------

def _expert_members(expert_idx, e):
    """(token, slot) pairs routed to expert e, in ascending assignment order."""
    ei = np.asarray(expert_idx)
    T, k = ei.shape
    a = np.nonzero(ei.reshape(-1) == e)[0]
    return a // k, a % k


def layer_per_expert(x, logits, w1, w2, dy, k: int, act: str, renormalize: bool, w3=None,
                     backward: bool = True, keep_weight_grads: bool = True):
    """Dense per-expert reference: for each expert, its own two-layer MLP.

    Each expert's weight slices are decoded to float64 when that expert is
    reached, so host memory holds one expert's weights at a time.  With
    ``keep_weight_grads=False`` every expert's dW1 / dW2 (/ dW3) is still
    computed, then dropped instead of stored (a full-size layer's weight
    gradients in float64 can exceed host memory); the other results are
    unchanged.
    """
    logits = np.asarray(logits, dtype=np.float32)
    T, E = logits.shape
    X = as_f64(x)
    w1 = np.asarray(w1)
    w2 = np.asarray(w2)
    w3 = np.asarray(w3) if act == "swiglu" else None
    d = X.shape[1]
    F = w1.shape[1] // E
    dyf = as_f64(dy) if backward else None
    expert_idx, gate_w = route_topk(logits, k, renormalize)
    y = np.zeros((T, d))
    dx = np.zeros((T, d))
    d_gate = np.zeros((T, k))
    keep = backward and keep_weight_grads
    dW1 = np.zeros((d, E * F)) if keep else None
    dW2 = np.zeros((E * F, d)) if keep else None
    dW3 = np.zeros((d, E * F)) if keep and act == "swiglu" else None
    for e in range(E):
        tok, slot = _expert_members(expert_idx, e)
        if tok.size == 0:
            continue
        cols = slice(e * F, (e + 1) * F)
        W1e = as_f64(w1[:, cols])
        W2e = as_f64(w2[cols])
        Xe = X[tok]
        w = gate_w[tok, slot][:, None]
        if act == "gelu":
            He = Xe @ W1e
            Ae = gelu(He)
        else:
            W3e = as_f64(w3[:, cols])
            H1 = Xe @ W1e
            H3 = Xe @ W3e
            Ae = silu(H1) * H3
        Ye = Ae @ W2e
        np.add.at(y, tok, w * Ye)
        if not backward:
            continue
        dYe = w * dyf[tok]
        d_gate[tok, slot] = np.einsum("ij,ij->i", dyf[tok], Ye)
        dAe = dYe @ W2e.T
        dW2e = Ae.T @ dYe
        if act == "gelu":
            dHe = dAe * gelu_grad(He)
            dW1e = Xe.T @ dHe
            dXe = dHe @ W1e.T
        else:
            dH1 = dAe * H3 * silu_grad(H1)
            dH3 = dAe * silu(H1)
            dW1e = Xe.T @ dH1
            dW3e = Xe.T @ dH3
            dXe = dH1 @ W1e.T + dH3 @ W3e.T
        if keep:
            dW2[cols] = dW2e
            dW1[:, cols] = dW1e
            if act == "swiglu":
                dW3[:, cols] = dW3e
        np.add.at(dx, tok, dXe)
    out = dict(expert_idx=expert_idx, gate_w=gate_w, y=y)
    if backward:
        out.update(dx=dx, d_gate=d_gate,
                   d_logits=route_topk_backward(logits, expert_idx, d_gate, renormalize))
        if keep:
            out.update(dW1=dW1, dW2=dW2)
            if act == "swiglu":
                out["dW3"] = dW3
    return out


def layer_deep_per_expert(x, logits, w1s, w2s, dy, k: int, act: str, renormalize: bool, w3s=None):
    """Deeper experts (section 1.2: with more expert layers the pattern
    continues SDD -> DSD -> SDD -> DSD ...): each expert is a stack of L
    two-layer blocks applied to its tokens in turn,

        h_0 = x,   h_l = act(h_{l-1} W1_l) W2_l   (l = 1..L),

    with the activation between each SDD and its DSD only (the page names
    no other), and the gated combine on h_L.  ``w1s`` / ``w2s`` (/ ``w3s``)
    are lists of L weights in the one-block layouts ([d, E*F] / [E*F, d]).
    Dense per-expert loops; the backward is the chain rule through the
    blocks in reverse.  Returns y, dx, d_gate, d_logits and the lists dW1s,
    dW2s (, dW3s)."""
    logits = np.asarray(logits, dtype=np.float32)
    T, E = logits.shape
    L = len(w1s)
    X = as_f64(x)
    W1 = [as_f64(w) for w in w1s]
    W2 = [as_f64(w) for w in w2s]
    W3 = [as_f64(w) for w in w3s] if act == "swiglu" else None
    d = X.shape[1]
    F = W1[0].shape[1] // E
    dyf = as_f64(dy)
    expert_idx, gate_w = route_topk(logits, k, renormalize)
    y = np.zeros((T, d))
    dx = np.zeros((T, d))
    d_gate = np.zeros((T, k))
    dW1 = [np.zeros_like(w) for w in W1]
    dW2 = [np.zeros_like(w) for w in W2]
    dW3 = [np.zeros_like(w) for w in W1] if act == "swiglu" else None
    for e in range(E):
        tok, slot = _expert_members(expert_idx, e)
        if tok.size == 0:
            continue
        cols = slice(e * F, (e + 1) * F)
        w = gate_w[tok, slot][:, None]
        hs = [X[tok]]  # h_0 .. h_L of this expert's tokens
        saved = []
        for l in range(L):
            if act == "gelu":
                Hl = hs[-1] @ W1[l][:, cols]
                Al = gelu(Hl)
                saved.append((Hl, Al))
            else:
                H1 = hs[-1] @ W1[l][:, cols]
                H3 = hs[-1] @ W3[l][:, cols]
                Al = silu(H1) * H3
                saved.append((H1, H3, Al))
            hs.append(Al @ W2[l][cols])
        np.add.at(y, tok, w * hs[-1])
        d_gate[tok, slot] = np.einsum("ij,ij->i", dyf[tok], hs[-1])
        g = w * dyf[tok]  # gradient w.r.t. h_L
        for l in reversed(range(L)):
            Al = saved[l][-1]
            dW2[l][cols] = Al.T @ g
            dA = g @ W2[l][cols].T
            if act == "gelu":
                dH = dA * gelu_grad(saved[l][0])
                dW1[l][:, cols] = hs[l].T @ dH
                g = dH @ W1[l][:, cols].T
            else:
                H1, H3, _ = saved[l]
                dH1 = dA * H3 * silu_grad(H1)
                dH3 = dA * silu(H1)
                dW1[l][:, cols] = hs[l].T @ dH1
                dW3[l][:, cols] = hs[l].T @ dH3
                g = dH1 @ W1[l][:, cols].T + dH3 @ W3[l][:, cols].T
        np.add.at(dx, tok, g)
    out = dict(expert_idx=expert_idx, gate_w=gate_w, y=y, dx=dx, d_gate=d_gate, dW1s=dW1, dW2s=dW2,
               d_logits=route_topk_backward(logits, expert_idx, d_gate, renormalize))
    if act == "swiglu":
        out["dW3s"] = dW3
    return out


# ----------------------------------------------------------------------------
# sampled forms for workloads too large to run whole on the CPU
# ----------------------------------------------------------------------------

def layer_rows(x, expert_idx, gate_w, w1, w2, dy, tokens, F: int, act: str, w3=None):
    """y, dx and d_gate rows of the given tokens only (rows are independent).

    ``expert_idx`` / ``gate_w`` come from ``route_topk``; ``F`` is the hidden
    width of one expert.  Weight slices are decoded one expert at a time.
    """
    tokens = np.asarray(tokens, dtype=np.int64)
    ei = np.asarray(expert_idx)[tokens]
    gw = np.asarray(gate_w, dtype=np.float64)[tokens]
    X = as_f64(np.asarray(x)[tokens])
    dyf = as_f64(np.asarray(dy)[tokens])
    n, k = ei.shape
    d = X.shape[1]
    y = np.zeros((n, d))
    dx = np.zeros((n, d))
    d_gate = np.zeros((n, k))
    for e in sorted(set(int(v) for v in ei.reshape(-1))):
        cols = slice(e * F, (e + 1) * F)
        W1e = as_f64(np.asarray(w1)[:, cols])
        W2e = as_f64(np.asarray(w2)[cols])
        W3e = as_f64(np.asarray(w3)[:, cols]) if act == "swiglu" else None
        i, j = np.nonzero(ei == e)
        Xe = X[i]
        w = gw[i, j][:, None]
        if act == "gelu":
            He = Xe @ W1e
            Ae = gelu(He)
        else:
            H1 = Xe @ W1e
            H3 = Xe @ W3e
            Ae = silu(H1) * H3
        Ye = Ae @ W2e
        np.add.at(y, i, w * Ye)
        dYe = w * dyf[i]
        d_gate[i, j] = np.einsum("ij,ij->i", dyf[i], Ye)
        dAe = dYe @ W2e.T
        if act == "gelu":
            dXe = (dAe * gelu_grad(He)) @ W1e.T
        else:
            dXe = (dAe * H3 * silu_grad(H1)) @ W1e.T + (dAe * silu(H1)) @ W3e.T
        np.add.at(dx, i, dXe)
    return dict(y=y, dx=dx, d_gate=d_gate)


def weight_grad_columns(x, expert_idx, gate_w, w1, w2, dy, e: int, cols, F: int, act: str, w3=None):
    """Selected hidden units of expert e: dW1[:, e*F+f], dW3[:, e*F+f], dW2[e*F+f, :].

    A hidden unit f of expert e depends only on column f of W1 / W3 and row f
    of W2, so each is computed exactly from all tokens routed to e.
    """
    cols = np.asarray(cols, dtype=np.int64)
    g = e * F + cols
    tok, slot = _expert_members(expert_idx, e)
    X = as_f64(np.asarray(x)[tok])
    w = np.asarray(gate_w, dtype=np.float64)[tok, slot][:, None]
    dYe = w * as_f64(np.asarray(dy)[tok])
    W1c = as_f64(np.asarray(w1)[:, g])
    W2r = as_f64(np.asarray(w2)[g])
    dA = dYe @ W2r.T
    out = {}
    if act == "gelu":
        H = X @ W1c
        A = gelu(H)
        out["dW1"] = X.T @ (dA * gelu_grad(H))
    else:
        W3c = as_f64(np.asarray(w3)[:, g])
        H1 = X @ W1c
        H3 = X @ W3c
        A = silu(H1) * H3
        out["dW1"] = X.T @ (dA * H3 * silu_grad(H1))
        out["dW3"] = X.T @ (dA * silu(H1))
    out["dW2"] = A.T @ dYe
    return out
