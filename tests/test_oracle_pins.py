"""Pins of the fp64 oracle against facts fixed by the page and by mathematics.

None of these tests compares the oracle with itself.  Each one checks it
against a hand-worked example (tests/golden), a closed form, an invariant, a
special case that reduces to a library routine, or brute force on a tiny
input -- chosen so that a dropped term, a wrong index or a transposed operand
fails at least one of them.  Source: George Lin's blog post on MoE training,
section 1 (MegaBlocks).
"""

import itertools
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import dmoe_synth as syn
import oracle as O

B = 128


def _bits(a):
    return syn.f32_to_bf16_bits(np.asarray(a, dtype=np.float32))


# ----------------------------------------------------------------------------
# activations: library routines and closed forms
# ----------------------------------------------------------------------------

def test_gelu_matches_torch_and_closed_forms():
    x = np.linspace(-8, 8, 2001)
    ref = torch.nn.functional.gelu(torch.from_numpy(x), approximate="none").numpy()
    assert np.max(np.abs(O.gelu(x) - ref)) < 1e-14
    assert O.gelu(np.array(0.0)) == 0.0
    # Phi(1) = 0.8413447460685429 (standard normal table)
    assert abs(O.gelu(np.array(1.0)) - 0.8413447460685429) < 1e-15
    assert abs(O.gelu(np.array(30.0)) - 30.0) < 1e-12
    assert abs(O.gelu(np.array(-30.0))) < 1e-12


def test_activation_gradients_match_autograd():
    x = torch.linspace(-6, 6, 1001, dtype=torch.float64, requires_grad=True)
    g, = torch.autograd.grad(torch.nn.functional.gelu(x).sum(), x)
    assert np.max(np.abs(O.gelu_grad(x.detach().numpy()) - g.numpy())) < 1e-13
    s, = torch.autograd.grad(torch.nn.functional.silu(x).sum(), x)
    assert np.max(np.abs(O.silu_grad(x.detach().numpy()) - s.numpy())) < 1e-13
    ref = torch.nn.functional.silu(x).detach().numpy()
    assert np.max(np.abs(O.silu(x.detach().numpy()) - ref)) < 1e-13


def test_bf16_decode_matches_torch():
    bits = np.arange(0, 65536, 7, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    got = O.bf16_to_f64(bits)
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.array_equal(got[~both_nan], ref[~both_nan])


# ----------------------------------------------------------------------------
# a1 routing
# ----------------------------------------------------------------------------

def test_route_hand_example(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "hand_route.json")))
    logits = np.array(g["logits"], dtype=np.float32)
    for c in g["cases"]:
        ei, w = O.route_topk(logits, c["k"], c["renormalize"])
        assert ei.tolist() == c["expert_idx"]
        assert np.allclose(w, c["gate_w"], rtol=1e-14, atol=0)


def test_gate_hand_example(golden_dir):
    """Linear gate then router on a hand-worked integer case (exact logits,
    a tie resolved to the lower expert id)."""
    g = json.load(open(os.path.join(golden_dir, "hand_gate.json")))
    x = syn.f32_to_bf16_bits(np.array(g["x"], dtype=np.float32))
    w = syn.f32_to_bf16_bits(np.array(g["w_gate"], dtype=np.float32))
    logits = O.gate_logits(x, w)
    assert np.array_equal(logits, np.array(g["logits"]))
    for c in g["cases"]:
        ei, gw = O.route_topk(logits.astype(np.float32), c["k"], c["renormalize"])
        assert ei.tolist() == c["expert_idx"]
        assert np.allclose(gw, c["gate_w"], rtol=1e-14, atol=0)


def test_gate_one_hot_rows_select_columns():
    """A gate row that is the unit vector of dimension j gives that expert
    the token's j-th feature, exactly."""
    T, d, E = 50, 24, 7
    x = syn.normal_bf16(21, 1, (T, d))
    cols = np.array([3, 0, 23, 3, 11, 5, 17])
    wf = np.zeros((E, d), dtype=np.float32)
    wf[np.arange(E), cols] = 1.0
    logits = O.gate_logits(x, syn.f32_to_bf16_bits(wf))
    assert np.array_equal(logits, O.bf16_to_f64(x)[:, cols])


def test_gate_matches_torch_linear():
    """A linear layer without bias, as the library computes it."""
    T, d, E = 40, 96, 12
    x = syn.normal_bf16(22, 1, (T, d))
    w = syn.normal_bf16(22, 2, (E, d), 0.1)
    ref = torch.nn.functional.linear(torch.from_numpy(O.bf16_to_f64(x)), torch.from_numpy(O.bf16_to_f64(w)))
    assert np.allclose(O.gate_logits(x, w), ref.numpy(), rtol=1e-13, atol=1e-13)


def test_route_softmax_matches_scipy():
    logits = syn.normal_f32(3, 1, (64, 37), 3.0)
    p = O.softmax_rows(logits)
    ref = scipy.special.softmax(logits.astype(np.float64), axis=1)
    assert np.max(np.abs(p - ref)) < 1e-15


def test_route_brute_force_with_ties():
    # integer logits force many ties; brute force with a python sort
    z = syn.integers(5, 1, -2, 3, (200, 9)).astype(np.float32)
    for k in (1, 2, 3, 9):
        for renorm in (False, True):
            ei, w = O.route_topk(z, k, renorm)
            for t in range(z.shape[0]):
                want = sorted(range(9), key=lambda e: (-z[t, e], e))[:k]
                assert ei[t].tolist() == want
                ex = np.exp(z[t].astype(np.float64) - z[t].max())
                p = ex / ex.sum()
                ww = p[want] / (p[want].sum() if renorm else 1.0)
                assert np.allclose(w[t], ww, rtol=1e-13, atol=0)


def test_route_renorm_invariants():
    z = syn.normal_f32(11, 1, (300, 16))
    _, w = O.route_topk(z, 16, True)
    assert np.allclose(w.sum(1), 1.0, atol=1e-14)
    _, w1 = O.route_topk(z, 1, True)
    assert np.all(w1 == 1.0)
    _, wall = O.route_topk(z, 16, False)
    assert np.allclose(wall.sum(1), 1.0, atol=1e-14)  # all experts = whole softmax
    assert np.all(np.diff(wall, axis=1) <= 0)  # best first


# ----------------------------------------------------------------------------
# a2 permute + pad
# ----------------------------------------------------------------------------

def _hand_topo(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "hand_permute_topology.json")))
    ei = np.zeros((g["T"], 1), dtype=np.int32)
    ei[7, 0] = 1
    return g, ei


def test_permute_hand_example(golden_dir):
    g, ei = _hand_topo(golden_dir)
    pp = O.permute_pad(ei, g["E"])
    assert pp["tokens_per_expert"].tolist() == g["tokens_per_expert"]
    assert pp["padded_offsets"].tolist() == g["padded_offsets"]
    assert pp["P"] == g["P"]
    want_dest = [t if t < 7 else (256 if t == 7 else t - 1) for t in range(g["T"])]
    assert pp["dest_row"].tolist() == want_dest
    want_src = [-1] * g["P"]
    for r in range(7):
        want_src[r] = r
    for r in range(7, 129):
        want_src[r] = r + 1
    want_src[256] = 7
    assert pp["src_of_row"].tolist() == want_src


@pytest.mark.parametrize("T,k,E", [(1, 1, 1), (37, 2, 5), (300, 3, 4), (129, 1, 3), (256, 2, 2)])
def test_permute_invariants(T, k, E):
    ei = syn.integers(T * 31 + E, 2, 0, E, (T, k)).astype(np.int32)
    d = 16
    x = _bits(syn.normal_f32(T, 3, (T, d)))
    pp = O.permute_pad(ei, E, x)
    counts = np.bincount(ei.reshape(-1), minlength=E)
    assert pp["tokens_per_expert"].tolist() == counts.tolist()
    pad = (-(-counts // B)) * B
    assert pp["P"] == pad.sum()
    assert pp["padded_offsets"].tolist() == [0] + np.cumsum(pad).tolist()
    dest = pp["dest_row"]
    # dropless: every assignment has a row, rows are distinct
    assert np.all(dest >= 0) and len(set(dest.tolist())) == T * k
    # each token appears exactly k times among the rows
    src = pp["src_of_row"]
    toks = src[src >= 0] // k
    assert np.bincount(toks, minlength=T).tolist() == [k] * T
    # rows hold the right token, in ascending assignment order per expert
    xf = O.bf16_to_f64(x)
    for a in range(T * k):
        e = ei.reshape(-1)[a]
        assert pp["padded_offsets"][e] <= dest[a] < pp["padded_offsets"][e] + counts[e]
        assert src[dest[a]] == a
        assert np.array_equal(pp["x_perm"][dest[a]], xf[a // k])
    for e in range(E):
        rows = src[pp["padded_offsets"][e]:pp["padded_offsets"][e] + counts[e]]
        assert np.all(np.diff(rows) > 0)
        n_pad = pad[e] - counts[e]
        assert 0 <= n_pad <= B - 1
        pad_rows = slice(pp["padded_offsets"][e] + counts[e], pp["padded_offsets"][e + 1])
        assert np.all(src[pad_rows] == -1)
        assert np.all(pp["x_perm"][pad_rows] == 0.0)


def test_permute_edge_cases():
    # all tokens on one expert; exactly 128; 129; empty experts
    for counts in ([0, 128, 0], [129, 0, 0], [0, 0, 1], [128, 128, 0], [0, 0, 0, 255]):
        ei = np.repeat(np.arange(len(counts)), counts).astype(np.int32)[:, None]
        pp = O.permute_pad(ei, len(counts))
        want = [0]
        for c in counts:
            want.append(want[-1] + (-(-c // B)) * B)
        assert pp["padded_offsets"].tolist() == want
        assert pp["dest_row"].tolist() == [
            want[e] + i for e, c in enumerate(counts) for i in range(c)]


def test_permute_rejects_bad_ids():
    with pytest.raises(ValueError):
        O.permute_pad(np.array([[0], [3]], dtype=np.int32), 3)


# ----------------------------------------------------------------------------
# a3 topology
# ----------------------------------------------------------------------------

def test_topology_hand_example(golden_dir):
    g, ei = _hand_topo(golden_dir)
    pp = O.permute_pad(ei, g["E"])
    tp = O.build_topology(pp["padded_offsets"], g["F"])
    assert tp["nnz"] == g["nnz"]
    for key in ("row_offsets", "column_indices", "row_indices", "column_offsets_t",
                "row_indices_t", "block_offsets_t"):
        assert tp[key].tolist() == g[key], key


def _topo_by_dense_mask(padded_offsets, F):
    """Independent construction: a dense block mask enumerated by numpy."""
    po = np.asarray(padded_offsets)
    E = po.size - 1
    nb = F // B
    R = po[-1] // B
    mask = np.zeros((R, E * nb), dtype=bool)
    for e in range(E):
        mask[po[e] // B:po[e + 1] // B, e * nb:(e + 1) * nb] = True
    rr, cc = np.nonzero(mask)  # row-major order = BCSR order
    pos = -np.ones(mask.shape, dtype=np.int64)
    pos[rr, cc] = np.arange(rr.size)
    ct, rt = np.nonzero(mask.T)  # column-major order
    return dict(
        row_offsets=np.concatenate([[0], np.cumsum(mask.sum(1))]),
        column_indices=cc, row_indices=rr,
        column_offsets_t=np.concatenate([[0], np.cumsum(mask.sum(0))]),
        row_indices_t=rt, block_offsets_t=pos[rt, ct], nnz=rr.size)


@pytest.mark.parametrize("counts,F", [
    ([3, 0, 130, 128, 1], 256), ([0, 0, 0, 1], 128), ([500, 7, 256, 0, 0, 300], 384),
    ([1] * 9, 512), ([1000], 128)])
def test_topology_matches_dense_mask_and_closed_forms(counts, F):
    ei = np.repeat(np.arange(len(counts)), counts).astype(np.int32)[:, None]
    pp = O.permute_pad(ei, len(counts))
    tp = O.build_topology(pp["padded_offsets"], F)
    ref = _topo_by_dense_mask(pp["padded_offsets"], F)
    for key, v in ref.items():
        assert np.array_equal(np.asarray(tp[key]), np.asarray(v)), key
    nb = F // B
    # closed form: nnz = sum_i ceil(T_i/128) * F/128
    assert tp["nnz"] == sum(-(-c // B) for c in counts) * nb
    assert np.all(np.diff(tp["row_offsets"]) == nb)
    # COO row index = expansion of the BCSR row offsets
    assert tp["row_indices"].tolist() == [
        r for r in range(tp["R"]) for _ in range(tp["row_offsets"][r], tp["row_offsets"][r + 1])]
    # transpose index is a permutation reproducing column-major order
    bo = tp["block_offsets_t"]
    assert sorted(bo.tolist()) == list(range(tp["nnz"]))
    keys = [(tp["column_indices"][q], tp["row_indices"][q]) for q in bo]
    assert keys == sorted(keys)
    assert np.array_equal(tp["row_indices"][bo], tp["row_indices_t"])
    # row fill: the rows of each block that hold a token, counted from the
    # permutation itself
    tf = O.build_topology(pp["padded_offsets"], F, pp["tokens_per_expert"])
    held = (pp["src_of_row"] >= 0).reshape(-1, B).sum(axis=1) if tp["R"] else np.zeros(0, dtype=np.int64)
    assert np.array_equal(tf["row_fill"], held)
    assert np.all((tf["row_fill"] >= 1) & (tf["row_fill"] <= B))


# ----------------------------------------------------------------------------
# a4/a5/a9/a10 block-sparse products against dense products of the dense
# block-sparse matrix (numpy matmul on the mathematical definition)
# ----------------------------------------------------------------------------

def _small_topo(counts=(5, 0, 140, 128), F=256):
    ei = np.repeat(np.arange(len(counts)), counts).astype(np.int32)[:, None]
    pp = O.permute_pad(ei, len(counts))
    return pp, O.build_topology(pp["padded_offsets"], F)


def _dense_of(blocks, tp, P):
    S = np.zeros((P, tp["E"] * tp["nb"] * B))
    for q in range(tp["nnz"]):
        r, c = tp["row_indices"][q], tp["column_indices"][q]
        S[r * B:(r + 1) * B, c * B:(c + 1) * B] = blocks[q]
    return S


def _mask_of(tp, P):
    return _dense_of(np.ones((tp["nnz"], B, B)), tp, P)


def test_sdd_is_masked_dense_product():
    pp, tp = _small_topo()
    P, K = pp["P"], 64
    rng = np.random.default_rng(0)
    X = rng.standard_normal((P, K))
    W = rng.standard_normal((K, tp["E"] * tp["nb"] * B))
    got = _dense_of(O.sdd(X, W, tp), tp, P)
    assert np.allclose(got, (X @ W) * _mask_of(tp, P), atol=1e-12)
    got_t = _dense_of(O.sdd(X, W.T.copy(), tp, b_trans=True), tp, P)
    assert np.allclose(got_t, (X @ W) * _mask_of(tp, P), atol=1e-12)


def test_dsd_dsdt_dstd_are_dense_products():
    pp, tp = _small_topo()
    P = pp["P"]
    N = 32
    rng = np.random.default_rng(1)
    blocks = rng.standard_normal((tp["nnz"], B, B))
    blocks2 = rng.standard_normal((tp["nnz"], B, B))
    S = _dense_of(blocks, tp, P)
    S2 = _dense_of(blocks2, tp, P)
    EF = S.shape[1]
    W = rng.standard_normal((EF, N))
    Wt = rng.standard_normal((N, EF))
    Wt2 = rng.standard_normal((N, EF))
    D = rng.standard_normal((P, N))
    assert np.allclose(O.dsd(blocks, W, tp, P), S @ W, atol=1e-11)
    assert np.allclose(O.dsd(blocks, Wt, tp, P, w_trans=True), S @ Wt.T, atol=1e-11)
    assert np.allclose(O.dsd(blocks, Wt, tp, P, w_trans=True, blocks2=blocks2, W2=Wt2),
                       S @ Wt.T + S2 @ Wt2.T, atol=1e-11)
    assert np.allclose(O.dstd(blocks, D, tp), S.T @ D, atol=1e-11)
    assert np.allclose(O.dstd(blocks, D, tp, c_trans=True), (S.T @ D).T, atol=1e-11)


# ----------------------------------------------------------------------------
# a6/a7/a11 combine: identities and adjointness
# ----------------------------------------------------------------------------

def test_combine_identity_experts_give_back_x():
    # experts that return their input, weights renormalised -> y == x
    T, k, E, d = 50, 3, 5, 8
    logits = syn.normal_f32(21, 1, (T, E))
    ei, w = O.route_topk(logits, k, True)
    x = syn.normal_f32(21, 2, (T, d)).astype(np.float64)
    pp = O.permute_pad(ei, E, x)
    y = O.unpermute_combine(pp["x_perm"], pp["dest_row"], w, T, k)
    assert np.allclose(y, x, atol=1e-14)
    y1 = O.unpermute_combine(pp["x_perm"], pp["dest_row"], None, T, k)
    assert np.allclose(y1, k * x, atol=1e-13)


def test_combine_backward_is_adjoint():
    T, k, E, d = 40, 2, 4, 6
    ei, w = O.route_topk(syn.normal_f32(22, 1, (T, E)), k, False)
    pp = O.permute_pad(ei, E)
    rng = np.random.default_rng(2)
    Yp = rng.standard_normal((pp["P"], d))
    Yp[pp["src_of_row"] < 0] = 0.0
    dy = rng.standard_normal((T, d))
    dy_perm, d_gate = O.combine_backward(dy, Yp, pp["src_of_row"], w, k)
    y = O.unpermute_combine(Yp, pp["dest_row"], w, T, k)
    # <combine(Yp), dy> == <Yp, dy_perm>
    assert abs(np.sum(y * dy) - np.sum(Yp * dy_perm)) < 1e-11
    # d_gate by finite differences on the weights (linear: exact)
    h = 1e-3
    for a in (0, 5, 17, 79):
        w2 = w.copy().reshape(-1)
        w2[a] += h
        y2 = O.unpermute_combine(Yp, pp["dest_row"], w2.reshape(T, k), T, k)
        assert abs((np.sum(y2 * dy) - np.sum(y * dy)) / h - d_gate.reshape(-1)[a]) < 1e-9
    assert np.all(dy_perm[pp["src_of_row"] < 0] == 0.0)


# ----------------------------------------------------------------------------
# the layer: E=1 dense MLP, per-expert vs block-sparse, capacity form,
# finite differences and autograd
# ----------------------------------------------------------------------------

def _tiny_inputs(T, d, E, F, k, act, seed):
    cfg = syn.custom("t", T, d, E, F, k, act=act, seed=seed)
    return cfg, syn.make_inputs(cfg)


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_single_expert_is_dense_mlp(act):
    cfg, inp = _tiny_inputs(64, 128, 1, 256, 1, act, 31)
    out = O.layer_per_expert(inp["x"], inp["logits"], inp["w1"], inp["w2"], inp["dy"], 1, act,
                             False, w3=inp.get("w3"))
    x = torch.from_numpy(O.bf16_to_f64(inp["x"]))
    W1 = torch.from_numpy(O.bf16_to_f64(inp["w1"]))
    W2 = torch.from_numpy(O.bf16_to_f64(inp["w2"]))
    if act == "gelu":
        h = torch.nn.functional.gelu(x @ W1)
    else:
        W3 = torch.from_numpy(O.bf16_to_f64(inp["w3"]))
        h = torch.nn.functional.silu(x @ W1) * (x @ W3)
    ref = h @ W2  # one expert: gate weight is softmax over 1 expert = 1
    assert np.max(np.abs(out["y"] - ref.numpy())) < 1e-12


@pytest.mark.parametrize("act,k,renorm", [("gelu", 1, False), ("gelu", 2, True), ("swiglu", 2, False),
                                          ("swiglu", 3, True)])
def test_blocksparse_chain_equals_per_expert(act, k, renorm):
    cfg, inp = _tiny_inputs(150, 128, 3, 256, k, act, 40 + k)
    a = O.layer_blocksparse(inp["x"], inp["logits"], inp["w1"], inp["w2"], inp["dy"], k, act, renorm,
                            w3=inp.get("w3"))
    b = O.layer_per_expert(inp["x"], inp["logits"], inp["w1"], inp["w2"], inp["dy"], k, act, renorm,
                           w3=inp.get("w3"))
    for key in ("y", "dx", "d_gate", "dW1", "dW2") + (("dW3",) if act == "swiglu" else ()):
        scale = np.max(np.abs(b[key]))
        assert np.max(np.abs(a[key] - b[key])) <= 1e-12 * max(scale, 1e-300), key
    # pad rows of the permuted input are zero, so they add nothing to dW1
    assert np.all(a["x_perm"][a["src_of_row"] < 0] == 0)


def test_capacity_batched_gemm_form_agrees():
    """Batched per-expert GEMM with a capacity large enough that nothing drops."""
    T, d, E, F, k = 90, 16, 4, 24, 2
    rng = np.random.default_rng(3)
    x = rng.standard_normal((T, d))
    W1 = rng.standard_normal((d, E * F))
    W2 = rng.standard_normal((E * F, d))
    logits = syn.normal_f32(9, 1, (T, E))
    ei, w = O.route_topk(logits, k, False)
    out = O.layer_per_expert(x, logits, W1, W2, np.zeros((T, d)), k, "gelu", False, backward=False)
    cap = int(np.bincount(ei.reshape(-1), minlength=E).max())
    buf = np.zeros((E, cap, d))
    slot_of = {}
    fill = [0] * E
    for t in range(T):
        for j in range(k):
            e = ei[t, j]
            buf[e, fill[e]] = x[t]
            slot_of[(t, j)] = (e, fill[e])
            fill[e] += 1
    W1b = W1.reshape(d, E, F).transpose(1, 0, 2)
    W2b = W2.reshape(E, F, d)
    Yb = np.matmul(O.gelu(np.matmul(buf, W1b)), W2b)
    y = np.zeros((T, d))
    for (t, j), (e, s) in slot_of.items():
        y[t] += w[t, j] * Yb[e, s]
    assert np.max(np.abs(y - out["y"])) < 1e-11


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_backward_by_finite_differences(act):
    T, d, E, F, k = 7, 5, 3, 4, 2
    rng = np.random.default_rng(4)
    x = rng.standard_normal((T, d))
    W1 = rng.standard_normal((d, E * F)) * 0.5
    W3 = rng.standard_normal((d, E * F)) * 0.5
    W2 = rng.standard_normal((E * F, d)) * 0.5
    dy = rng.standard_normal((T, d))
    logits = syn.normal_f32(4, 1, (T, E))
    kw = dict(w3=W3) if act == "swiglu" else {}
    g = O.layer_per_expert(x, logits, W1, W2, dy, k, act, True, **kw)

    def loss(x_, W1_, W2_, W3_):
        kk = dict(w3=W3_) if act == "swiglu" else {}
        return float(np.sum(O.layer_per_expert(x_, logits, W1_, W2_, dy, k, act, True,
                                               backward=False, **kk)["y"] * dy))

    h = 1e-6
    for name, arr, grad in (("x", x, g["dx"]), ("W1", W1, g["dW1"]), ("W2", W2, g["dW2"])) + (
            (("W3", W3, g["dW3"]),) if act == "swiglu" else ()):
        for idx in itertools.islice(np.ndindex(arr.shape), 0, None, 3):
            args = dict(x=x, W1=W1, W2=W2, W3=W3)
            p = arr.copy(); p[idx] += h
            m = arr.copy(); m[idx] -= h
            args[name] = p
            lp = loss(args["x"], args["W1"], args["W2"], args["W3"])
            args[name] = m
            lm = loss(args["x"], args["W1"], args["W2"], args["W3"])
            fd = (lp - lm) / (2 * h)
            assert abs(fd - grad[idx]) < 1e-6 * max(1.0, abs(fd)), (name, idx)
    # d_gate: y is linear in each gate weight
    for t, j in ((0, 0), (3, 1), (6, 0)):
        y = O.layer_per_expert(x, logits, W1, W2, dy, k, act, True, backward=False, **kw)["y"]
        e = g["expert_idx"][t, j]
        Ye = O.layer_per_expert(x[t:t + 1], np.eye(E, dtype=np.float32)[e:e + 1] * 50, W1, W2,
                                dy[t:t + 1], 1, act, True, backward=False, **kw)["y"]
        assert abs(float(dy[t] @ Ye[0]) - g["d_gate"][t, j]) < 1e-10
        del y


def test_backward_matches_autograd_swiglu():
    T, d, E, F, k = 12, 6, 3, 5, 2
    rng = np.random.default_rng(5)
    x = rng.standard_normal((T, d))
    W1 = rng.standard_normal((d, E * F)) * 0.4
    W3 = rng.standard_normal((d, E * F)) * 0.4
    W2 = rng.standard_normal((E * F, d)) * 0.4
    dy = rng.standard_normal((T, d))
    logits = syn.normal_f32(5, 1, (T, E))
    g = O.layer_per_expert(x, logits, W1, W2, dy, k, "swiglu", False, w3=W3)
    tx, t1, t3, t2 = (torch.tensor(a, requires_grad=True) for a in (x, W1, W3, W2))
    tw = torch.tensor(g["gate_w"], requires_grad=True)
    y = torch.zeros(T, d, dtype=torch.float64)
    for t in range(T):
        for j in range(k):
            e = int(g["expert_idx"][t, j])
            c = slice(e * F, (e + 1) * F)
            hid = torch.nn.functional.silu(tx[t] @ t1[:, c]) * (tx[t] @ t3[:, c])
            y = y.index_add(0, torch.tensor([t]), (tw[t, j] * (hid @ t2[c]))[None])
    (y * torch.from_numpy(dy)).sum().backward()
    for got, ref in ((g["dx"], tx.grad), (g["dW1"], t1.grad), (g["dW3"], t3.grad), (g["dW2"], t2.grad),
                     (g["d_gate"], tw.grad)):
        assert np.max(np.abs(got - ref.numpy())) < 1e-12


def test_sampled_forms_agree_with_full_layer():
    cfg, inp = _tiny_inputs(200, 128, 4, 256, 2, "swiglu", 77)
    full = O.layer_per_expert(inp["x"], inp["logits"], inp["w1"], inp["w2"], inp["dy"], 2, "swiglu",
                              True, w3=inp["w3"])
    toks = [0, 3, 50, 199]
    rows = O.layer_rows(inp["x"], full["expert_idx"], full["gate_w"], inp["w1"], inp["w2"], inp["dy"],
                        toks, 256, "swiglu", w3=inp["w3"])
    for key in ("y", "dx", "d_gate"):
        assert np.allclose(rows[key], full[key][toks], rtol=0, atol=1e-12)
    cols = [0, 7, 255]
    wg = O.weight_grad_columns(inp["x"], full["expert_idx"], full["gate_w"], inp["w1"], inp["w2"],
                               inp["dy"], 2, cols, 256, "swiglu", w3=inp["w3"])
    g = [2 * 256 + c for c in cols]
    assert np.allclose(wg["dW1"], full["dW1"][:, g], atol=1e-12)
    assert np.allclose(wg["dW3"], full["dW3"][:, g], atol=1e-12)
    assert np.allclose(wg["dW2"], full["dW2"][g], atol=1e-12)


# ----------------------------------------------------------------------------
# the generator shapes the workloads as described
# ----------------------------------------------------------------------------

def test_skewed_generator_load_shape():
    cfg = syn.CONFIGS["skewed"]
    logits = syn.make_logits(cfg)
    ei, _ = O.route_topk(logits, 1, False)
    counts = np.bincount(ei.reshape(-1), minlength=cfg.E)
    top10 = np.sort(counts)[::-1][:10].sum() / cfg.T
    assert 0.70 < top10 < 0.80
    assert (counts == 0).sum() >= 2
    assert (counts < 128).sum() >= 20


def test_padded_rows_bound():
    for cfg in syn.CONFIGS.values():
        if cfg.T * cfg.E > 2 ** 20:
            logits = syn.make_logits(cfg)
        else:
            logits = syn.make_logits(cfg)
        ei, _ = O.route_topk(logits, cfg.k, cfg.renorm)
        counts = np.bincount(ei.reshape(-1), minlength=cfg.E)
        P = int(((-(-counts // B)) * B).sum())
        assert P <= cfg.P_max


# ----------------------------------------------------------------------------
# router backward (gradient of the gate weights w.r.t. the logits)
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("renorm", [False, True])
@pytest.mark.parametrize("k", [1, 2, 5])
def test_route_backward_finite_differences(k, renorm):
    T, E = 6, 7
    z = syn.normal_f32(70 + k, 1, (T, E), 2.0).astype(np.float64)
    ei, _ = O.route_topk(z.astype(np.float32), k, renorm)
    g = np.random.default_rng(k).standard_normal((T, k))
    got = O.route_topk_backward(z.astype(np.float32), ei, g, renorm)

    def weights(zz):
        # the same experts, weights of the perturbed logits (the choice is
        # locally constant: logits differ by far more than the step)
        p = scipy.special.softmax(zz, axis=1)
        w = np.take_along_axis(p, ei.astype(np.int64), axis=1)
        return w / w.sum(1, keepdims=True) if renorm else w

    h = 1e-6
    zf = z.astype(np.float32).astype(np.float64)
    for t in range(T):
        for e in range(E):
            zp = zf.copy(); zp[t, e] += h
            zm = zf.copy(); zm[t, e] -= h
            fd = np.sum((weights(zp) - weights(zm)) * g) / (2 * h)
            assert abs(fd - got[t, e]) < 1e-7, (t, e)


def test_route_backward_matches_autograd():
    T, E, k = 9, 16, 3
    z = syn.normal_f32(81, 1, (T, E))
    for renorm in (False, True):
        ei, _ = O.route_topk(z, k, renorm)
        g = np.random.default_rng(9).standard_normal((T, k))
        tz = torch.tensor(z.astype(np.float64), requires_grad=True)
        w = torch.softmax(tz, dim=1).gather(1, torch.from_numpy(ei.astype(np.int64)))
        if renorm:
            w = w / w.sum(1, keepdim=True)
        (w * torch.from_numpy(g)).sum().backward()
        assert np.max(np.abs(O.route_topk_backward(z, ei, g, renorm) - tz.grad.numpy())) < 1e-14


def test_route_backward_closed_forms():
    # renormalised top-1: the weight is 1 whatever the logits -> zero gradient;
    # unrenormalised k = E: the weights sum to 1 -> equal d_gate gives zero
    z = syn.normal_f32(5, 5, (20, 6))
    ei, _ = O.route_topk(z, 1, True)
    assert np.max(np.abs(O.route_topk_backward(z, ei, np.ones((20, 1)), True))) < 1e-14
    ei, _ = O.route_topk(z, 6, False)
    assert np.max(np.abs(O.route_topk_backward(z, ei, np.full((20, 6), 3.0), False))) < 1e-14


# ----------------------------------------------------------------------------
# deeper experts (section 1.2: SDD -> DSD -> SDD -> DSD ...)
# ----------------------------------------------------------------------------

def _deep_case(seed, T, d, E, F, L, act):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, d))
    w1s = [rng.standard_normal((d, E * F)) * 0.5 for _ in range(L)]
    w2s = [rng.standard_normal((E * F, d)) * 0.5 for _ in range(L)]
    w3s = [rng.standard_normal((d, E * F)) * 0.5 for _ in range(L)] if act == "swiglu" else None
    dy = rng.standard_normal((T, d))
    logits = syn.normal_f32(seed, 1, (T, E))
    return x, w1s, w2s, w3s, dy, logits


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_deep_experts_top1_is_the_block_applied_twice(act):
    """With top-1 routing and renormalised weights (gate weight exactly 1),
    a two-block expert is the one-block layer applied twice with the same
    routing: y = layer(layer(x; W_1); W_2)."""
    x, w1s, w2s, w3s, dy, logits = _deep_case(21, 9, 6, 3, 4, 2, act)
    kw = lambda l: dict(w3=w3s[l]) if act == "swiglu" else {}  # noqa: E731
    deep = O.layer_deep_per_expert(x, logits, w1s, w2s, dy, 1, act, True, w3s=w3s)
    h1 = O.layer_per_expert(x, logits, w1s[0], w2s[0], dy, 1, act, True, backward=False, **kw(0))["y"]
    h2 = O.layer_per_expert(h1, logits, w1s[1], w2s[1], dy, 1, act, True, backward=False, **kw(1))["y"]
    assert np.max(np.abs(deep["y"] - h2)) < 1e-12
    assert np.all(deep["gate_w"] == 1.0)


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_deep_experts_one_block_is_the_layer(act):
    """L = 1 gives the one-block layer's outputs and gradients."""
    x, w1s, w2s, w3s, dy, logits = _deep_case(22, 8, 5, 3, 4, 1, act)
    kw = dict(w3=w3s[0]) if act == "swiglu" else {}
    a = O.layer_deep_per_expert(x, logits, w1s, w2s, dy, 2, act, False, w3s=w3s)
    b = O.layer_per_expert(x, logits, w1s[0], w2s[0], dy, 2, act, False, **kw)
    for key in ("y", "dx", "d_gate", "d_logits"):
        assert np.max(np.abs(a[key] - b[key])) < 1e-12, key
    assert np.max(np.abs(a["dW1s"][0] - b["dW1"])) < 1e-12
    assert np.max(np.abs(a["dW2s"][0] - b["dW2"])) < 1e-12


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_deep_experts_backward_by_finite_differences(act):
    T, d, E, F, k, L = 6, 4, 3, 3, 2, 3
    x, w1s, w2s, w3s, dy, logits = _deep_case(23, T, d, E, F, L, act)
    g = O.layer_deep_per_expert(x, logits, w1s, w2s, dy, k, act, False, w3s=w3s)

    def loss(x_, w1s_, w2s_, w3s_):
        return float(np.sum(O.layer_deep_per_expert(x_, logits, w1s_, w2s_, dy, k, act, False,
                                                    w3s=w3s_)["y"] * dy))

    h = 1e-6
    params = [("x", None, x, g["dx"])]
    for l in range(L):
        params += [("w1", l, w1s[l], g["dW1s"][l]), ("w2", l, w2s[l], g["dW2s"][l])]
        if act == "swiglu":
            params.append(("w3", l, w3s[l], g["dW3s"][l]))
    for name, l, arr, grad in params:
        for idx in itertools.islice(np.ndindex(arr.shape), 0, None, 5):
            vals = []
            for sgn in (1, -1):
                p = arr.copy()
                p[idx] += sgn * h
                xs, a1, a2, a3 = x, list(w1s), list(w2s), (list(w3s) if w3s else None)
                if name == "x":
                    xs = p
                elif name == "w1":
                    a1[l] = p
                elif name == "w2":
                    a2[l] = p
                else:
                    a3[l] = p
                vals.append(loss(xs, a1, a2, a3))
            fd = (vals[0] - vals[1]) / (2 * h)
            assert abs(fd - grad[idx]) < 1e-6 * max(1.0, abs(fd)), (name, l, idx)


def test_deep_experts_match_autograd_swiglu():
    T, d, E, F, k, L = 10, 5, 3, 4, 2, 2
    x, w1s, w2s, w3s, dy, logits = _deep_case(24, T, d, E, F, L, "swiglu")
    g = O.layer_deep_per_expert(x, logits, w1s, w2s, dy, k, "swiglu", True, w3s=w3s)
    tx = torch.tensor(x, requires_grad=True)
    t1 = [torch.tensor(w, requires_grad=True) for w in w1s]
    t2 = [torch.tensor(w, requires_grad=True) for w in w2s]
    t3 = [torch.tensor(w, requires_grad=True) for w in w3s]
    tw = torch.tensor(g["gate_w"], requires_grad=True)
    y = torch.zeros(T, d, dtype=torch.float64)
    for t in range(T):
        for j in range(k):
            c = slice(int(g["expert_idx"][t, j]) * F, (int(g["expert_idx"][t, j]) + 1) * F)
            h = tx[t]
            for l in range(L):
                h = (torch.nn.functional.silu(h @ t1[l][:, c]) * (h @ t3[l][:, c])) @ t2[l][c]
            y = y.index_add(0, torch.tensor([t]), (tw[t, j] * h)[None])
    (y * torch.from_numpy(dy)).sum().backward()
    pairs = [(g["dx"], tx.grad), (g["d_gate"], tw.grad)]
    for l in range(L):
        pairs += [(g["dW1s"][l], t1[l].grad), (g["dW2s"][l], t2[l].grad), (g["dW3s"][l], t3[l].grad)]
    for got, ref in pairs:
        assert np.max(np.abs(got - ref.numpy())) < 1e-11


# ----------------------------------------------------------------------------
# block-size variants (section 1.3 compares 64x64, 128x128 and 256x256)
# ----------------------------------------------------------------------------

def _topo_by_dense_mask_b(padded_offsets, F, Bs):
    po = np.asarray(padded_offsets)
    E = po.size - 1
    nb = F // Bs
    R = po[-1] // Bs
    mask = np.zeros((R, E * nb), dtype=bool)
    for e in range(E):
        mask[po[e] // Bs:po[e + 1] // Bs, e * nb:(e + 1) * nb] = True
    rr, cc = np.nonzero(mask)
    pos = -np.ones(mask.shape, dtype=np.int64)
    pos[rr, cc] = np.arange(rr.size)
    ct, rt = np.nonzero(mask.T)
    return dict(row_offsets=np.concatenate([[0], np.cumsum(mask.sum(1))]), column_indices=cc, row_indices=rr,
                column_offsets_t=np.concatenate([[0], np.cumsum(mask.sum(0))]), row_indices_t=rt,
                block_offsets_t=pos[rt, ct], nnz=rr.size)


@pytest.mark.parametrize("Bs", [64, 256])
@pytest.mark.parametrize("counts,F", [([3, 0, 130, 128, 1], 256), ([500, 7, 256, 0, 0, 300], 512), ([1000], 256)])
def test_block_size_topology_and_padding(Bs, counts, F):
    ei = np.repeat(np.arange(len(counts)), counts).astype(np.int32)[:, None]
    pp = O.permute_pad(ei, len(counts), block=Bs)
    # groups padded to the block size, at most Bs - 1 pad rows each
    assert np.array_equal(np.diff(pp["padded_offsets"]), [-(-c // Bs) * Bs for c in counts])
    tp = O.build_topology(pp["padded_offsets"], F, pp["tokens_per_expert"], block=Bs)
    ref = _topo_by_dense_mask_b(pp["padded_offsets"], F, Bs)
    for key, v in ref.items():
        assert np.array_equal(np.asarray(tp[key]), np.asarray(v)), key
    held = (pp["src_of_row"] >= 0).reshape(-1, Bs).sum(axis=1) if tp["R"] else np.zeros(0, dtype=np.int64)
    assert np.array_equal(tp["row_fill"], held)


@pytest.mark.parametrize("Bs", [64, 256])
@pytest.mark.parametrize("act,k,renorm", [("gelu", 2, True), ("swiglu", 1, False)])
def test_block_size_chain_equals_per_expert(Bs, act, k, renorm):
    """Any block size gives the dense per-expert MLP (no blocks at all)."""
    cfg, inp = _tiny_inputs(300, 128, 3, 512, k, act, 50 + k)
    a = O.layer_blocksparse(inp["x"], inp["logits"], inp["w1"], inp["w2"], inp["dy"], k, act, renorm,
                            w3=inp.get("w3"), block=Bs)
    b = O.layer_per_expert(inp["x"], inp["logits"], inp["w1"], inp["w2"], inp["dy"], k, act, renorm,
                           w3=inp.get("w3"))
    assert a["topo"]["block"] == Bs and a["P"] % Bs == 0
    for key in ("y", "dx", "d_gate", "dW1", "dW2") + (("dW3",) if act == "swiglu" else ()):
        scale = np.max(np.abs(b[key]))
        assert np.max(np.abs(a[key] - b[key])) <= 1e-12 * max(scale, 1e-300), key
