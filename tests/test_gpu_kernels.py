"""Parity of every C-ABI call against the fp64 oracle, one call at a time.

Integer outputs (routing indices, bins, offsets, permutation, topology)
must match bit for bit; copies (x_perm) too.  Float outputs must satisfy
the single-call bound of helpers.TOL_SINGLE.  Sizes span several 128-row
tiles, ragged expert groups (0, 1, 5, 127, 128, 129, 300 tokens) and, for
the products, more tiles than SMs so that every CTA loops.
"""

import numpy as np
import pytest
import torch

import dmoe_synth as syn
import oracle as O
from helpers import (RMS_SINGLE, TOL_SINGLE, assert_close, bf16_from_bits, bf16_from_f64, counts_routing, dev,
                     f32, host, i32, load_topology)

pytestmark = pytest.mark.gpu

dm = None


@pytest.fixture(scope="module", autouse=True)
def _lib():
    global dm
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dropless_moe_block_gb300 import build
    build.build()
    import dropless_moe_block_gb300 as m
    dm = m
    dm.get_error(clear=True)
    yield


@pytest.fixture(autouse=True)
def _no_device_error():
    yield
    assert dm.get_error(clear=True) == 0


@pytest.fixture(params=[True, False], ids=["m64", "m128"])
def fill(request):
    """Products run with the row fill (M = 64 on half-empty row blocks) and
    without it (M = 128 everywhere)."""
    return request.param


@pytest.fixture(params=[128, 256, "pair", "pair512"], ids=["n128", "n256", "pair", "pair512"])
def tile_n(request):
    """Runs a product test once per tile width (forced where the shape
    allows, one CTA per tile), once with CTA pairs (M = 256 x N = 256 tiles
    over two SMs, forced where the shape allows) and once with pair tiles of
    two N = 256 sub-tiles sharing their A slices (256 x 512, forced where the
    shape allows; 256 x 256 pairs elsewhere)."""
    if request.param in ("pair", "pair512"):
        dm.set_tile_n(0)
        dm.set_pair(2 if request.param == "pair" else 3)
    else:
        dm.set_tile_n(request.param)
        dm.set_pair(1)
    yield request.param
    dm.set_tile_n(0)
    dm.set_pair(0)


# ------------------------------------------------------------------ routing

ROUTE_CASES = [
    (512, 4, 1, False, "normal"), (8192, 64, 1, False, "normal"), (4096, 64, 8, False, "normal"),
    (8192, 8, 2, True, "normal"), (333, 37, 5, True, "normal"), (700, 1024, 8, False, "normal"),
    (300, 9, 3, False, "ties"), (1, 1, 1, True, "normal"), (64, 16, 16, True, "normal"),
    (1000, 200, 4, True, "ties"),
]


@pytest.mark.parametrize("T,E,k,renorm,kind", ROUTE_CASES)
def test_route_topk(T, E, k, renorm, kind):
    if kind == "ties":
        logits = syn.integers(T + E, 1, -3, 3, (T, E)).astype(np.float32)
    else:
        logits = syn.normal_f32(T * 7 + E, 1, (T, E), 2.0)
    ei_ref, w_ref = O.route_topk(logits, k, renorm)
    ei = torch.empty(T, k, dtype=torch.int32, device=dev())
    w = torch.empty(T, k, dtype=torch.float32, device=dev())
    dm.route_topk(f32(logits), k, renorm, ei, w)
    assert np.array_equal(host(ei), ei_ref)
    # fp32 softmax vs fp64: a few ulp of the sum of E terms
    assert np.max(np.abs(host(w) - w_ref)) <= 1e-5


@pytest.mark.parametrize("name", ["tiny", "moe_xs", "skewed", "mixtral", "fine"])
def test_route_topk_workloads(name):
    cfg = syn.CONFIGS[name]
    logits = syn.make_logits(cfg)
    ei_ref, w_ref = O.route_topk(logits, cfg.k, cfg.renorm)
    ei = torch.empty(cfg.T, cfg.k, dtype=torch.int32, device=dev())
    w = torch.empty(cfg.T, cfg.k, dtype=torch.float32, device=dev())
    dm.route_topk(f32(logits), cfg.k, cfg.renorm, ei, w)
    assert np.array_equal(host(ei), ei_ref)
    assert np.max(np.abs(host(w) - w_ref)) <= 1e-5


@pytest.mark.parametrize("T,E,k,renorm,kind", ROUTE_CASES)
def test_route_topk_backward(T, E, k, renorm, kind):
    """fp32 on both inputs: the kernel's softmax and products against fp64."""
    if kind == "ties":
        logits = syn.integers(T + E, 1, -3, 3, (T, E)).astype(np.float32)
    else:
        logits = syn.normal_f32(T * 7 + E, 1, (T, E), 2.0)
    ei_ref, w_ref = O.route_topk(logits, k, renorm)
    d_gate = syn.normal_f32(T, 9, (T, k))
    ref = O.route_topk_backward(logits, ei_ref, d_gate, renorm)
    out = torch.full((T, E), float("nan"), dtype=torch.float32, device=dev())
    dm.route_topk_backward(f32(logits), i32(ei_ref), f32(w_ref), f32(d_gate), renorm, out)
    got = host(out)
    scale = max(1.0, float(np.max(np.abs(ref))))
    assert np.max(np.abs(got - ref)) <= 2e-6 * scale


# ---------------------------------------------------------- permute + pad

def _run_permute(ei_np, E, x_bits):
    T, k = ei_np.shape
    d = x_bits.shape[1]
    P_max = dm.padded_rows_max(T, k, E)
    z = lambda n, dt: torch.zeros(max(1, n), dtype=dt, device=dev())  # noqa: E731
    out = dict(tpe=z(E, torch.int32), po=z(E + 1, torch.int32), dest=z(T * k, torch.int32),
               src=torch.full((max(1, P_max),), 12345, dtype=torch.int32, device=dev()),
               xp=torch.full((max(1, P_max), d), 7.0, dtype=torch.bfloat16, device=dev()),
               P=z(1, torch.int32), ws=z(dm.permute_pad_workspace_size(T, k, E), torch.uint8))
    x = bf16_from_bits(x_bits) if T else torch.zeros(0, d, dtype=torch.bfloat16, device=dev())
    dm.permute_pad(x, i32(ei_np).reshape(T, k), E, P_max, out["tpe"], out["po"], out["dest"], out["src"],
                   out["xp"], out["P"], out["ws"])
    torch.cuda.synchronize()
    return out, P_max


def _check_permute(ei_np, E, x_bits):
    T, k = ei_np.shape
    ref = O.permute_pad(ei_np, E)
    out, P_max = _run_permute(ei_np, E, x_bits)
    P = ref["P"]
    assert int(out["P"].item()) == P
    assert np.array_equal(host(out["tpe"])[:E], ref["tokens_per_expert"])
    assert np.array_equal(host(out["po"])[:E + 1], ref["padded_offsets"])
    assert np.array_equal(host(out["dest"])[:T * k], ref["dest_row"])
    src = host(out["src"])
    assert np.array_equal(src[:P], ref["src_of_row"])
    assert np.all(src[P:P_max] == -1)
    # x_perm: row p is x[src // k] bit for bit, pad rows are +0.0
    xp = out["xp"].view(torch.int16).cpu().numpy().view(np.uint16)[:P]
    want = np.zeros((P, x_bits.shape[1]), dtype=np.uint16)
    held = ref["src_of_row"] >= 0
    want[held] = x_bits[ref["src_of_row"][held] // k]
    assert np.array_equal(xp, want)
    return out


GATE_CASES = [
    # T, d, E, k, renormalize: a ragged last tile, every MMA width N = 32 ..
    # 256 (E padded up to a power of two >= 32), K from one slice to 64,
    # d split over clusters of 1, 2 and 4 CTAs (few tiles, enough slices)
    (1, 64, 1, 1, False),
    (300, 512, 64, 1, False),
    (777, 256, 8, 2, True),
    (256, 3584, 64, 8, False),
    (130, 4096, 8, 2, True),
    (200, 128, 100, 3, False),
    (129, 192, 256, 8, True),
    (100, 1024, 256, 4, False),
    (70, 1024, 100, 2, True),
    (20000, 512, 64, 2, False),
]


@pytest.mark.parametrize("T,d,E,k,renorm", GATE_CASES)
def test_gate_route_topk(T, d, E, k, renorm):
    """Linear gate + router in one kernel: the logits against the oracle's
    fp64 product within the fp32 summation bound, the routing decision on
    the GPU's fp32 logits exactly as the oracle and as dmoe_route_topk."""
    x = syn.normal_bf16(31, 1, (T, d))
    w = syn.normal_bf16(31, 2, (E, d), 1.0 / np.sqrt(d))
    logits = torch.full((T, E), float("nan"), dtype=torch.float32, device=dev())
    ei = torch.full((T, k), -7, dtype=torch.int32, device=dev())
    gw = torch.full((T, k), float("nan"), dtype=torch.float32, device=dev())
    dm.gate_route_topk(bf16_from_bits(x), bf16_from_bits(w), k, renorm, logits, ei, gw)
    torch.cuda.synchronize()
    assert dm.get_error(clear=True) == 0
    lg = host(logits)
    ref = O.gate_logits(x, w)
    # bf16 x bf16 products are exact in fp32; a sum of d of them is within
    # d * 2^-24 * sum |terms| of the exact value (twice that as margin)
    S = np.abs(O.bf16_to_f64(x)) @ np.abs(O.bf16_to_f64(w)).T
    assert np.all(np.abs(lg - ref) <= 2.0 * d * 2.0 ** -24 * S)
    ri, rw = O.route_topk(lg.astype(np.float32), k, renorm)
    assert np.array_equal(host(ei), ri)
    assert np.max(np.abs(host(gw) - rw)) <= 1e-5
    ei2 = torch.empty_like(ei)
    gw2 = torch.empty_like(gw)
    dm.route_topk(logits, k, renorm, ei2, gw2)
    assert torch.equal(ei2, ei) and torch.equal(gw2, gw)


def test_gate_route_topk_empty_batch():
    x = torch.empty((0, 128), dtype=torch.bfloat16, device=dev())
    w = torch.ones((8, 128), dtype=torch.bfloat16, device=dev())
    z = torch.empty((0, 8), dtype=torch.float32, device=dev())
    dm.gate_route_topk(x, w, 2, False, z, torch.empty((0, 2), dtype=torch.int32, device=dev()),
                       torch.empty((0, 2), dtype=torch.float32, device=dev()))
    torch.cuda.synchronize()
    assert dm.get_error(clear=True) == 0


@pytest.mark.parametrize("name", ["tiny", "moe_xs", "skewed", "mixtral", "fine"])
def test_permute_pad_workloads(name):
    cfg = syn.CONFIGS[name]
    ei, _ = O.route_topk(syn.make_logits(cfg), cfg.k, cfg.renorm)
    _check_permute(ei, cfg.E, syn.make_x(cfg))


EDGE_COUNTS = [
    [5, 0, 140, 128, 300, 1],  # ragged, empty, exactly 128
    [0, 0, 0, 129],            # all on the last expert, one over a block
    [1],                        # one token, one expert
    [127, 128, 129, 255, 256, 257, 0, 0],
    [0] * 63 + [1000],          # 64 experts, one busy
]


@pytest.mark.parametrize("counts", EDGE_COUNTS)
def test_permute_pad_edges(counts):
    ei = counts_routing(counts)
    # shuffle token order so groups interleave in batch order
    perm = np.random.default_rng(len(counts)).permutation(ei.shape[0])
    ei = np.ascontiguousarray(ei[perm])
    x = syn.normal_bf16(3, 2, (ei.shape[0], 64))
    _check_permute(ei, len(counts), x)


def test_permute_pad_topk_many_slots():
    T, E, k = 1500, 1024, 8
    ei, _ = O.route_topk(syn.normal_f32(9, 1, (T, E)), k, False)
    _check_permute(ei, E, syn.normal_bf16(9, 2, (T, 16)))


def test_permute_pad_empty_batch():
    out, P_max = _run_permute(np.zeros((0, 2), dtype=np.int32), 4, np.zeros((0, 32), dtype=np.uint16))
    assert int(out["P"].item()) == 0
    assert np.all(host(out["po"]) == 0)


def test_permute_pad_repeatable():
    cfg = syn.CONFIGS["fine"]
    ei, _ = O.route_topk(syn.make_logits(cfg), cfg.k, cfg.renorm)
    x = syn.normal_bf16(1, 1, (cfg.T, 64))
    a, _ = _run_permute(ei, cfg.E, x)
    for _ in range(3):  # also exercises the self-resetting grid barrier
        b, _ = _run_permute(ei, cfg.E, x)
        for key in ("tpe", "po", "dest", "src", "P"):
            assert torch.equal(a[key], b[key])
        assert torch.equal(a["xp"].view(torch.int16), b["xp"].view(torch.int16))


# --------------------------------------------------------------- topology

def _check_topology(padded_offsets, E, F, P_max, tokens_per_expert=None):
    ref = O.build_topology(padded_offsets, F, tokens_per_expert)
    topo = dm.Topology(E, F, P_max)
    dm.build_topology(i32(padded_offsets), topo, i32(tokens_per_expert) if tokens_per_expert is not None else None)
    torch.cuda.synchronize()
    if tokens_per_expert is not None:
        rf = host(topo.row_fill)
        assert np.array_equal(rf[:ref["R"]], ref["row_fill"]) and np.all(rf[ref["R"]:] == 0)
    nnz, R = ref["nnz"], ref["R"]
    assert topo.nnz() == nnz and topo.P() == padded_offsets[-1]
    ro = host(topo.row_offsets)
    assert np.array_equal(ro[:R + 1], ref["row_offsets"])
    assert np.all(ro[R + 1:] == nnz)
    for key in ("column_indices", "row_indices", "row_indices_t", "block_offsets_t"):
        assert np.array_equal(host(getattr(topo, key))[:nnz], ref[key]), key
    assert np.array_equal(host(topo.column_offsets_t), ref["column_offsets_t"])


@pytest.mark.parametrize("name", ["tiny", "moe_xs", "skewed", "mixtral", "fine"])
def test_topology_workloads(name):
    cfg = syn.CONFIGS[name]
    ei, _ = O.route_topk(syn.make_logits(cfg), cfg.k, cfg.renorm)
    pp = O.permute_pad(ei, cfg.E)
    _check_topology(pp["padded_offsets"], cfg.E, cfg.F, cfg.P_max, pp["tokens_per_expert"])


@pytest.mark.parametrize("counts,F", [(EDGE_COUNTS[0], 256), (EDGE_COUNTS[1], 128), (EDGE_COUNTS[3], 384),
                                      (EDGE_COUNTS[4], 512), ([0, 0, 0], 256)])
def test_topology_edges(counts, F):
    ei = counts_routing(counts) if sum(counts) else np.zeros((0, 1), dtype=np.int32)
    pp = O.permute_pad(ei, len(counts))
    _check_topology(pp["padded_offsets"], len(counts), F, syn.padded_rows_max(max(1, sum(counts)), 1, len(counts)),
                    pp["tokens_per_expert"])


def test_topology_after_permute_chain():
    cfg = syn.CONFIGS["skewed"]
    ei, _ = O.route_topk(syn.make_logits(cfg), cfg.k, cfg.renorm)
    out, P_max = _run_permute(ei, cfg.E, syn.normal_bf16(2, 2, (cfg.T, 8)))
    ref = O.build_topology(O.permute_pad(ei, cfg.E)["padded_offsets"], cfg.F)
    topo = dm.Topology(cfg.E, cfg.F, P_max)
    dm.build_topology(out["po"], topo, out["tpe"])
    assert topo.nnz() == ref["nnz"]
    assert np.array_equal(host(topo.block_offsets_t)[:ref["nnz"]], ref["block_offsets_t"])


# ------------------------------------------------- fused dispatch (a1-a3)

def _run_dispatch(logits, x_bits, E, k, renorm, F, with_topo=True):
    T = logits.shape[0]
    d = x_bits.shape[1]
    P_max = dm.padded_rows_max(T, k, E)
    z = lambda n, dt: torch.zeros(max(1, n), dtype=dt, device=dev())  # noqa: E731
    out = dict(ei=torch.full((max(1, T * k),), -7, dtype=torch.int32, device=dev()), w=z(T * k, torch.float32),
               tpe=z(E, torch.int32), po=z(E + 1, torch.int32), dest=z(T * k, torch.int32),
               src=torch.full((max(1, P_max),), 12345, dtype=torch.int32, device=dev()),
               xp=torch.full((max(1, P_max), d), 7.0, dtype=torch.bfloat16, device=dev()),
               P=z(1, torch.int32), ws=z(dm.permute_pad_workspace_size(T, k, E), torch.uint8))
    topo = dm.Topology(E, F, P_max)
    x = bf16_from_bits(x_bits) if T else torch.zeros(0, d, dtype=torch.bfloat16, device=dev())
    lg = f32(logits) if T else torch.zeros(0, E, dtype=torch.float32, device=dev())
    dm.dispatch(lg, x, k, renorm, out["ei"], out["w"], out["tpe"], out["po"], out["dest"], out["src"], out["xp"],
                out["P"], out["ws"], P_max, topo if with_topo else None)
    if not with_topo:
        dm.build_topology(out["po"], topo, out["tpe"])
    torch.cuda.synchronize()
    return out, topo, P_max


def _check_dispatch(logits, x_bits, E, k, renorm, F, with_topo=True):
    """Every output of the fused launch against the oracle's route, permute
    and topology (integers and copies bit for bit, weights to 1e-5)."""
    T = logits.shape[0]
    ei_ref, w_ref = O.route_topk(logits, k, renorm)
    ref = O.permute_pad(ei_ref, E)
    tref = O.build_topology(ref["padded_offsets"], F, ref["tokens_per_expert"])
    out, topo, P_max = _run_dispatch(logits, x_bits, E, k, renorm, F, with_topo)
    assert np.array_equal(host(out["ei"])[:T * k].reshape(T, k), ei_ref)
    if T:
        assert np.max(np.abs(host(out["w"])[:T * k].reshape(T, k) - w_ref)) <= 1e-5
    P = ref["P"]
    assert int(out["P"].item()) == P and topo.P() == P
    assert np.array_equal(host(out["tpe"])[:E], ref["tokens_per_expert"])
    assert np.array_equal(host(out["po"])[:E + 1], ref["padded_offsets"])
    assert np.array_equal(host(out["dest"])[:T * k], ref["dest_row"])
    src = host(out["src"])
    assert np.array_equal(src[:P], ref["src_of_row"])
    assert np.all(src[P:P_max] == -1)
    xp = out["xp"].view(torch.int16).cpu().numpy().view(np.uint16)[:P]
    want = np.zeros((P, x_bits.shape[1]), dtype=np.uint16)
    held = ref["src_of_row"] >= 0
    want[held] = x_bits[ref["src_of_row"][held] // k]
    assert np.array_equal(xp, want)
    nnz, R = tref["nnz"], tref["R"]
    assert topo.nnz() == nnz
    ro = host(topo.row_offsets)
    assert np.array_equal(ro[:R + 1], tref["row_offsets"])
    assert np.all(ro[R + 1:] == nnz)
    for key in ("column_indices", "row_indices", "row_indices_t", "block_offsets_t"):
        assert np.array_equal(host(getattr(topo, key))[:nnz], tref[key]), key
    assert np.array_equal(host(topo.column_offsets_t), tref["column_offsets_t"])
    rf = host(topo.row_fill)
    assert np.array_equal(rf[:R], tref["row_fill"]) and np.all(rf[R:] == 0)
    return out


@pytest.mark.parametrize("name", ["tiny", "moe_xs", "skewed", "mixtral", "fine"])
@pytest.mark.parametrize("with_topo", [True, False], ids=["with_topology", "then_topology_kernel"])
def test_dispatch_workloads(name, with_topo):
    cfg = syn.CONFIGS[name]
    _check_dispatch(syn.make_logits(cfg), syn.make_x(cfg), cfg.E, cfg.k, cfg.renorm, cfg.F, with_topo)


@pytest.mark.parametrize("T,E,k,renorm,d,F,kind", [
    (1, 1, 1, True, 64, 128, "normal"),          # one token, one expert
    (300, 9, 3, False, 32, 256, "ties"),         # equal logits: lower id first
    (1500, 1024, 8, False, 16, 128, "normal"),   # widest router (32 logits per lane)
    (64, 16, 16, True, 64, 384, "normal"),       # k = E
    (777, 37, 5, True, 128, 256, "normal"),      # ragged everything
    (50, 200, 2, False, 8, 128, "normal"),       # fewer tokens than blocks of the grid
])
def test_dispatch_edges(T, E, k, renorm, d, F, kind):
    if kind == "ties":
        logits = syn.integers(T + E, 1, -3, 3, (T, E)).astype(np.float32)
    else:
        logits = syn.normal_f32(T * 7 + E, 1, (T, E), 2.0)
    _check_dispatch(logits, syn.normal_bf16(T + 5, 2, (T, d)), E, k, renorm, F)


def test_dispatch_empty_batch():
    out, topo, _ = _run_dispatch(np.zeros((0, 4), dtype=np.float32), np.zeros((0, 32), dtype=np.uint16), 4, 2,
                                 False, 256)
    assert int(out["P"].item()) == 0 and topo.nnz() == 0 and topo.P() == 0
    assert np.all(host(out["po"]) == 0)
    assert np.all(host(topo.column_offsets_t) == 0)


def test_dispatch_matches_separate_calls():
    """The fused launch and route_topk -> permute_pad -> build_topology give
    the same bits (the weights included), repeatedly (the grid barrier resets)."""
    cfg = syn.CONFIGS["fine"]
    logits, x_bits = syn.make_logits(cfg), syn.normal_bf16(4, 4, (cfg.T, 64))
    T, E, k = cfg.T, cfg.E, cfg.k
    ei = torch.empty(T, k, dtype=torch.int32, device=dev())
    w = torch.empty(T, k, dtype=torch.float32, device=dev())
    dm.route_topk(f32(logits), k, cfg.renorm, ei, w)
    sep, P_max = _run_permute(host(ei), E, x_bits)
    topo_sep = dm.Topology(E, cfg.F, P_max)
    dm.build_topology(sep["po"], topo_sep, sep["tpe"])
    for _ in range(3):
        fused, topo, _ = _run_dispatch(logits, x_bits, E, k, cfg.renorm, cfg.F)
        assert torch.equal(fused["ei"][:T * k], ei.view(-1)) and torch.equal(fused["w"][:T * k], w.view(-1))
        for key in ("tpe", "po", "dest", "src", "P"):
            assert torch.equal(fused[key], sep[key]), key
        assert torch.equal(fused["xp"].view(torch.int16), sep["xp"].view(torch.int16))
        for key in ("row_offsets", "column_indices", "row_indices", "column_offsets_t", "row_indices_t",
                    "block_offsets_t", "nnz_dev", "P_dev", "row_fill"):
            assert torch.equal(getattr(topo, key), getattr(topo_sep, key)), key


# ------------------------------------------------------ block-sparse GEMMs

class Setup:
    """Routing with given expert counts, oracle metadata loaded on the GPU.
    With row_fill, row blocks holding at most 64 tokens run at M = 64."""

    def __init__(self, counts, F, seed=0, row_fill=True, block=128):
        self.E = len(counts)
        self.F = F
        self.B = block
        ei = counts_routing(counts)
        self.T = ei.shape[0]
        self.pp = O.permute_pad(ei, self.E, block=block)
        self.tp = O.build_topology(self.pp["padded_offsets"], F, self.pp["tokens_per_expert"], block=block)
        self.P = self.pp["P"]
        self.P_max = syn.padded_rows_max(self.T, 1, self.E, block)
        self.topo = dm.Topology(self.E, F, self.P_max, row_fill=row_fill, block=block)
        load_topology(self.topo, self.tp, self.P)
        self.nnz = self.tp["nnz"]
        self.seed = seed
        self.stream = 100

    def dense_rows(self, n, std=1.0):
        """[P_max, n] bf16 bits, pad rows (and rows >= P) zero."""
        self.stream += 1
        a = syn.normal_bf16(self.seed, self.stream, (self.P_max, n), std)
        a[self.P:] = 0
        a[:self.P][self.pp["src_of_row"] < 0] = 0
        return a

    def mat(self, shape, std=1.0):
        self.stream += 1
        return syn.normal_bf16(self.seed, self.stream, shape, std)

    def blocks(self, std=1.0):
        """Random blocks whose padding rows are zero, as in the layer (the
        activation of a zero row is zero)."""
        self.stream += 1
        b = syn.normal_bf16(self.seed, self.stream, (max(1, self.topo.nnz_max), self.B, self.B), std)
        fill = self.tp["row_fill"][self.tp["row_indices"]]
        for q in range(self.nnz):
            b[q, fill[q]:] = 0
        return b

    def empty_blocks(self):
        return torch.full((max(1, self.topo.nnz_max), self.B, self.B), float("nan"), dtype=torch.bfloat16,
                          device=dev())


SMALL = ([5, 0, 140, 128, 300, 1], 256)          # 16 blocks, ragged
MANY = ([700, 3, 1200, 0, 2500, 900, 130, 1], 512)  # 164 row blocks... > #SMs tiles


@pytest.mark.parametrize("shape", [SMALL, MANY])
@pytest.mark.parametrize("K", [64, 256, 1024])
@pytest.mark.parametrize("b_trans", [False, True])
def test_sdd_store(shape, K, b_trans, tile_n, fill):
    s = Setup(*shape, seed=K + int(b_trans), row_fill=fill)
    X = s.dense_rows(K)
    EF = s.E * s.F
    W = s.mat((EF, K) if b_trans else (K, EF), 1.0 / np.sqrt(K))
    out = s.empty_blocks()
    dm.sdd(bf16_from_bits(X), bf16_from_bits(W), K, s.topo, dm.EPI_STORE, out, b_trans=b_trans)
    ref = O.sdd(X[:s.P], W, s.tp, b_trans=b_trans)
    assert_close(host(out)[:s.nnz], ref, TOL_SINGLE, RMS_SINGLE, "sdd")


@pytest.mark.parametrize("shape", [SMALL, MANY])
def test_sdd_gelu_fwd(shape, tile_n, fill):
    s = Setup(*shape, seed=11, row_fill=fill)
    K = 512
    X = s.dense_rows(K)
    W = s.mat((K, s.E * s.F), 1.0 / np.sqrt(K))
    G, Aa = s.empty_blocks(), s.empty_blocks()
    dm.sdd(bf16_from_bits(X), bf16_from_bits(W), K, s.topo, dm.EPI_GELU_FWD, G, Aa)
    ref = O.sdd(X[:s.P], W, s.tp)
    assert_close(host(G)[:s.nnz], O.gelu_grad(ref), TOL_SINGLE, RMS_SINGLE, "gelu'(H)")
    assert_close(host(Aa)[:s.nnz], O.gelu(ref), TOL_SINGLE, RMS_SINGLE, "gelu(H)")


@pytest.mark.parametrize("shape", [SMALL, MANY])
def test_sdd_swiglu_fwd(shape, tile_n, fill):
    s = Setup(*shape, seed=12, row_fill=fill)
    K = 384
    X = s.dense_rows(K)
    W1 = s.mat((K, s.E * s.F), 1.0 / np.sqrt(K))
    W3 = s.mat((K, s.E * s.F), 1.0 / np.sqrt(K))
    G1, G3, Aa = s.empty_blocks(), s.empty_blocks(), s.empty_blocks()
    dm.sdd(bf16_from_bits(X), bf16_from_bits(W1), K, s.topo, dm.EPI_SWIGLU_FWD, G1, G3, Aa,
           B2=bf16_from_bits(W3))
    r1 = O.sdd(X[:s.P], W1, s.tp)
    r3 = O.sdd(X[:s.P], W3, s.tp)
    assert_close(host(G1)[:s.nnz], r3 * O.silu_grad(r1), TOL_SINGLE, RMS_SINGLE, "H3 silu'(H1)")
    assert_close(host(G3)[:s.nnz], O.silu(r1), TOL_SINGLE, RMS_SINGLE, "silu(H1)")
    assert_close(host(Aa)[:s.nnz], O.silu(r1) * r3, TOL_SINGLE, RMS_SINGLE, "silu(H1)*H3")


@pytest.mark.parametrize("shape", [SMALL, MANY])
def test_sdd_gelu_bwd(shape, tile_n, fill):
    s = Setup(*shape, seed=13, row_fill=fill)
    K = 256
    dY = s.dense_rows(K)
    W2 = s.mat((s.E * s.F, K), 1.0 / np.sqrt(K))
    Gb = s.blocks()  # stored gelu'(H) factors
    dH = s.empty_blocks()
    dm.sdd(bf16_from_bits(dY), bf16_from_bits(W2), K, s.topo, dm.EPI_GELU_BWD, dH, b_trans=True,
           aux0=bf16_from_bits(Gb))
    dA = O.sdd(dY[:s.P], W2, s.tp, b_trans=True)
    ref = dA * O.bf16_to_f64(Gb[:s.nnz])
    assert_close(host(dH)[:s.nnz], ref, TOL_SINGLE, RMS_SINGLE, "dH")


@pytest.mark.parametrize("shape", [SMALL, MANY])
def test_sdd_swiglu_bwd(shape, tile_n, fill):
    s = Setup(*shape, seed=14, row_fill=fill)
    K = 256
    dY = s.dense_rows(K)
    W2 = s.mat((s.E * s.F, K), 1.0 / np.sqrt(K))
    G1b, G3b = s.blocks(), s.blocks()  # stored da/dh1, da/dh3 factors
    dH1, dH3 = s.empty_blocks(), s.empty_blocks()
    dm.sdd(bf16_from_bits(dY), bf16_from_bits(W2), K, s.topo, dm.EPI_SWIGLU_BWD, dH1, dH3, b_trans=True,
           aux0=bf16_from_bits(G1b), aux1=bf16_from_bits(G3b))
    dA = O.sdd(dY[:s.P], W2, s.tp, b_trans=True)
    assert_close(host(dH1)[:s.nnz], dA * O.bf16_to_f64(G1b[:s.nnz]), TOL_SINGLE, RMS_SINGLE, "dH1")
    assert_close(host(dH3)[:s.nnz], dA * O.bf16_to_f64(G3b[:s.nnz]), TOL_SINGLE, RMS_SINGLE, "dH3")


@pytest.mark.parametrize("shape", [SMALL, MANY])
@pytest.mark.parametrize("N", [128, 512])
def test_dsd(shape, N, tile_n, fill):
    s = Setup(*shape, seed=20 + N, row_fill=fill)
    S = s.blocks(1.0 / 16)
    W = s.mat((s.E * s.F, N))
    C = torch.full((s.P_max, N), float("nan"), dtype=torch.bfloat16, device=dev())
    dm.dsd(s.topo, bf16_from_bits(S), bf16_from_bits(W), N, C)
    ref = O.dsd(S[:s.nnz], W, s.tp, s.P)
    assert_close(host(C)[:s.P], ref, TOL_SINGLE, RMS_SINGLE, "dsd")


@pytest.mark.parametrize("shape", [SMALL, MANY])
@pytest.mark.parametrize("second", [False, True])
@pytest.mark.parametrize("N", [256, 512])
def test_dsd_t(shape, second, N, tile_n, fill):
    s = Setup(*shape, seed=30 + int(second) + N, row_fill=fill)
    S, W = s.blocks(1.0 / 16), s.mat((N, s.E * s.F))
    S2, W2 = (s.blocks(1.0 / 16), s.mat((N, s.E * s.F))) if second else (None, None)
    C = torch.full((s.P_max, N), float("nan"), dtype=torch.bfloat16, device=dev())
    dm.dsd_t(s.topo, bf16_from_bits(S), bf16_from_bits(W), N, C,
             S2=bf16_from_bits(S2) if second else None, Bm2=bf16_from_bits(W2) if second else None)
    ref = O.dsd(S[:s.nnz], W, s.tp, s.P, w_trans=True,
                blocks2=S2[:s.nnz] if second else None, W2=W2)
    assert_close(host(C)[:s.P], ref, TOL_SINGLE, RMS_SINGLE, "dsd_t")


@pytest.mark.parametrize("shape", [SMALL, MANY, ([0, 300, 0, 0, 5], 256), ([0, 300, 0, 0, 5], 512)])
@pytest.mark.parametrize("c_trans", [False, True])
@pytest.mark.parametrize("N", [256, 512])
def test_dstd(shape, c_trans, N, tile_n):
    s = Setup(*shape, seed=40 + int(c_trans) + N)
    S = s.blocks(1.0 / 8)
    D = s.dense_rows(N)
    EF = s.E * s.F
    C = torch.full((N, EF) if c_trans else (EF, N), float("nan"), dtype=torch.bfloat16, device=dev())
    dm.dstd(s.topo, bf16_from_bits(S), bf16_from_bits(D), N, C, c_trans=c_trans)
    ref = O.dstd(S[:s.nnz], D[:s.P], s.tp, c_trans=c_trans)
    assert_close(host(C), ref, TOL_SINGLE, RMS_SINGLE, "dstd")
    # experts without tokens get exactly zero gradient
    for e, c in enumerate(shape[0]):
        if c == 0:
            sl = slice(e * s.F, (e + 1) * s.F)
            blk = host(C)[:, sl] if c_trans else host(C)[sl]
            assert np.all(blk == 0)


# ------------------------------------------------------------- combine

# ------------------------------------------- block-size variants (64, 256)

def _run_permute_block(ei_np, E, x_bits, block):
    T, k = ei_np.shape
    d = x_bits.shape[1]
    P_max = dm.padded_rows_max(T, k, E, block)
    z = lambda n, dt: torch.zeros(max(1, n), dtype=dt, device=dev())  # noqa: E731
    out = dict(tpe=z(E, torch.int32), po=z(E + 1, torch.int32), dest=z(T * k, torch.int32),
               src=torch.full((max(1, P_max),), 12345, dtype=torch.int32, device=dev()),
               xp=torch.full((max(1, P_max), d), 7.0, dtype=torch.bfloat16, device=dev()),
               P=z(1, torch.int32), ws=z(dm.permute_pad_workspace_size(T, k, E), torch.uint8))
    dm.permute_pad(bf16_from_bits(x_bits), i32(ei_np).reshape(T, k), E, P_max, out["tpe"], out["po"], out["dest"],
                   out["src"], out["xp"], out["P"], out["ws"], block=block)
    torch.cuda.synchronize()
    return out, P_max


@pytest.mark.parametrize("block", [64, 256])
@pytest.mark.parametrize("name", ["tiny", "moe_xs", "fine"])
def test_permute_and_topology_block_sizes(block, name):
    cfg = syn.CONFIGS[name]
    ei, _ = O.route_topk(syn.make_logits(cfg), cfg.k, cfg.renorm)
    x = syn.normal_bf16(5, 5, (cfg.T, 64))
    ref = O.permute_pad(ei, cfg.E, block=block)
    out, P_max = _run_permute_block(ei, cfg.E, x, block)
    P = ref["P"]
    assert int(out["P"].item()) == P
    for key, rk in (("tpe", "tokens_per_expert"), ("po", "padded_offsets"), ("dest", "dest_row")):
        assert np.array_equal(host(out[key])[:len(ref[rk])], ref[rk]), key
    src = host(out["src"])
    assert np.array_equal(src[:P], ref["src_of_row"]) and np.all(src[P:P_max] == -1)
    xp = out["xp"].view(torch.int16).cpu().numpy().view(np.uint16)[:P]
    want = np.zeros((P, x.shape[1]), dtype=np.uint16)
    held = ref["src_of_row"] >= 0
    want[held] = x[ref["src_of_row"][held] // cfg.k]
    assert np.array_equal(xp, want)
    tref = O.build_topology(ref["padded_offsets"], cfg.F, ref["tokens_per_expert"], block=block)
    topo = dm.Topology(cfg.E, cfg.F, P_max, block=block)
    dm.build_topology(out["po"], topo, out["tpe"])
    torch.cuda.synchronize()
    nnz, R = tref["nnz"], tref["R"]
    assert topo.nnz() == nnz and topo.P() == P
    ro = host(topo.row_offsets)
    assert np.array_equal(ro[:R + 1], tref["row_offsets"]) and np.all(ro[R + 1:] == nnz)
    for key in ("column_indices", "row_indices", "row_indices_t", "block_offsets_t"):
        assert np.array_equal(host(getattr(topo, key))[:nnz], tref[key]), key
    assert np.array_equal(host(topo.column_offsets_t), tref["column_offsets_t"])
    assert np.array_equal(host(topo.row_fill)[:R], tref["row_fill"])


@pytest.mark.parametrize("block", [64, 256])
@pytest.mark.parametrize("shape", [SMALL, MANY])
def test_products_block_sizes(block, shape, tile_n):
    """SDD (store / GELU / SwiGLU, both directions), DSD, DSD^T and DSTD on
    B x B blocks against the oracle's products at the same block size."""
    s = Setup(*shape, seed=70 + block, block=block)
    K, N = 256, 256
    B = block
    X = s.dense_rows(K)
    W1 = s.mat((K, s.E * s.F), 1.0 / np.sqrt(K))
    W3 = s.mat((K, s.E * s.F), 1.0 / np.sqrt(K))
    W2 = s.mat((s.E * s.F, K), 1.0 / np.sqrt(K))
    nnz = s.nnz
    # SDD store and GELU forward
    out = s.empty_blocks()
    dm.sdd(bf16_from_bits(X), bf16_from_bits(W1), K, s.topo, dm.EPI_STORE, out)
    ref = O.sdd(X[:s.P], W1, s.tp)
    assert_close(host(out)[:nnz], ref, TOL_SINGLE, RMS_SINGLE, "sdd")
    G, Aa = s.empty_blocks(), s.empty_blocks()
    dm.sdd(bf16_from_bits(X), bf16_from_bits(W1), K, s.topo, dm.EPI_GELU_FWD, G, Aa)
    assert_close(host(G)[:nnz], O.gelu_grad(ref), TOL_SINGLE, RMS_SINGLE, "gelu'")
    assert_close(host(Aa)[:nnz], O.gelu(ref), TOL_SINGLE, RMS_SINGLE, "gelu")
    # SwiGLU forward
    G1, G3, A3 = s.empty_blocks(), s.empty_blocks(), s.empty_blocks()
    dm.sdd(bf16_from_bits(X), bf16_from_bits(W1), K, s.topo, dm.EPI_SWIGLU_FWD, G1, G3, A3, B2=bf16_from_bits(W3))
    r3 = O.sdd(X[:s.P], W3, s.tp)
    assert_close(host(G1)[:nnz], r3 * O.silu_grad(ref), TOL_SINGLE, RMS_SINGLE, "H3 silu'(H1)")
    assert_close(host(A3)[:nnz], O.silu(ref) * r3, TOL_SINGLE, RMS_SINGLE, "silu(H1) H3")
    # backward SDD with the GELU factor (transposed weight)
    dY = s.dense_rows(K)
    Gb = s.blocks()
    dH = s.empty_blocks()
    dm.sdd(bf16_from_bits(dY), bf16_from_bits(W2), K, s.topo, dm.EPI_GELU_BWD, dH, b_trans=True,
           aux0=bf16_from_bits(Gb))
    ref_dh = O.sdd(dY[:s.P], W2, s.tp, b_trans=True) * O.bf16_to_f64(Gb[:nnz])
    assert_close(host(dH)[:nnz], ref_dh, TOL_SINGLE, RMS_SINGLE, "dH")
    # DSD, DSD^T, DSTD (both layouts)
    S = s.blocks(1.0 / 16)
    Wn = s.mat((s.E * s.F, N))
    C = torch.full((s.P_max, N), float("nan"), dtype=torch.bfloat16, device=dev())
    dm.dsd(s.topo, bf16_from_bits(S), bf16_from_bits(Wn), N, C)
    assert_close(host(C)[:s.P], O.dsd(S[:nnz], Wn, s.tp, s.P), TOL_SINGLE, RMS_SINGLE, "dsd")
    Wt = s.mat((N, s.E * s.F))
    Ct = torch.full((s.P_max, N), float("nan"), dtype=torch.bfloat16, device=dev())
    dm.dsd_t(s.topo, bf16_from_bits(S), bf16_from_bits(Wt), N, Ct)
    assert_close(host(Ct)[:s.P], O.dsd(S[:nnz], Wt, s.tp, s.P, w_trans=True), TOL_SINGLE, RMS_SINGLE, "dsd_t")
    D = s.dense_rows(N)
    for c_trans in (False, True):
        Cw = torch.full((N, s.E * s.F) if c_trans else (s.E * s.F, N), float("nan"), dtype=torch.bfloat16,
                        device=dev())
        dm.dstd(s.topo, bf16_from_bits(S), bf16_from_bits(D), N, Cw, c_trans=c_trans)
        assert_close(host(Cw), O.dstd(S[:nnz], D[:s.P], s.tp, c_trans=c_trans), TOL_SINGLE, RMS_SINGLE,
                     f"dstd c_trans={c_trans}")


@pytest.mark.parametrize("T,E,k,renorm,d", [(512, 4, 1, False, 256), (777, 8, 2, True, 512),
                                            (300, 64, 8, False, 136), (64, 3, 3, True, 8),
                                            (200, 16, 10, False, 264), (96, 8, 5, True, 3584)])
def test_unpermute_combine(T, E, k, renorm, d):
    ei, w = O.route_topk(syn.normal_f32(T, 1, (T, E)), k, renorm)
    pp = O.permute_pad(ei, E)
    P_max = syn.padded_rows_max(T, k, E)
    Yp = syn.normal_bf16(T, 2, (P_max, d))
    y = torch.full((T, d), float("nan"), dtype=torch.bfloat16, device=dev())
    dm.unpermute_combine(bf16_from_bits(Yp), i32(pp["dest_row"]), f32(w), T, k, y)
    ref = O.unpermute_combine(Yp, pp["dest_row"], w, T, k)
    assert_close(host(y), ref, TOL_SINGLE, RMS_SINGLE, "y")
    y1 = torch.empty_like(y)
    dm.unpermute_combine(bf16_from_bits(Yp), i32(pp["dest_row"]), None, T, k, y1)
    assert_close(host(y1), O.unpermute_combine(Yp, pp["dest_row"], None, T, k), TOL_SINGLE, RMS_SINGLE, "sum")


@pytest.mark.parametrize("k", [1, 3, 10])
def test_unpermute_combine_bad_row_reported(k):
    """An out-of-range source row is reported through the error word and its
    slot left out of the token's sum; every other token is unaffected."""
    T, E, d = 96, 16, 64
    ei, w = O.route_topk(syn.normal_f32(T, 7, (T, E)), k, False)
    pp = O.permute_pad(ei, E)
    P_max = syn.padded_rows_max(T, k, E)
    Yp = syn.normal_bf16(T, 8, (P_max, d))
    dest = pp["dest_row"].copy()
    dest[5 * k] = P_max  # token 5, slot 0
    y = torch.full((T, d), float("nan"), dtype=torch.bfloat16, device=dev())
    dm.unpermute_combine(bf16_from_bits(Yp), i32(dest), f32(w), T, k, y)
    torch.cuda.synchronize()
    assert dm.get_error(clear=True) == (4 << 8) | 5
    w_kept = np.array(w, dtype=np.float32).reshape(T, k).copy()
    w_kept[5, 0] = 0.0
    ref = O.unpermute_combine(Yp, pp["dest_row"], w_kept, T, k)
    assert_close(host(y), ref, TOL_SINGLE, RMS_SINGLE, "y")


@pytest.mark.parametrize("T,E,k,renorm,d", [(512, 4, 1, False, 256), (777, 8, 2, True, 512),
                                            (300, 64, 8, False, 136)])
def test_combine_backward(T, E, k, renorm, d):
    ei, w = O.route_topk(syn.normal_f32(T, 3, (T, E)), k, renorm)
    pp = O.permute_pad(ei, E)
    P_max = syn.padded_rows_max(T, k, E)
    Yp = syn.normal_bf16(T, 4, (P_max, d))
    dy = syn.normal_bf16(T, 5, (T, d))
    src = np.full(P_max, -1, dtype=np.int64)
    src[:pp["P"]] = pp["src_of_row"]
    dyp = torch.full((P_max, d), float("nan"), dtype=torch.bfloat16, device=dev())
    dg = torch.full((T, k), float("nan"), dtype=torch.float32, device=dev())
    P_dev = i32([pp["P"]])
    dm.combine_backward(bf16_from_bits(dy), bf16_from_bits(Yp), i32(src), f32(w), P_dev, k, P_max, dyp, dg)
    ref_dyp, ref_dg = O.combine_backward(dy, Yp[:pp["P"]], pp["src_of_row"], w, k)
    got = host(dyp)[:pp["P"]]
    assert_close(got, ref_dyp, TOL_SINGLE, RMS_SINGLE, "dy_perm")
    assert np.all(got[pp["src_of_row"] < 0] == 0)
    assert_close(host(dg), ref_dg, TOL_SINGLE, RMS_SINGLE, "d_gate")


def test_bad_expert_id_sets_device_error_word():
    """An out-of-range id is reported through the error word, not a trap."""
    T, E, d = 256, 4, 64
    ei = np.zeros((T, 1), dtype=np.int32)
    ei[17, 0] = 9
    P_max = dm.padded_rows_max(T, 1, E)
    z = lambda n, dt: torch.zeros(n, dtype=dt, device=dev())  # noqa: E731
    dest = z(T, torch.int32)
    dm.permute_pad(bf16_from_bits(syn.normal_bf16(1, 1, (T, d))), i32(ei), E, P_max, z(E, torch.int32),
                   z(E + 1, torch.int32), dest, z(P_max, torch.int32), z(P_max * d, torch.bfloat16).view(P_max, d),
                   z(1, torch.int32), z(dm.permute_pad_workspace_size(T, 1, E), torch.uint8))
    code = dm.get_error(clear=True)
    assert code == (2 << 8) | 5
    assert int(dest[17].item()) == -1


def test_permute_after_barrier_timeout_is_exact():
    """A permutation whose grid barrier timed out leaves its workspace ready:
    every block departs the barrier, waited or not, and the last one resets
    the counters, so the next call on the same workspace waits for all
    blocks again and is bit-exact (no GPU fault: the timed-out call's wait
    simply ends at its limit)."""
    cfg = syn.CONFIGS["fine"]
    ei, _ = O.route_topk(syn.make_logits(cfg), cfg.k, cfg.renorm)
    x_bits = syn.normal_bf16(1, 1, (cfg.T, 64))
    T, k, E = cfg.T, cfg.k, cfg.E
    P_max = dm.padded_rows_max(T, k, E)
    z = lambda n, dt: torch.zeros(max(1, n), dtype=dt, device=dev())  # noqa: E731
    out = dict(tpe=z(E, torch.int32), po=z(E + 1, torch.int32), dest=z(T * k, torch.int32),
               src=z(P_max, torch.int32), xp=z(P_max * 64, torch.bfloat16).view(P_max, 64), P=z(1, torch.int32),
               ws=z(dm.permute_pad_workspace_size(T, k, E), torch.uint8))
    x, eid = bf16_from_bits(x_bits), i32(ei).reshape(T, k)
    args = (x, eid, E, P_max, out["tpe"], out["po"], out["dest"], out["src"], out["xp"], out["P"], out["ws"])
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    dm.selftest_permute_timeout(*args, 2_000_000)
    t1.record()
    torch.cuda.synchronize()
    assert dm.get_error(clear=True) == (1 << 8) | 4  # DMOE_SITE_PERMUTE_BARRIER | DMOE_ERR_TIMEOUT
    assert 1.5 <= t0.elapsed_time(t1) <= 500.0  # ms: ended at its limit
    assert int(out["P"].item()) == 0 and int(out["tpe"].abs().sum().item()) == 0  # nothing past the barrier
    assert int(out["ws"][:256].abs().sum().item()) == 0  # counters reset
    for _ in range(2):
        dm.permute_pad(*args)
        torch.cuda.synchronize()
        assert dm.get_error(clear=True) == 0
        ref = O.permute_pad(ei, E)
        assert int(out["P"].item()) == ref["P"]
        assert np.array_equal(host(out["po"]), ref["padded_offsets"])
        assert np.array_equal(host(out["dest"]), ref["dest_row"])
        assert np.array_equal(host(out["src"])[:ref["P"]], ref["src_of_row"])


def test_bounded_wait_gives_up_and_reports():
    """A wait on a flag that nothing sets ends at its limit, reports
    DMOE_SITE_SELFTEST | DMOE_ERR_TIMEOUT through the error word, and the
    context stays usable (a router call afterwards is exact)."""
    dm.get_error(clear=True)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    dm.selftest_bounded_wait(2_000_000)
    t1.record()
    torch.cuda.synchronize()
    assert dm.get_error(clear=True) == (6 << 8) | 4
    assert 1.5 <= t0.elapsed_time(t1) <= 500.0  # ms: ended at its limit, not hung
    T, E, k = 300, 16, 2
    logits = syn.normal_f32(9, 1, (T, E))
    ei = torch.empty((T, k), dtype=torch.int32, device=dev())
    gw = torch.empty((T, k), dtype=torch.float32, device=dev())
    dm.route_topk(f32(logits), k, False, ei, gw)
    torch.cuda.synchronize()
    assert dm.get_error(clear=True) == 0
    ri, rw = O.route_topk(logits, k, False)
    assert np.array_equal(host(ei), ri) and np.max(np.abs(host(gw) - rw)) <= 1e-5
