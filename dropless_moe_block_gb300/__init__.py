"""GB300 (sm_103a) dropless MoE block -- Python binding of ``libdmoe.so``.

Thin ctypes marshalling over the C ABI declared in ``include/dmoe.h``: each
function below has the name of the C entry point without the ``dmoe_``
prefix, takes torch tensors that already live on the GPU, checks their
dtype / shape / contiguity, and passes raw pointers and the current CUDA
stream.  All arithmetic runs in the library's CUDA kernels; there is no
Python or CPU fallback: a missing library or a non-sm_103 device raises.

``DMoELayer`` strings the calls into the forward and backward pass of one
dropless MoE layer (route -> permute+pad -> topology -> SDD(+act) -> DSD ->
combine, and the reverse), following section 1 of George Lin's blog post on
MoE training (MegaBlocks).  PyTorch only allocates device memory and
provides the stream.
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = [
    "DmoeError", "lib", "version", "padded_rows_max", "get_error", "launch_count", "set_tile_n", "set_pair",
    "Topology",
    "route_topk", "route_topk_backward", "permute_pad", "permute_pad_workspace_size", "build_topology", "dispatch", "sdd", "dsd", "dsd_t",
    "dstd", "unpermute_combine", "combine_backward", "DMoELayer", "StepRunner",
    "EPI_STORE", "EPI_GELU_FWD", "EPI_SWIGLU_FWD", "EPI_GELU_BWD", "EPI_SWIGLU_BWD", "BLOCK",
]

BLOCK = 128
EPI_STORE, EPI_GELU_FWD, EPI_SWIGLU_FWD, EPI_GELU_BWD, EPI_SWIGLU_BWD = range(5)

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libdmoe.so")

_STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "CUDA error", 4: "device wait timed out",
           5: "invalid data found on the device"}


class DmoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {_STATUS.get(status & 0xff, status)} (status {status})")
        self.status = status


class _Topo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "row_offsets", "column_indices", "row_indices", "column_offsets_t", "row_indices_t",
        "block_offsets_t", "nnz_dev", "P_dev", "row_fill")] + [
        (n, ctypes.c_int32) for n in ("E", "F", "P_max", "nnz_max", "block")]


_lib = None
_lock = threading.Lock()
_P = ctypes.c_void_p
_I = ctypes.c_int
_SIGS = {
    "dmoe_version": (ctypes.c_char_p, []),
    "dmoe_status_string": (ctypes.c_char_p, [_I]),
    "dmoe_padded_rows_max": (ctypes.c_int64, [_I, _I, _I]),
    "dmoe_padded_rows_max_block": (ctypes.c_int64, [_I, _I, _I, _I]),
    "dmoe_get_error": (_I, [ctypes.POINTER(ctypes.c_int32), _I]),
    "dmoe_launch_count": (ctypes.c_int64, []),
    "dmoe_set_tile_n": (_I, [_I]),
    "dmoe_set_pair": (_I, [_I]),
    "dmoe_route_topk": (_I, [_P, _I, _I, _I, _I, _P, _P, _P]),
    "dmoe_route_topk_backward": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P]),
    "dmoe_gate_route_topk": (_I, [_P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P]),
    "dmoe_selftest_bounded_wait": (_I, [ctypes.c_int64, _P]),
    "dmoe_selftest_permute_timeout": (_I, [_P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t,
                                           ctypes.c_int64, _P]),
    "dmoe_permute_pad_workspace_size": (ctypes.c_size_t, [_I, _I, _I]),
    "dmoe_permute_pad": (_I, [_P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "dmoe_permute_pad_block": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "dmoe_build_topology": (_I, [_P, _P, ctypes.POINTER(_Topo), _P]),
    "dmoe_dispatch": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.POINTER(_Topo),
                           _P, ctypes.c_size_t, _P]),
    "dmoe_sdd": (_I, [_P, _P, _P, _I, _I, ctypes.POINTER(_Topo), _I, _P, _P, _P, _P, _P, _P]),
    "dmoe_dsd": (_I, [ctypes.POINTER(_Topo), _P, _P, _I, _P, _P]),
    "dmoe_dsd_t": (_I, [ctypes.POINTER(_Topo), _P, _P, _P, _P, _I, _P, _P]),
    "dmoe_dstd": (_I, [ctypes.POINTER(_Topo), _P, _P, _I, _I, _P, _P]),
    "dmoe_unpermute_combine": (_I, [_P, _I, _P, _P, _I, _I, _I, _P, _P]),
    "dmoe_combine_backward": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P]),
}


def lib():
    """The loaded ``libdmoe.so`` (raises if it has not been built)."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(
                        f"{LIB_PATH} is missing: build it with `python -m dropless_moe_block_gb300.build`")
                h = ctypes.CDLL(LIB_PATH)
                for name, (res, args) in _SIGS.items():
                    f = getattr(h, name)
                    f.restype = res
                    f.argtypes = args
                _lib = h
    return _lib


def _check(fn: str, status: int):
    if status != 0:
        raise DmoeError(fn, status)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t, dtype, name, numel=None, shape=None):
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name} needs at least {numel} elements, has {t.numel()}")
    return t


def _opt(t, dtype, name, numel=None):
    return None if t is None else _need(t, dtype, name, numel)


# --------------------------------------------------------------------- utility

def version() -> str:
    return lib().dmoe_version().decode()


def padded_rows_max(T: int, k: int, E: int, block: int = BLOCK) -> int:
    return int(lib().dmoe_padded_rows_max_block(T, k, E, block))


def get_error(clear: bool = True) -> int:
    """Device error word (0 = none); synchronises the device."""
    v = ctypes.c_int32(0)
    _check("dmoe_get_error", lib().dmoe_get_error(ctypes.byref(v), int(clear)))
    return int(v.value)


def launch_count() -> int:
    return int(lib().dmoe_launch_count())


def selftest_bounded_wait(limit_ns: int, stream=None) -> None:
    """One warp waits, for limit_ns, on a device flag nothing sets, then
    records DMOE_SITE_SELFTEST | DMOE_ERR_TIMEOUT in the error word (the
    failure path of every bounded wait of the library)."""
    _check("dmoe_selftest_bounded_wait", lib().dmoe_selftest_bounded_wait(int(limit_ns), _stream(stream)))


def selftest_permute_timeout(x, expert_idx, E: int, P_max: int, tokens_per_expert, padded_offsets, dest_row,
                             src_of_row, x_perm, P_dev, ws, limit_ns: int, stream=None) -> None:
    """The permutation with a grid barrier that cannot complete: every block
    gives up after limit_ns, records DMOE_SITE_PERMUTE_BARRIER |
    DMOE_ERR_TIMEOUT, writes nothing past the barrier and leaves ``ws``
    ready for the next call."""
    T, d = x.shape
    k = expert_idx.shape[1]
    _need(x, torch.bfloat16, "x")
    _need(expert_idx, torch.int32, "expert_idx", shape=(T, k))
    _need(ws, torch.uint8, "ws")
    _check("dmoe_selftest_permute_timeout", lib().dmoe_selftest_permute_timeout(
        _ptr(x), _ptr(expert_idx), T, d, E, k, P_max, _ptr(tokens_per_expert), _ptr(padded_offsets), _ptr(dest_row),
        _ptr(src_of_row), _ptr(x_perm), _ptr(P_dev), _ptr(ws), ws.numel(), int(limit_ns), _stream(stream)))


def set_tile_n(bn: int) -> None:
    """0: tile width chosen per call; 128 / 256: forced where the shape allows."""
    _check("dmoe_set_tile_n", lib().dmoe_set_tile_n(int(bn)))


def set_pair(mode: int) -> None:
    """CTA pairs in the block-sparse products: 0 chosen per call, 1 never,
    2 wherever the shape allows (256 x 256 pair tiles), 3 wherever the shape
    allows, with 256 x 512 pair tiles where it allows those."""
    _check("dmoe_set_pair", lib().dmoe_set_pair(int(mode)))


# -------------------------------------------------------------------- topology

class Topology:
    """Device arrays of the hybrid BCSR-COO topology + transpose index."""

    def __init__(self, E: int, F: int, P_max: int, device="cuda", row_fill: bool = True, block: int = BLOCK):
        if block not in (64, 128, 256):
            raise ValueError("block must be 64, 128 or 256")
        if F % block or F % BLOCK or P_max % block:
            raise ValueError("F must be a multiple of 128 and of the block, P_max of the block")
        self.E, self.F, self.P_max, self.block = E, F, P_max, block
        nb = F // block
        self.nnz_max = (P_max // block) * nb
        i32 = dict(dtype=torch.int32, device=device)
        self.row_offsets = torch.zeros(P_max // block + 1, **i32)
        self.column_indices = torch.zeros(max(1, self.nnz_max), **i32)
        self.row_indices = torch.zeros(max(1, self.nnz_max), **i32)
        self.column_offsets_t = torch.zeros(E * nb + 1, **i32)
        self.row_indices_t = torch.zeros(max(1, self.nnz_max), **i32)
        self.block_offsets_t = torch.zeros(max(1, self.nnz_max), **i32)
        self.nnz_dev = torch.zeros(1, **i32)
        self.P_dev = torch.zeros(1, **i32)
        # rows holding tokens per row block: blocks with at most 64 run the
        # products with M = 64 (None: every block counts as full)
        self.row_fill = torch.zeros(max(1, P_max // block), **i32) if row_fill else None
        self._c = _Topo(*[t.data_ptr() if t is not None else None for t in (
            self.row_offsets, self.column_indices, self.row_indices, self.column_offsets_t, self.row_indices_t,
            self.block_offsets_t, self.nnz_dev, self.P_dev, self.row_fill)], E, F, P_max, self.nnz_max, block)

    @property
    def c(self):
        return ctypes.byref(self._c)

    def nnz(self) -> int:
        return int(self.nnz_dev.item())

    def P(self) -> int:
        return int(self.P_dev.item())


# ------------------------------------------------------------------ entry points

def route_topk(logits, k: int, renormalize: bool, expert_idx, gate_w, stream=None):
    T, E = logits.shape
    _need(logits, torch.float32, "logits")
    _need(expert_idx, torch.int32, "expert_idx", shape=(T, k))
    _need(gate_w, torch.float32, "gate_w", shape=(T, k))
    _check("dmoe_route_topk", lib().dmoe_route_topk(
        _ptr(logits), T, E, k, int(bool(renormalize)), _ptr(expert_idx), _ptr(gate_w), _stream(stream)))


def gate_route_topk(x, w_gate, k: int, renormalize: bool, logits, expert_idx, gate_w, stream=None):
    """Linear gate (logits = x . w_gate^T, w_gate [E, d]) fused into top-k routing."""
    T, d = x.shape
    E = w_gate.shape[0]
    _need(x, torch.bfloat16, "x", T * d)
    _need(w_gate, torch.bfloat16, "w_gate", E * d)
    _need(logits, torch.float32, "logits", shape=(T, E))
    _need(expert_idx, torch.int32, "expert_idx", shape=(T, k))
    _need(gate_w, torch.float32, "gate_w", shape=(T, k))
    _check("dmoe_gate_route_topk", lib().dmoe_gate_route_topk(
        _ptr(x), _ptr(w_gate), T, d, E, k, int(bool(renormalize)), _ptr(logits), _ptr(expert_idx), _ptr(gate_w),
        _stream(stream)))


def route_topk_backward(logits, expert_idx, gate_w, d_gate, renormalize: bool, d_logits, stream=None):
    T, E = logits.shape
    k = expert_idx.shape[1]
    _need(logits, torch.float32, "logits")
    _need(expert_idx, torch.int32, "expert_idx", shape=(T, k))
    _need(gate_w, torch.float32, "gate_w", shape=(T, k))
    _need(d_gate, torch.float32, "d_gate", shape=(T, k))
    _need(d_logits, torch.float32, "d_logits", shape=(T, E))
    _check("dmoe_route_topk_backward", lib().dmoe_route_topk_backward(
        _ptr(logits), _ptr(expert_idx), _ptr(gate_w), _ptr(d_gate), T, E, k, int(bool(renormalize)),
        _ptr(d_logits), _stream(stream)))


def permute_pad_workspace_size(T: int, k: int, E: int) -> int:
    return int(lib().dmoe_permute_pad_workspace_size(T, k, E))


def permute_pad(x, expert_idx, E: int, P_max: int, tokens_per_expert, padded_offsets, dest_row, src_of_row,
                x_perm, P_dev, ws, block: int = BLOCK, stream=None):
    T, d = x.shape
    k = expert_idx.shape[1]
    _need(x, torch.bfloat16, "x")
    _need(expert_idx, torch.int32, "expert_idx", shape=(T, k))
    _need(tokens_per_expert, torch.int32, "tokens_per_expert", E)
    _need(padded_offsets, torch.int32, "padded_offsets", E + 1)
    _need(dest_row, torch.int32, "dest_row", T * k)
    _need(src_of_row, torch.int32, "src_of_row", P_max)
    _need(x_perm, torch.bfloat16, "x_perm", P_max * d)
    _need(P_dev, torch.int32, "P_dev", 1)
    _need(ws, torch.uint8, "ws")
    if block == BLOCK:
        _check("dmoe_permute_pad", lib().dmoe_permute_pad(
            _ptr(x), _ptr(expert_idx), T, d, E, k, P_max, _ptr(tokens_per_expert), _ptr(padded_offsets),
            _ptr(dest_row), _ptr(src_of_row), _ptr(x_perm), _ptr(P_dev), _ptr(ws), ws.numel(), _stream(stream)))
    else:
        _check("dmoe_permute_pad_block", lib().dmoe_permute_pad_block(
            _ptr(x), _ptr(expert_idx), T, d, E, k, block, P_max, _ptr(tokens_per_expert), _ptr(padded_offsets),
            _ptr(dest_row), _ptr(src_of_row), _ptr(x_perm), _ptr(P_dev), _ptr(ws), ws.numel(), _stream(stream)))


def build_topology(padded_offsets, topo: Topology, tokens_per_expert=None, stream=None):
    """Topology from the padded offsets; with ``tokens_per_expert`` also the
    row fill (``topo.row_fill``)."""
    _need(padded_offsets, torch.int32, "padded_offsets", topo.E + 1)
    _opt(tokens_per_expert, torch.int32, "tokens_per_expert", topo.E)
    _check("dmoe_build_topology", lib().dmoe_build_topology(_ptr(padded_offsets), _ptr(tokens_per_expert), topo.c,
                                                            _stream(stream)))


def dispatch(logits, x, k: int, renormalize: bool, expert_idx, gate_w, tokens_per_expert, padded_offsets, dest_row,
             src_of_row, x_perm, P_dev, ws, P_max: int, topo: Topology = None, stream=None):
    """route_topk + permute_pad (+ build_topology when ``topo`` is given) in
    one launch, with the results of the separate calls."""
    T, d = x.shape
    E = logits.shape[1]
    if topo is not None and (topo.E != E or topo.P_max != P_max):
        raise ValueError("topo was built for another E or P_max")
    _need(logits, torch.float32, "logits", T * E)
    _need(x, torch.bfloat16, "x")
    _need(expert_idx, torch.int32, "expert_idx", T * k)
    _need(gate_w, torch.float32, "gate_w", T * k)
    _need(tokens_per_expert, torch.int32, "tokens_per_expert", E)
    _need(padded_offsets, torch.int32, "padded_offsets", E + 1)
    _need(dest_row, torch.int32, "dest_row", T * k)
    _need(src_of_row, torch.int32, "src_of_row", P_max)
    _need(x_perm, torch.bfloat16, "x_perm", P_max * d)
    _need(P_dev, torch.int32, "P_dev", 1)
    _need(ws, torch.uint8, "ws")
    _check("dmoe_dispatch", lib().dmoe_dispatch(
        _ptr(logits), _ptr(x), T, d, E, k, int(bool(renormalize)), P_max, _ptr(expert_idx), _ptr(gate_w),
        _ptr(tokens_per_expert), _ptr(padded_offsets), _ptr(dest_row), _ptr(src_of_row), _ptr(x_perm), _ptr(P_dev),
        topo.c if topo is not None else None, _ptr(ws), ws.numel(), _stream(stream)))


def sdd(A, B, K: int, topo: Topology, epilogue: int, out0, out1=None, out2=None, B2=None, b_trans=False,
        aux0=None, aux1=None, stream=None):
    blk = topo.nnz_max * topo.block * topo.block
    _need(A, torch.bfloat16, "A", topo.P_max * K)
    _need(B, torch.bfloat16, "B", topo.E * topo.F * K)
    _opt(B2, torch.bfloat16, "B2", topo.E * topo.F * K)
    for n, t in (("aux0", aux0), ("aux1", aux1), ("out0", out0), ("out1", out1), ("out2", out2)):
        _opt(t, torch.bfloat16, n, blk)
    _check("dmoe_sdd", lib().dmoe_sdd(
        _ptr(A), _ptr(B), _ptr(B2), K, int(bool(b_trans)), topo.c, epilogue, _ptr(aux0), _ptr(aux1), _ptr(out0),
        _ptr(out1), _ptr(out2), _stream(stream)))


def dsd(topo: Topology, S, Bm, N: int, C, stream=None):
    _need(S, torch.bfloat16, "S", topo.nnz_max * topo.block * topo.block)
    _need(Bm, torch.bfloat16, "Bm", topo.E * topo.F * N)
    _need(C, torch.bfloat16, "C", topo.P_max * N)
    _check("dmoe_dsd", lib().dmoe_dsd(topo.c, _ptr(S), _ptr(Bm), N, _ptr(C), _stream(stream)))


def dsd_t(topo: Topology, S, Bm, N: int, C, S2=None, Bm2=None, stream=None):
    _need(S, torch.bfloat16, "S", topo.nnz_max * topo.block * topo.block)
    _need(Bm, torch.bfloat16, "Bm", topo.E * topo.F * N)
    _opt(S2, torch.bfloat16, "S2", topo.nnz_max * topo.block * topo.block)
    _opt(Bm2, torch.bfloat16, "Bm2", topo.E * topo.F * N)
    _need(C, torch.bfloat16, "C", topo.P_max * N)
    _check("dmoe_dsd_t", lib().dmoe_dsd_t(topo.c, _ptr(S), _ptr(Bm), _ptr(S2), _ptr(Bm2), N, _ptr(C),
                                          _stream(stream)))


def dstd(topo: Topology, S, D, N: int, C, c_trans=False, stream=None):
    _need(S, torch.bfloat16, "S", topo.nnz_max * topo.block * topo.block)
    _need(D, torch.bfloat16, "D", topo.P_max * N)
    _need(C, torch.bfloat16, "C", topo.E * topo.F * N)
    _check("dmoe_dstd", lib().dmoe_dstd(topo.c, _ptr(S), _ptr(D), N, int(bool(c_trans)), _ptr(C), _stream(stream)))


def unpermute_combine(y_perm, dest_row, gate_w, T: int, k: int, y, stream=None):
    d = y.shape[1]
    _need(y_perm, torch.bfloat16, "y_perm")
    _need(dest_row, torch.int32, "dest_row", T * k)
    _opt(gate_w, torch.float32, "gate_w", T * k)
    _need(y, torch.bfloat16, "y", T * d)
    n_rows = y_perm.numel() // d
    _check("dmoe_unpermute_combine", lib().dmoe_unpermute_combine(
        _ptr(y_perm), n_rows, _ptr(dest_row), _ptr(gate_w), T, d, k, _ptr(y), _stream(stream)))


def combine_backward(dy, y_perm, src_of_row, gate_w, P_dev, k: int, P_max: int, dy_perm, d_gate=None,
                     stream=None):
    T, d = dy.shape
    _need(dy, torch.bfloat16, "dy")
    _opt(y_perm, torch.bfloat16, "y_perm", P_max * d)
    _need(src_of_row, torch.int32, "src_of_row", P_max)
    _opt(gate_w, torch.float32, "gate_w", T * k)
    _need(P_dev, torch.int32, "P_dev", 1)
    _need(dy_perm, torch.bfloat16, "dy_perm", P_max * d)
    _opt(d_gate, torch.float32, "d_gate", T * k)
    _check("dmoe_combine_backward", lib().dmoe_combine_backward(
        _ptr(dy), _ptr(y_perm), _ptr(src_of_row), _ptr(gate_w), _ptr(P_dev), T, d, k, P_max, _ptr(dy_perm),
        _ptr(d_gate), _stream(stream)))


# ----------------------------------------------------------------- whole layer

class DMoELayer:
    """Buffers and call sequence of one dropless MoE layer (fwd + bwd).

    Weights: ``w1`` (and ``w3`` for SwiGLU) bf16 [d, E*F], ``w2`` bf16
    [E*F, d].  With ``depth`` = L > 1 every expert is a stack of L
    SDD -> activation -> DSD blocks applied to its permuted rows in turn
    (h_l = act(h_{l-1} W1_l) W2_l), and the weights are lists of L tensors.
    Every intermediate lives in a preallocated device buffer sized for the
    worst-case padding (P_max), so a step never allocates.
    """

    def __init__(self, T: int, d: int, E: int, F: int, k: int, act: str = "gelu", renormalize: bool = False,
                 device="cuda", front: str = "separate", depth: int = 1, block: int = BLOCK):
        if act not in ("gelu", "swiglu"):
            raise ValueError(act)
        if depth < 1:
            raise ValueError("depth must be >= 1")
        self.depth = depth
        # block size of the format: 128 (the page's), 64 or 256 (its ablation)
        self.block = block
        self.T, self.d, self.E, self.F, self.k = T, d, E, F, k
        self.act, self.renormalize = act, renormalize
        # the calls before the first product: "separate" (three launches, the
        # default: in a captured step the small router and topology kernels
        # overlap their neighbours through programmatic dependent launch),
        # "route_permute" (route + permute in one launch, then the topology
        # kernel) or "fused" (route + permute + topology in one launch)
        if front not in self.FRONTS:
            raise ValueError(front)
        if block != BLOCK and front == "route_permute":
            raise ValueError("the route_permute front pads to 128 rows; use separate or fused")
        self.front = front
        self.P_max = padded_rows_max(T, k, E, block)
        self.topo = Topology(E, F, self.P_max, device, block=block)
        nnz_max = self.topo.nnz_max
        A = T * k
        bf, i32, f32 = torch.bfloat16, torch.int32, torch.float32
        dev = dict(device=device)
        z = lambda *s, dtype: torch.zeros(*s, dtype=dtype, **dev)  # noqa: E731
        self.expert_idx = z(T, k, dtype=i32)
        self.gate_w = z(T, k, dtype=f32)
        self.tokens_per_expert = z(E, dtype=i32)
        self.padded_offsets = z(E + 1, dtype=i32)
        self.dest_row = z(max(1, A), dtype=i32)
        self.src_of_row = z(max(1, self.P_max), dtype=i32)
        self.P_dev = z(1, dtype=i32)
        self.ws = z(max(16, permute_pad_workspace_size(T, k, E)), dtype=torch.uint8)
        self.x_perm = z(max(1, self.P_max), d, dtype=bf)
        blocks = lambda: z(max(1, nnz_max), block, block, dtype=bf)  # noqa: E731
        rows = lambda: z(max(1, self.P_max), d, dtype=bf)  # noqa: E731
        swi = act == "swiglu"
        L = depth
        # per expert block l: the derivative factors of the activation, stored
        # by the forward SDD for the backward one (gelu'(H); for SwiGLU
        # H3 silu'(H1) and silu(H1)), the activation, and the backward blocks
        self.Gs = [blocks() for _ in range(L)]
        self.G3s = [blocks() for _ in range(L)] if swi else [None] * L
        self.As = [blocks() for _ in range(L)]
        self.dHs = [blocks() for _ in range(L)]
        self.dH3s = [blocks() for _ in range(L)] if swi else [None] * L
        # permuted rows: h_0 = x_perm, h_l = output of block l (h_L = y_perm);
        # g_l = gradient w.r.t. h_l (g_L = dy_perm, g_0 = dx_perm)
        self.hs = [self.x_perm] + [rows() for _ in range(L)]
        self.gs = [rows() for _ in range(L + 1)]
        self.y = z(T, d, dtype=bf)
        self.d_gate = z(T, k, dtype=f32)
        self.dx = z(T, d, dtype=bf)
        self.d_logits = z(T, E, dtype=f32)
        self.gate_logits = z(T, E, dtype=f32)  # written when the layer runs its own linear gate
        self.dW1s = [z(d, E * F, dtype=bf) for _ in range(L)]
        self.dW3s = [z(d, E * F, dtype=bf) for _ in range(L)] if swi else [None] * L
        self.dW2s = [z(E * F, d, dtype=bf) for _ in range(L)]
        # one-block names
        self.G, self.G3, self.Aact = self.Gs[0], self.G3s[0], self.As[0]
        self.dH, self.dH3 = self.dHs[0], self.dH3s[0]
        self.y_perm, self.dy_perm, self.dx_perm = self.hs[L], self.gs[L], self.gs[0]
        self.dW1, self.dW3, self.dW2 = self.dW1s[0], self.dW3s[0], self.dW2s[0]

    FRONTS = ("fused", "route_permute", "separate")

    # each entry of the two lists is one C-ABI call (one kernel launch)
    def forward_calls(self, x, logits, w1, w2, w3=None, w_gate=None):
        """With ``w_gate`` ([E, d] bf16) the layer computes the router logits
        itself (``gate_route_topk``, into ``self.gate_logits``) and ``logits``
        is not read; the gradient of the gate's own GEMM is the caller's
        (``self.d_logits`` . w_gate into dx, d_logits^T . x for w_gate)."""
        T, d, E, F, k = self.T, self.d, self.E, self.F, self.k
        swi = self.act == "swiglu"
        if w_gate is not None:
            if self.front != "separate":
                raise ValueError("a layer with its own gate runs the separate front")
            logits = self.gate_logits
        self._logits = logits  # the router backward reads them
        if self.front != "separate":
            fused = self.front == "fused"
            front = [("dispatch", lambda: dispatch(logits, x, k, self.renormalize, self.expert_idx, self.gate_w,
                                                   self.tokens_per_expert, self.padded_offsets, self.dest_row,
                                                   self.src_of_row, self.x_perm, self.P_dev, self.ws, self.P_max,
                                                   self.topo if fused else None))]
            if not fused:
                front.append(("build_topology", lambda: build_topology(self.padded_offsets, self.topo,
                                                                       self.tokens_per_expert)))
        else:
            front = [
                ("gate_route_topk", lambda: gate_route_topk(x, w_gate, k, self.renormalize, self.gate_logits,
                                                            self.expert_idx, self.gate_w))
                if w_gate is not None else
                ("route_topk", lambda: route_topk(logits, k, self.renormalize, self.expert_idx, self.gate_w)),
                ("permute_pad", lambda: permute_pad(x, self.expert_idx, E, self.P_max, self.tokens_per_expert,
                                                    self.padded_offsets, self.dest_row, self.src_of_row,
                                                    self.x_perm, self.P_dev, self.ws, block=self.block)),
                ("build_topology", lambda: build_topology(self.padded_offsets, self.topo, self.tokens_per_expert)),
            ]
        calls = list(front)
        w1s, w2s, w3s = self._weights(w1, w2, w3)
        for l in range(self.depth):
            sfx = self._sfx(l)
            calls.append(("sdd_fwd" + sfx, (lambda l=l: sdd(self.hs[l], w1s[l], d, self.topo, EPI_SWIGLU_FWD,
                                                            self.Gs[l], self.G3s[l], self.As[l], B2=w3s[l]))
                          if swi else
                          (lambda l=l: sdd(self.hs[l], w1s[l], d, self.topo, EPI_GELU_FWD, self.Gs[l], self.As[l]))))
            calls.append(("dsd_fwd" + sfx, lambda l=l: dsd(self.topo, self.As[l], w2s[l], d, self.hs[l + 1])))
        calls.append(("unpermute_combine", lambda: unpermute_combine(self.y_perm, self.dest_row, self.gate_w, T, k,
                                                                     self.y)))
        return calls

    def backward_calls(self, dy, x, w1, w2, w3=None):
        T, d, k = self.T, self.d, self.k
        swi = self.act == "swiglu"
        logits = self._logits
        w1s, w2s, w3s = self._weights(w1, w2, w3)
        calls = [
            ("combine_backward", lambda: combine_backward(dy, self.y_perm, self.src_of_row, self.gate_w,
                                                          self.P_dev, k, self.P_max, self.dy_perm, self.d_gate)),
            ("route_backward", lambda: route_topk_backward(logits, self.expert_idx, self.gate_w, self.d_gate,
                                                           self.renormalize, self.d_logits)),
        ]
        for l in reversed(range(self.depth)):  # g_{l+1} -> dH_l -> g_l, dW*_l
            sfx = self._sfx(l)
            g_in, g_out = self.gs[l + 1], self.gs[l]
            calls += [
                ("sdd_bwd" + sfx, (lambda l=l, g_in=g_in: sdd(g_in, w2s[l], d, self.topo, EPI_SWIGLU_BWD, self.dHs[l],
                                                              self.dH3s[l], b_trans=True, aux0=self.Gs[l],
                                                              aux1=self.G3s[l])) if swi else
                 (lambda l=l, g_in=g_in: sdd(g_in, w2s[l], d, self.topo, EPI_GELU_BWD, self.dHs[l], b_trans=True,
                                             aux0=self.Gs[l]))),
                ("dstd_dw2" + sfx, lambda l=l, g_in=g_in: dstd(self.topo, self.As[l], g_in, d, self.dW2s[l])),
                ("dsd_t_dx" + sfx, (lambda l=l, g_out=g_out: dsd_t(self.topo, self.dHs[l], w1s[l], d, g_out,
                                                                   S2=self.dH3s[l], Bm2=w3s[l])) if swi else
                 (lambda l=l, g_out=g_out: dsd_t(self.topo, self.dHs[l], w1s[l], d, g_out))),
                ("dstd_dw1" + sfx, lambda l=l: dstd(self.topo, self.dHs[l], self.hs[l], d, self.dW1s[l],
                                                    c_trans=True)),
            ]
            if swi:
                calls.append(("dstd_dw3" + sfx, lambda l=l: dstd(self.topo, self.dH3s[l], self.hs[l], d,
                                                                 self.dW3s[l], c_trans=True)))
        calls.append(("unpermute_dx", lambda: unpermute_combine(self.dx_perm, self.dest_row, None, T, k, self.dx)))
        return calls

    def _sfx(self, l: int) -> str:
        """Call-name suffix of expert block l (none for a one-block layer)."""
        return "" if self.depth == 1 else f"_{l + 1}"

    def _weights(self, w1, w2, w3):
        def blocks(w, name):
            if w is None:
                return [None] * self.depth
            ws = list(w) if isinstance(w, (list, tuple)) else [w]
            if len(ws) != self.depth:
                raise ValueError(f"{name}: {len(ws)} blocks given, depth is {self.depth}")
            return ws
        if self.act == "swiglu" and w3 is None:
            raise ValueError("SwiGLU needs w3")
        return blocks(w1, "w1"), blocks(w2, "w2"), blocks(w3, "w3")

    # calls that may run on a second stream: each waits only for the
    # main-stream call that produced what it reads (the forward combine needs
    # the last block's output and nothing in the backward reads y; the router
    # backward needs d_gate; DSTD dW2 of block l needs the gradient w.r.t.
    # that block's output but not dH; DSTD dW1 / dW3 need dH but not the
    # block's input gradient)
    def _side_dep(self, name: str):
        if name == "unpermute_combine":
            return "dsd_fwd" + self._sfx(self.depth - 1)
        if name == "route_backward":
            return "combine_backward"
        for base in ("dstd_dw2", "dstd_dw1", "dstd_dw3"):
            if name == base or name.startswith(base + "_"):
                l = int(name[len(base) + 1:]) - 1 if name != base else 0
                if base != "dstd_dw2":
                    return "sdd_bwd" + self._sfx(l)
                return "combine_backward" if l == self.depth - 1 else "dsd_t_dx" + self._sfx(l + 1)
        return None

    # second-stream calls a main-stream call waits for: the forward combine
    # overlaps the combine backward only, and the backward SDD (a persistent
    # kernel that wants every SM) starts once both have left the GPU
    def _main_waits(self, name: str):
        if name == "sdd_bwd" + self._sfx(self.depth - 1):
            return ("unpermute_combine",)
        return ()

    def run(self, calls, side=None):
        """Issues ``calls`` on the current stream, in order.  With a ``side``
        stream, the calls ``_side_dep`` names go to it as soon as the call
        they read from has been issued, and the side stream rejoins the
        current stream at the end: independent products then fill each
        other's last wave."""
        if side is None:
            for _, f in calls:
                f()
            return
        main = torch.cuda.current_stream()
        deps = {name: self._side_dep(name) for name, _ in calls}
        needed = {dep for dep in deps.values() if dep is not None}
        marks = {}
        side_marks = {}
        waited = {w for name, _ in calls for w in self._main_waits(name)}
        forked = False
        for name, f in calls:
            dep = deps[name]
            if dep is not None and dep in marks:
                side.wait_event(marks[dep])
                forked = True
                with torch.cuda.stream(side):
                    f()
                if name in waited:
                    ev = torch.cuda.Event()
                    ev.record(side)
                    side_marks[name] = ev
            else:
                for w in self._main_waits(name):
                    if w in side_marks:
                        main.wait_event(side_marks[w])
                f()
                if name in needed:
                    ev = torch.cuda.Event()
                    ev.record(main)
                    marks[name] = ev
        if forked:
            join = torch.cuda.Event()
            join.record(side)
            main.wait_event(join)

    def capture(self, x, logits, w1, w2, w3=None, dy=None, events=None, concurrent=False, w_gate=None):
        """Records the forward pass (and the backward one when ``dy`` is given)
        into a CUDA graph; ``graph.replay()`` then runs every call as one launch
        on the current stream.  ``events`` (optional, len(calls) + 1 events
        created with ``external=True``) are recorded before the first call and
        after each call (sequential graph).  ``concurrent`` puts the
        forward combine and the independent backward products on a second
        stream inside the graph (see ``run``).  Returns (graph, number of kernels in the graph).
        The inputs are read from the same tensors at every replay."""
        calls = self.forward_calls(x, logits, w1, w2, w3, w_gate)
        if dy is not None:
            calls += self.backward_calls(dy, x, w1, w2, w3)
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):  # first run: per-kernel attributes, tensor maps
            for _, f in calls:
                f()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        n0 = launch_count()
        with torch.cuda.graph(graph, capture_error_mode="thread_local"):
            if events is not None:
                events[0].record()
                for i, (_, f) in enumerate(calls):
                    f()
                    events[i + 1].record()
            else:
                self.run(calls, side if concurrent else None)
        return graph, launch_count() - n0

    def forward(self, x, logits, w1, w2, w3=None, w_gate=None):
        for _, f in self.forward_calls(x, logits, w1, w2, w3, w_gate):
            f()
        return self.y

    def backward(self, dy, x, w1, w2, w3=None):
        for _, f in self.backward_calls(dy, x, w1, w2, w3):
            f()
        return self.dx


class StepRunner:
    """Fwd + bwd steps of a ``DMoELayer`` fed from host memory, with the
    host <-> device copies overlapped with compute: the inputs of step s+1
    are copied in (their own stream) while step s computes, and the results
    of step s are copied out (a third stream) while step s+1 computes.  Two
    device slots hold the inputs and two the results; each input slot has
    its own captured graph of the whole step.  Each step returns y, dx,
    d_gate and d_logits (the gradient the caller needs for the gate GEMM);
    weights and weight gradients stay on the device.  With ``w_gate`` the
    layer computes its router logits itself and no logits are copied in.
    """

    RESULTS = ("y", "dx", "d_gate", "d_logits")

    def __init__(self, layer: "DMoELayer", w1, w2, w3=None, w_gate=None):
        self.layer = layer
        T, d, E, k = layer.T, layer.d, layer.E, layer.k
        dev = layer.y.device
        bf = torch.bfloat16
        self.x = [torch.zeros(T, d, dtype=bf, device=dev) for _ in range(2)]
        self.gated = w_gate is not None
        self.logits = [None if self.gated else torch.zeros(T, E, dtype=torch.float32, device=dev) for _ in range(2)]
        self.dy = [torch.zeros(T, d, dtype=bf, device=dev) for _ in range(2)]
        # each slot's graph writes its step's results straight into that
        # slot's buffers (the layer's own result tensors are swapped out
        # while the graph is captured), so no device copy follows a step
        self.out = [tuple(torch.empty_like(getattr(layer, n)) for n in self.RESULTS) for _ in range(2)]
        own = tuple(getattr(layer, n) for n in self.RESULTS)
        self.graphs = []
        try:
            for i in range(2):
                for n, t in zip(self.RESULTS, self.out[i]):
                    setattr(layer, n, t)
                self.graphs.append(layer.capture(self.x[i], self.logits[i], w1, w2, w3, dy=self.dy[i],
                                                 concurrent=True, w_gate=w_gate)[0])
        finally:
            for n, t in zip(self.RESULTS, own):
                setattr(layer, n, t)
        self.h2d = torch.cuda.Stream(device=dev)
        self.d2h = torch.cuda.Stream(device=dev)
        ev = lambda: [torch.cuda.Event() for _ in range(2)]  # noqa: E731
        self.in_ready, self.in_free, self.out_ready, self.out_free = ev(), ev(), ev(), ev()
        self.steps_issued = 0

    def host_outputs(self):
        """Two pinned host result sets (y, dx, d_gate, d_logits) for ``run``."""
        return [tuple(torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in self.out[0]) for _ in range(2)]

    def run(self, host_x, host_logits, host_dy, host_out, steps: int):
        """Issues ``steps`` steps on the current stream (asynchronously): each
        copies host_x / host_logits / host_dy (pinned) in and leaves its y,
        dx, d_gate and d_logits in host_out[s % 2] (host_logits is not read
        with a gate).  Call ``finish()`` (or synchronise)
        before reading host memory."""
        comp = torch.cuda.current_stream()
        for _ in range(steps):
            i = self.steps_issued & 1
            self.h2d.wait_event(self.in_free[i])  # step s-2 has read slot i
            with torch.cuda.stream(self.h2d):
                self.x[i].copy_(host_x, non_blocking=True)
                if not self.gated:
                    self.logits[i].copy_(host_logits, non_blocking=True)
                self.dy[i].copy_(host_dy, non_blocking=True)
                self.in_ready[i].record()
            comp.wait_event(self.in_ready[i])
            comp.wait_event(self.out_free[i])  # step s-2's results have left slot i
            self.graphs[i].replay()
            self.in_free[i].record(comp)
            self.out_ready[i].record(comp)
            self.d2h.wait_event(self.out_ready[i])
            with torch.cuda.stream(self.d2h):
                for dst, src in zip(host_out[i], self.out[i]):
                    dst.copy_(src, non_blocking=True)
                self.out_free[i].record()
            self.steps_issued += 1

    def finish(self):
        """Makes the current stream wait for every copy issued so far."""
        comp = torch.cuda.current_stream()
        comp.wait_stream(self.h2d)
        comp.wait_stream(self.d2h)
