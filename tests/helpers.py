"""Shared helpers of the GPU parity tests (test infrastructure)."""

import numpy as np
import torch

import oracle as O

# Float tolerances.  A single product of bf16 inputs with an fp32
# accumulator and a bf16 output differs from the exact fp64 value by the
# final bf16 rounding (half an ulp: 2^-9 of the element) plus fp32
# accumulation error (K * 2^-24 of the sum of |terms|): 4e-3 of max|ref| is
# a safe bound that still catches a lost K slice.  A chain of calls with
# bf16 intermediates uses the 2e-2 bound stated for outputs and gradients.
BLOCK_ROWS = 128
TOL_SINGLE = 4e-3
TOL_CHAIN = 2e-2
RMS_SINGLE = 2e-3
RMS_CHAIN = 1e-2


def dev():
    return torch.device("cuda:0")


def bf16_from_bits(bits) -> torch.Tensor:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(dev())


def bf16_from_f64(a) -> torch.Tensor:
    """Exact for values that are bf16-representable (oracle copies of inputs)."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64))
    return t.to(torch.bfloat16).to(dev())


def i32(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev())


def f32(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev())


def host(t) -> np.ndarray:
    return t.detach().to("cpu").double().numpy() if t.is_floating_point() else t.detach().to("cpu").numpy()


def rel_err(got, ref):
    """(max |got - ref| / max |ref|, rms(got - ref) / rms(ref))."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    scale = np.max(np.abs(ref))
    if scale == 0:
        return float(np.max(np.abs(got))), float(np.sqrt(np.mean(got ** 2)))
    rms = np.sqrt(np.mean(ref ** 2))
    return float(np.max(np.abs(got - ref)) / scale), float(np.sqrt(np.mean((got - ref) ** 2)) / rms)


def assert_close(got, ref, tol, rms_tol, what=""):
    m, r = rel_err(got, ref)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    assert m <= tol and r <= rms_tol, f"{what}: max rel {m:.3e} (tol {tol}), rms rel {r:.3e} (tol {rms_tol})"
    return m, r


def load_topology(topo, tp, P):
    """Write the oracle's topology into a device Topology (oracle -> GPU input)."""
    nnz = tp["nnz"]
    R = P // tp.get("block", 128)
    ro = np.full(topo.row_offsets.numel(), nnz, dtype=np.int64)
    ro[:R + 1] = tp["row_offsets"]
    topo.row_offsets.copy_(i32(ro))
    for name in ("column_indices", "row_indices", "row_indices_t", "block_offsets_t"):
        buf = getattr(topo, name)
        buf.zero_()
        if nnz:
            buf[:nnz].copy_(i32(tp[name]))
    topo.column_offsets_t.copy_(i32(tp["column_offsets_t"]))
    topo.nnz_dev.fill_(nnz)
    topo.P_dev.fill_(P)
    if topo.row_fill is not None:
        rf = np.zeros(topo.row_fill.numel(), dtype=np.int64)
        rf[:R] = tp["row_fill"] if "row_fill" in tp else BLOCK_ROWS
        topo.row_fill.copy_(i32(rf))


def counts_routing(counts, k=1):
    """expert_idx [T, k] whose slot-0 experts have the given counts (k = 1)."""
    assert k == 1
    return np.repeat(np.arange(len(counts)), counts).astype(np.int32)[:, None]


def oracle_blocks_bits(blocks64):
    return blocks64  # kept float64; converted with bf16_from_f64 when uploaded
