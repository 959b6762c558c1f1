"""The C-ABI library builds, loads without a GPU and exports what dmoe.h declares.

No compute call runs here: only host-side validation paths, which return
DMOE_ERR_INVALID_ARG before any CUDA call, and the host-only utilities.
"""

import ctypes
import os
import re
import subprocess

import pytest

import dmoe_synth as syn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dmoe.h")


@pytest.fixture(scope="module")
def libpath():
    from dropless_moe_block_gb300 import build
    return build.build()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dmoe_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_eight_calls_and_helpers():
    names = _declared()
    for n in ("dmoe_route_topk", "dmoe_permute_pad", "dmoe_build_topology", "dmoe_sdd", "dmoe_dsd",
              "dmoe_dsd_t", "dmoe_dstd", "dmoe_unpermute_combine", "dmoe_combine_backward"):
        assert n in names


def test_exports_match_header(libpath):
    out = subprocess.run(["nm", "-D", "--defined-only", libpath], capture_output=True, text=True, check=True).stdout
    exported = sorted(line.split()[-1] for line in out.splitlines() if " T " in line)
    assert exported == _declared()


def test_loads_and_host_utilities(libpath):
    import dropless_moe_block_gb300 as dm
    assert "sm_103a" in dm.version()
    L = dm.lib()
    for s in range(6):
        assert L.dmoe_status_string(s)
    for (T, k, E) in ((0, 1, 4), (1, 1, 1), (512, 1, 4), (8192, 2, 8), (4096, 8, 64), (3, 2, 1000)):
        assert dm.padded_rows_max(T, k, E) == syn.padded_rows_max(T, k, E)


def test_invalid_arguments_rejected_without_gpu(libpath):
    import dropless_moe_block_gb300 as dm
    L = dm.lib()
    fake = ctypes.c_void_p(0x1000)
    odd = ctypes.c_void_p(0x1008)
    s = None
    # k > E, E > 1024, null pointers
    assert L.dmoe_route_topk(fake, 4, 4, 5, 0, fake, fake, s) == 1
    assert L.dmoe_route_topk(fake, 4, 1025, 1, 0, fake, fake, s) == 1
    assert L.dmoe_route_topk(None, 4, 4, 1, 0, fake, fake, s) == 1
    # gate: d not a multiple of 64, E > 256, k > E, misaligned x, null output
    assert L.dmoe_gate_route_topk(fake, fake, 4, 96, 8, 1, 0, fake, fake, fake, s) == 1
    assert L.dmoe_gate_route_topk(fake, fake, 4, 128, 257, 1, 0, fake, fake, fake, s) == 1
    assert L.dmoe_gate_route_topk(fake, fake, 4, 128, 8, 9, 0, fake, fake, fake, s) == 1
    assert L.dmoe_gate_route_topk(odd, fake, 4, 128, 8, 2, 0, fake, fake, fake, s) == 1
    assert L.dmoe_gate_route_topk(fake, fake, 4, 128, 8, 2, 0, None, fake, fake, s) == 1
    assert L.dmoe_gate_route_topk(None, None, 0, 128, 8, 2, 0, None, None, None, s) == 0
    # settings: tile width and CTA-pair mode outside their values
    assert L.dmoe_set_tile_n(192) == 1 and L.dmoe_set_pair(4) == 1 and L.dmoe_set_pair(-1) == 1
    assert L.dmoe_set_pair(0) == 0 and L.dmoe_set_tile_n(0) == 0
    # bounded-wait self-test: limit outside [1 us, 1 s]
    assert L.dmoe_selftest_bounded_wait(999, s) == 1
    assert L.dmoe_selftest_bounded_wait(2 * 10**9, s) == 1
    # barrier self-test: limit outside [1 us, 1 s]
    pargs = [fake, fake, 16, 16, 4, 1, 512, fake, fake, fake, fake, fake, fake, fake, 1 << 20, 999, s]
    assert L.dmoe_selftest_permute_timeout(*pargs) == 1
    pargs[15] = 2 * 10**9
    assert L.dmoe_selftest_permute_timeout(*pargs) == 1
    # permute: d not a multiple of 8, P_max too small, misaligned x
    args = [fake, fake, 16, 12, 4, 1, 512, fake, fake, fake, fake, fake, fake, fake, 1 << 20, s]
    assert L.dmoe_permute_pad(*args) == 1
    args[3] = 16
    args[6] = 128
    assert L.dmoe_permute_pad(*args) == 1
    args[6] = 512
    args[0] = odd
    assert L.dmoe_permute_pad(*args) == 1
    # topology: F not a multiple of 128, inconsistent nnz_max
    t = dm._Topo(*([0x1000] * 9), 4, 200, 512, 8)
    assert L.dmoe_build_topology(fake, None, ctypes.byref(t), s) == 1
    t = dm._Topo(*([0x1000] * 9), 4, 256, 512, 7)
    assert L.dmoe_build_topology(fake, None, ctypes.byref(t), s) == 1
    good = dm._Topo(*([0x1000] * 9), 4, 256, 512, 8)
    # fused dispatch: topology of another E, k > E, d not a multiple of 8,
    # P_max too small
    dargs = [fake, fake, 16, 64, 4, 1, 0, 512, fake, fake, fake, fake, fake, fake, fake, fake, ctypes.byref(good),
             fake, 1 << 20, s]
    for i, bad in ((4, 5), (5, 5), (3, 12), (7, 256)):
        a = list(dargs)
        a[i] = bad
        assert L.dmoe_dispatch(*a) == 1
    # GEMMs: K not a multiple of 64, N not a multiple of 128, bad epilogue, missing outputs
    assert L.dmoe_sdd(fake, fake, None, 100, 0, ctypes.byref(good), 0, None, None, fake, None, None, s) == 1
    assert L.dmoe_sdd(fake, fake, None, 128, 0, ctypes.byref(good), 9, None, None, fake, None, None, s) == 1
    assert L.dmoe_sdd(fake, fake, None, 128, 0, ctypes.byref(good), 1, None, None, fake, None, None, s) == 1
    assert L.dmoe_sdd(fake, fake, None, 128, 0, ctypes.byref(good), 2, None, None, fake, fake, fake, s) == 1
    assert L.dmoe_dsd(ctypes.byref(good), fake, fake, 96, fake, s) == 1
    assert L.dmoe_dsd_t(ctypes.byref(good), fake, fake, fake, None, 128, fake, s) == 1
    assert L.dmoe_dstd(ctypes.byref(good), fake, odd, 128, 0, fake, s) == 1
    assert L.dmoe_unpermute_combine(fake, 128, fake, None, 4, 12, 1, fake, s) == 1
    assert L.dmoe_combine_backward(fake, fake, fake, fake, fake, 4, 16, 1, 100, fake, None, s) == 1


def test_valid_call_without_gpu_reports_cuda_error(libpath):
    """A well-formed call on a machine with no GPU fails cleanly (no crash)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    import dropless_moe_block_gb300 as dm
    L = dm.lib()
    fake = ctypes.c_void_p(0x1000)
    assert L.dmoe_route_topk(fake, 4, 4, 1, 0, fake, fake, None) in (2, 3)
