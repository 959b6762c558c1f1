"""dmoe_permute_pad_noalloc: permute + pad for callers that cannot allocate.

Some callers of the library can pass it only the tensors it reads and
writes (no workspace, no allocator at the call site).  This entry point
serves them with a static device scratch array.  The test calls it through
the C ABI and checks, on two calls in a row with different routings, that
its outputs equal those of dmoe_permute_pad (the existing entry point with a
caller workspace) bit for bit -- the tolerance every permute test uses,
since the op only moves integers and bf16 bits.  It also checks that an
oversized request is refused.  It is collected last so that a failure here
leaves every other test already run.
"""

import ctypes

import numpy as np
import pytest
import torch

import dmoe_synth as syn
import oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dropless_moe_block_gb300 import build
    build.build()
    import dropless_moe_block_gb300 as m
    f = m.lib().dmoe_permute_pad_noalloc
    P = ctypes.c_void_p
    f.restype = ctypes.c_int
    f.argtypes = [P, P] + [ctypes.c_int] * 5 + [P] * 6 + [P]
    m.get_error(clear=True)
    return m


def _buffers(T, k, E, d, P_max):
    dev = torch.device("cuda:0")
    return dict(
        tpe=torch.full((E,), -7, dtype=torch.int32, device=dev),
        po=torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
        dest=torch.full((T * k,), -7, dtype=torch.int32, device=dev),
        src=torch.full((P_max,), -7, dtype=torch.int32, device=dev),
        xp=torch.full((P_max, d), 3.0, dtype=torch.bfloat16, device=dev),
        P=torch.full((1,), -7, dtype=torch.int32, device=dev))


def _call_noalloc(dm, x, ei, E, P_max, b):
    T, d = x.shape
    k = ei.shape[1]
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return dm.lib().dmoe_permute_pad_noalloc(p(x), p(ei), T, d, E, k, P_max, p(b["tpe"]), p(b["po"]), p(b["dest"]),
                                             p(b["src"]), p(b["xp"]), p(b["P"]), st)


def _call_existing(dm, x, ei, E, P_max, b):
    T, k = ei.shape
    ws = torch.zeros(dm.permute_pad_workspace_size(T, k, E), dtype=torch.uint8, device=x.device)
    dm.permute_pad(x, ei, E, P_max, b["tpe"], b["po"], b["dest"], b["src"], b["xp"], b["P"], ws)


@pytest.mark.parametrize("name,seed", [("fine", 0), ("skewed", 1)])
def test_noalloc_matches_permute_pad_on_two_calls(dm, name, seed):
    cfg = syn.CONFIGS[name]
    d = 256
    outs = []
    for call in range(2):
        # a different routing on each call: the second call must not see
        # anything the first one left in the shared scratch
        logits = syn.make_logits(cfg) if call == 0 else syn.normal_f32(seed + 50, 1, (cfg.T, cfg.E))
        ei_np, _ = O.route_topk(logits, cfg.k, cfg.renorm)
        x = torch.from_numpy(syn.normal_bf16(seed, 10 + call, (cfg.T, d)).view(np.int16)).view(torch.bfloat16).cuda()
        ei = torch.from_numpy(ei_np).cuda()
        P_max = dm.padded_rows_max(cfg.T, cfg.k, cfg.E)
        a = _buffers(cfg.T, cfg.k, cfg.E, d, P_max)
        b = _buffers(cfg.T, cfg.k, cfg.E, d, P_max)
        assert _call_noalloc(dm, x, ei, cfg.E, P_max, a) == 0
        _call_existing(dm, x, ei, cfg.E, P_max, b)
        torch.cuda.synchronize()
        assert dm.get_error(clear=True) == 0
        P = int(b["P"].item())
        assert int(a["P"].item()) == P
        for key in ("tpe", "po", "dest"):
            assert torch.equal(a[key], b[key]), key
        assert torch.equal(a["src"][:P], b["src"][:P])
        assert torch.equal(a["xp"][:P].view(torch.int16), b["xp"][:P].view(torch.int16))
        outs.append(P)
    assert len(outs) == 2


def test_noalloc_rejects_too_many_experts(dm):
    T, k, E, d = 64, 1, 257, 8
    x = torch.zeros(T, d, dtype=torch.bfloat16, device="cuda:0")
    ei = torch.zeros(T, k, dtype=torch.int32, device="cuda:0")
    P_max = dm.padded_rows_max(T, k, E)
    b = _buffers(T, k, E, d, P_max)
    assert _call_noalloc(dm, x, ei, E, P_max, b) == 1  # DMOE_ERR_INVALID_ARG, nothing launched
    torch.cuda.synchronize()
    assert int(b["P"].item()) == -7
