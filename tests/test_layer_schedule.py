"""The two-stream schedule of a captured layer step, checked on the CPU.

``DMoELayer.run`` puts some calls (the forward combine, the router backward
and the weight-gradient products) on a second stream, each after
an event recorded behind one main-stream call, and joins the streams at the
end of the step.  Here the data each call reads and writes is written out
from the layer's definition (the forward SDD -> act -> DSD blocks, the
combine and its backward, the chain rule of the backward products), and
the schedule the layer builds is checked against it: every call on the
second stream must start after the last writer of everything it reads, and
no main-stream call after its fork point may touch what it reads or writes
before the join.
"""

import re

import pytest

import dropless_moe_block_gb300 as dm


def accesses(name: str, depth: int, swiglu: bool):
    """(reads, writes) of one call, as buffer names; block l = 0..depth-1,
    h_l = input rows of block l (h_0 = x_perm, h_depth = y_perm), g_l = the
    gradient w.r.t. h_l (g_depth = dy_perm, g_0 = dx_perm)."""
    m = re.match(r"(.*?)(?:_(\d+))?$", name)
    base, l = m.group(1), (int(m.group(2)) - 1 if m.group(2) else 0)
    if base in ("route_topk", "gate_route_topk"):
        return {"logits"}, {"expert_idx", "gate_w"}
    if base == "permute_pad":
        return {"x", "expert_idx"}, {"h0", "dest_row", "src_of_row", "padded_offsets", "P"}
    if base == "build_topology":
        return {"padded_offsets"}, {"topo"}
    if base == "sdd_fwd":
        w = {f"W1_{l}"} | ({f"W3_{l}"} if swiglu else set())
        return {f"h{l}", "topo"} | w, {f"G_{l}", f"A_{l}"} | ({f"G3_{l}"} if swiglu else set())
    if base == "dsd_fwd":
        return {f"A_{l}", f"W2_{l}", "topo"}, {f"h{l + 1}"}
    if base == "unpermute_combine":
        return {f"h{depth}", "dest_row", "gate_w"}, {"y"}
    if base == "combine_backward":
        return {"dy", f"h{depth}", "src_of_row", "gate_w", "P"}, {f"g{depth}", "d_gate"}
    if base == "route_backward":
        return {"logits", "expert_idx", "gate_w", "d_gate"}, {"d_logits"}
    if base == "sdd_bwd":
        aux = {f"G_{l}"} | ({f"G3_{l}"} if swiglu else set())
        return {f"g{l + 1}", f"W2_{l}", "topo"} | aux, {f"dH_{l}"} | ({f"dH3_{l}"} if swiglu else set())
    if base == "dstd_dw2":
        return {f"A_{l}", f"g{l + 1}", "topo"}, {f"dW2_{l}"}
    if base == "dsd_t_dx":
        r = {f"dH_{l}", f"W1_{l}", "topo"} | ({f"dH3_{l}", f"W3_{l}"} if swiglu else set())
        return r, {f"g{l}"}
    if base == "dstd_dw1":
        return {f"dH_{l}", f"h{l}", "topo"}, {f"dW1_{l}"}
    if base == "dstd_dw3":
        return {f"dH3_{l}", f"h{l}", "topo"}, {f"dW3_{l}"}
    if base == "unpermute_dx":
        return {"g0", "dest_row"}, {"dx"}
    raise KeyError(name)


def schedule(layer, names):
    """Stream of every call and the happens-before relation the layer's
    ``run`` builds: program order within each stream, an edge from the fork
    call (main stream) to each second-stream call, and an edge from each
    second-stream call a main-stream call waits for (``_main_waits``)."""
    deps = {n: layer._side_dep(n) for n in names}
    stream = {}
    for n in names:
        d = deps[n]
        stream[n] = "side" if d is not None and d in stream and stream[d] == "main" else "main"
    order = {n: i for i, n in enumerate(names)}
    before = {n: set() for n in names}  # before[b] = calls that complete before b starts
    last = {"main": None, "side": None}
    for n in names:
        prev = last[stream[n]]
        if prev is not None:
            before[n] |= before[prev] | {prev}
        if stream[n] == "side":
            before[n] |= before[deps[n]] | {deps[n]}
        else:
            for w in layer._main_waits(n):
                if stream.get(w) == "side" and order[w] < order[n]:
                    before[n] |= before[w] | {w}
        last[stream[n]] = n
    return stream, order, before


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
@pytest.mark.parametrize("depth", [1, 2, 3])
def test_second_stream_calls_are_ordered(act, depth):
    swi = act == "swiglu"
    layer = dm.DMoELayer(64, 64, 4, 128, 2, act, device="cpu", depth=depth)
    w = [None] * depth
    calls = layer.forward_calls(None, None, w, w, w if swi else None)
    calls += layer.backward_calls(None, None, w, w, w if swi else None)
    names = [n for n, _ in calls]
    stream, order, before = schedule(layer, names)
    side = [n for n in names if stream[n] == "side"]
    # the forward combine, the weight-gradient products and the router
    # backward leave the main stream
    assert {re.sub(r"_\d+$", "", n) for n in side} == \
        {"unpermute_combine", "route_backward", "dstd_dw2", "dstd_dw1"} | ({"dstd_dw3"} if swi else set())
    for s in side:
        reads, writes = accesses(s, depth, swi)
        # read-after-write: the last writer of every input has completed
        for buf in reads:
            writers = [n for n in names[:order[s]] if buf in accesses(n, depth, swi)[1]]
            if writers:
                assert writers[-1] in before[s], (s, buf, writers[-1])
        # no main-stream call after the fork point conflicts with the side call
        # unless it waits for it (nothing else orders them before the join at
        # the end of the step)
        fork = layer._side_dep(s)
        for m in names[order[fork] + 1:]:
            if stream[m] != "main" or s in before[m]:
                continue
            mr, mw = accesses(m, depth, swi)
            assert not (mw & (reads | writes)) and not (mr & writes), (s, m)
    # side calls run in program order among themselves, so a side call that
    # reads what an earlier side call wrote is ordered too (checked above);
    # and every output of the step is written by some call
    produced = set().union(*(accesses(n, depth, swi)[1] for n in names))
    for out in ("y", "dx", "d_gate", "d_logits"):
        assert out in produced
    for l in range(depth):
        assert {f"dW1_{l}", f"dW2_{l}"} <= produced and (f"dW3_{l}" in produced) == swi


def test_schedule_model_catches_a_bad_fork_point():
    """The check above fails when a weight-gradient product forks before its
    input exists (the model is not vacuous)."""
    layer = dm.DMoELayer(64, 64, 4, 128, 2, "gelu", device="cpu")
    calls = layer.forward_calls(None, None, None, None) + layer.backward_calls(None, None, None, None)
    names = [n for n, _ in calls]
    orig = layer._side_dep
    layer._side_dep = lambda n: "combine_backward" if n == "dstd_dw1" else orig(n)  # dH not yet written
    stream, order, before = schedule(layer, names)
    assert stream["dstd_dw1"] == "side"
    writers = [n for n in names[:order["dstd_dw1"]] if "dH_0" in accesses(n, 1, False)[1]]
    assert writers == ["sdd_bwd"] and "sdd_bwd" not in before["dstd_dw1"]


def test_backward_sdd_waits_for_the_forward_combine():
    """The forward combine runs beside the combine backward, and the
    backward SDD of the last block starts after both."""
    for depth in (1, 2):
        layer = dm.DMoELayer(64, 64, 4, 128, 2, "gelu", device="cpu", depth=depth)
        w = [None] * depth
        names = [n for n, _ in layer.forward_calls(None, None, w, w) + layer.backward_calls(None, None, w, w)]
        stream, order, before = schedule(layer, names)
        sdd = "sdd_bwd" + layer._sfx(depth - 1)
        assert stream["unpermute_combine"] == "side" and stream["combine_backward"] == "main"
        assert "unpermute_combine" not in before["combine_backward"]
        assert {"unpermute_combine", "combine_backward"} <= before[sdd]
