"""Column sums (the bias gradients db2, dbo, dbqkv) against the oracle.

db[j] = sum_r G[r, j] is computed in fp32 from bf16 G: per thread over its
rows in order, then across lanes, warps and row chunks.  Every partial sum
is bounded by sum_r |G[r, j]|, so after at most `depth` additions the
error is at most depth * 2^-24 * sum_r |G[r, j]| -- the bound each column
is held to here.  depth counts the thread's rows (T / 32), the shuffle,
warp and chunk levels (at most 700 with the 640-CTA target).

The shapes cross the kernel's boundaries: fewer rows than one 32-row step,
one 256-row batch and a ragged one, a single row chunk (db written
directly) and many, column counts that leave a 64-column block partly
empty.
"""

import numpy as np
import pytest
import torch

import oracle
from tensor_transformer_mlp_forward_gb300 import binding, inputs

CASES = [
    (1, 8, 1),
    (31, 64, 2),
    (33, 72, 3),
    (255, 136, 4),
    (257, 520, 5),
    (1000, 1000, 6),
    (4099, 2056, 7),
    (8192, 1024, 8),
]


def _g(T, n, seed):
    w = inputs.custom(T=T, h=n, F=8, t=1, seed=seed)
    return inputs.make_inputs(w, keys=("dY",))["dY"]


def test_oracle_column_sum_closed_form():
    """The oracle's fp64 sum of bf16 values is exact to 2^-52 relative:
    its sum of a column of equal values is that value times T."""
    T, n = 4099, 16
    G = torch.full((T, n), 0.375, dtype=torch.bfloat16)
    assert np.array_equal(oracle.db2(G), np.full(n, 0.375 * T))


@pytest.mark.gpu
@pytest.mark.parametrize("T,n,seed", CASES)
def test_column_sums_within_fp32_bound(T, n, seed):
    cpu = _g(T, n, seed)
    ref = oracle.db2(cpu)
    mag = oracle.db2(cpu.abs())
    db = binding.tp_mlp_bias_grad(cpu.cuda())
    again = binding.tp_mlp_bias_grad(cpu.cuda())
    torch.cuda.synchronize()
    assert binding.device_status() == binding.TPMLP_OK
    got = db.cpu().double().numpy()
    depth = T // 32 + 700
    bound = depth * 2.0 ** -24 * mag + 1e-30
    worst = float(np.max(np.abs(got - ref) / bound))
    assert worst <= 1.0, (T, n, worst)
    assert torch.equal(db, again)  # a fixed order of additions


def _workspace_floats(T, n):
    return max(1, int(binding.lib().tp_mlp_bias_grad_workspace_floats(T, n)))


@pytest.mark.gpu
def test_many_calls_with_changing_grids_share_nothing():
    """Seventy calls in a row whose grids change from call to call (row
    chunks and column blocks), every one on the same workspace: each result
    equals a lone reference call bit for bit, so no completion count or
    partial row carries over from one call to the next."""
    shapes = [(8192, 1024), (2048, 20480), (300, 200), (4099, 2056), (33, 72), (1000, 1000),
              (257, 520)]
    G = {s: _g(*s, seed=40 + i).cuda() for i, s in enumerate(shapes)}
    ref = {s: binding.tp_mlp_bias_grad(G[s]) for s in shapes}
    torch.cuda.synchronize()
    ws = torch.full((max(_workspace_floats(*s) for s in shapes),), float("nan"), device="cuda")
    got = []
    for k in range(70):
        s = shapes[(k * 3) % len(shapes)]
        got.append((s, binding.tp_mlp_bias_grad(G[s], partial=ws[:_workspace_floats(*s)])))
    torch.cuda.synchronize()
    assert binding.device_status() == binding.TPMLP_OK
    for s, db in got:
        assert torch.equal(db, ref[s]), s


@pytest.mark.gpu
def test_two_streams_ordered_by_events_and_graph_replays():
    """Column sums issued on two streams that only events order, and a CUDA
    graph of one call replayed while eager calls run on another stream: each
    call counts in its own workspace, so every result is the lone call's."""
    a, b = _g(2048, 20480, seed=50).cuda(), _g(8192, 1024, seed=51).cuda()
    ref_a, ref_b = binding.tp_mlp_bias_grad(a), binding.tp_mlp_bias_grad(b)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    ws1 = torch.empty(_workspace_floats(2048, 20480), device="cuda")
    ws2 = torch.empty(_workspace_floats(8192, 1024), device="cuda")
    outs = []
    for k in range(8):
        e = torch.cuda.Event()
        with torch.cuda.stream(s1):
            outs.append((ref_a, binding.tp_mlp_bias_grad(a, partial=ws1)))
            e.record(s1)
        with torch.cuda.stream(s2):
            s2.wait_event(e)  # ordered after s1's call only through this event
            outs.append((ref_b, binding.tp_mlp_bias_grad(b, partial=ws2)))
    torch.cuda.synchronize()
    # a graph of one call, replayed beside eager calls on another stream
    db_g = torch.empty_like(ref_a)
    ws_g = torch.empty_like(ws1)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        binding.tp_mlp_bias_grad(a, db=db_g, partial=ws_g)
    torch.cuda.synchronize()
    for k in range(6):
        db_g.fill_(float("nan"))
        graph.replay()
        with torch.cuda.stream(s2):
            outs.append((ref_b, binding.tp_mlp_bias_grad(b, partial=ws2)))
        torch.cuda.current_stream().wait_stream(s2)
        outs.append((ref_a, db_g.clone()))
    torch.cuda.synchronize()
    assert binding.device_status() == binding.TPMLP_OK
    for ref, got in outs:
        assert torch.equal(got, ref)
