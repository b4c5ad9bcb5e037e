"""Head-parallel causal self-attention block on the GPU against the fp64
oracle, through the C ABI.

Tolerances are the block's (bf16 inputs, fp32 accumulation): max|gpu - ref|
/ max|ref| <= 1e-2 for forward outputs (Y, QKV, O) and <= 2e-2 for every
gradient (dX, dWqkv, dbqkv, dWo, dbo).  Small cases compare every element
with the full oracle; the full-size GPT-2 and MT-NLG shapes compare sampled
heads (their attention output and every parameter gradient of the head) with
the oracle's per-head entry points.
"""

import numpy as np
import pytest
import torch

import oracle
from tensor_transformer_mlp_forward_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

TOL_FWD = 1e-2
TOL_BWD = 2e-2


def rel(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    den = float(np.max(np.abs(ref)))
    err = float(np.max(np.abs(got - ref)))
    return err / den if den > 0 else err


def np64(x: torch.Tensor) -> np.ndarray:
    return x.detach().to("cpu", torch.float64).numpy()


def run_gpu(w: inputs.AttnWorkload, cpu):
    g = {k: v.cuda() for k, v in cpu.items()}
    Y, QKV, O, lse = binding.tp_attn_forward(g["X"], g["Wqkv"], g["bqkv"], g["Wo"], g["bo"],
                                             g["residual"], w.nb, w.nh, w.t)
    dX, dWqkv, dbqkv, dWo, dbo = binding.tp_attn_backward(g["dY"], g["X"], g["Wqkv"], g["Wo"],
                                                          QKV, O, lse, w.nb, w.nh, w.t)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    return dict(Y=Y, QKV=QKV, O=O, lse=lse, dX=dX, dWqkv=dWqkv, dbqkv=dbqkv, dWo=dWo, dbo=dbo)


# Every compiled head dim (64, 96, 128, 160), several query/key tiles, ragged
# sequence tails against the 128-row and 64-row tiles, t from 1 to nh.
SMALL = [
    inputs.ATTN_TINY,                                              # d = 64, one tile
    inputs.attn_custom(nb=1, s=200, h=192, nh=2, t=1, seed=21),    # d = 96, ragged
    inputs.attn_custom(nb=2, s=130, h=256, nh=2, t=2, seed=22),    # d = 128, 2-row tail
    inputs.attn_custom(nb=1, s=384, h=128, nh=2, t=2, seed=23),    # d = 64, 3 x 128 tiles
    inputs.attn_custom(nb=3, s=72, h=384, nh=4, t=4, seed=24),     # d = 96, t = nh
    inputs.attn_custom(nb=1, s=1, h=64, nh=1, t=1, seed=25),       # one token
    inputs.attn_custom(nb=2, s=257, h=512, nh=4, t=2, seed=26),    # d = 128, 3 tiles + 1
    inputs.attn_custom(nb=2, s=200, h=320, nh=2, t=2, seed=30),    # d = 160: 64-key tiles
    inputs.attn_custom(nb=1, s=300, h=480, nh=3, t=3, seed=31),    # d = 160, 3 query pairs
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: f"nb{w.nb}_s{w.s}_h{w.h}_nh{w.nh}_t{w.t}")
def test_attention_block_vs_oracle(w):
    cpu = inputs.make_attn_inputs(w)
    out = run_gpu(w, cpu)
    Y, QKV, O = oracle.attn_forward(cpu["X"], cpu["Wqkv"], cpu["bqkv"], cpu["Wo"], cpu["bo"],
                                    cpu["residual"], w.nb, w.nh, w.t)
    dX, dWqkv, dbqkv, dWo, dbo = oracle.attn_backward(cpu["dY"], cpu["X"], cpu["Wqkv"],
                                                      cpu["bqkv"], cpu["Wo"], w.nb, w.nh, w.t)
    errs = {}
    for name, ref, tol in (("Y", Y, TOL_FWD), ("QKV", QKV, TOL_FWD), ("O", O, TOL_FWD),
                           ("dX", dX, TOL_BWD), ("dWqkv", dWqkv, TOL_BWD),
                           ("dbqkv", dbqkv, TOL_BWD), ("dWo", dWo, TOL_BWD), ("dbo", dbo, TOL_BWD)):
        errs[name] = (rel(np64(out[name]), ref), tol)
    bad = {k: v for k, v in errs.items() if not v[0] <= v[1]}
    assert not bad, f"{w}: {errs}"
    assert torch.isfinite(out["lse"]).all()


def test_attention_lse_is_row_logsumexp():
    """lse (log2 domain, scaled scores) of each (head, token) against the
    oracle's QKV: log2 sum_k 2^(c q.k) over the visible keys."""
    w = inputs.attn_custom(nb=2, s=150, h=192, nh=2, t=1, seed=27)
    cpu = inputs.make_attn_inputs(w)
    out = run_gpu(w, cpu)
    _, QKV, _ = oracle.attn_forward(cpu["X"], cpu["Wqkv"], cpu["bqkv"], cpu["Wo"], cpu["bo"],
                                    cpu["residual"], w.nb, w.nh, w.t)
    d, h, s = w.d, w.h, w.s
    c = np.log2(np.e) / np.sqrt(d)
    ref = np.zeros((w.nh, w.T))
    for n in range(w.nb):
        for j in range(w.nh):
            q = QKV[n * s:(n + 1) * s, j * d:(j + 1) * d]
            k = QKV[n * s:(n + 1) * s, h + j * d:h + (j + 1) * d]
            u = c * (q @ k.T)
            u[np.triu_indices(s, 1)] = -np.inf
            mx = u.max(axis=1, keepdims=True)
            ref[j, n * s:(n + 1) * s] = (mx + np.log2(np.exp2(u - mx).sum(axis=1, keepdims=True)))[:, 0]
    got = np64(out["lse"])
    # lse is built from the bf16-rounded QKV: compare absolutely (log2 units)
    assert np.max(np.abs(got - ref)) < 5e-2


def test_attention_empty_batch():
    w = inputs.attn_custom(nb=0, s=64, h=128, nh=2, t=2, seed=28)
    dev = torch.device("cuda")
    X = torch.empty((0, w.h), dtype=torch.bfloat16, device=dev)
    Wqkv = torch.randn((w.h, 3 * w.h), device=dev).to(torch.bfloat16)
    Wo = torch.randn((w.h, w.h), device=dev).to(torch.bfloat16)
    bqkv = torch.zeros(3 * w.h, dtype=torch.bfloat16, device=dev)
    bo = torch.zeros(w.h, dtype=torch.bfloat16, device=dev)
    Y, QKV, O, lse = binding.tp_attn_forward(X, Wqkv, bqkv, Wo, bo, X, 0, w.nh, w.t)
    dWqkv = torch.full((w.h, 3 * w.h), 7.0, dtype=torch.bfloat16, device=dev)
    dWo = torch.full((w.h, w.h), 7.0, dtype=torch.bfloat16, device=dev)
    _, dWqkv, dbqkv, dWo, dbo = binding.tp_attn_backward(X, X, Wqkv, Wo, QKV, O, lse, 0, w.nh,
                                                         w.t, dWqkv=dWqkv, dWo=dWo)
    torch.cuda.synchronize()
    assert Y.shape == (0, w.h)
    for g in (dWqkv, dbqkv, dWo, dbo):
        assert float(g.abs().max()) == 0.0


def test_attention_shard_count_changes_nothing_but_the_sum_order():
    """t only groups heads into shards: QKV, O and every gradient but the
    g-summed Y are bit-identical across t (the projection's shards fall on
    64-column boundaries here, so even Y is)."""
    base = inputs.attn_custom(nb=2, s=192, h=512, nh=4, t=1, seed=29)
    cpu = inputs.make_attn_inputs(base)
    outs = [run_gpu(inputs.attn_custom(nb=2, s=192, h=512, nh=4, t=t, seed=29), cpu)
            for t in (1, 2, 4)]
    for o in outs[1:]:
        for k in ("Y", "QKV", "O", "lse", "dX", "dWqkv", "dbqkv", "dWo", "dbo"):
            assert torch.equal(o[k], outs[0][k]), k


def test_attention_kernels_on_two_streams():
    """The persistent attention kernels take their work items from counters
    of their own launch: attention on two streams at once gives the same
    bits as one call after the other on one stream."""
    shapes = [(2, 384, 512, 4), (3, 256, 640, 5)]  # nb, s, h, nh
    g = torch.Generator(device="cuda").manual_seed(42)
    data = []
    for nb, s, h, nh in shapes:
        T = nb * s
        QKV = (torch.randn(T, 3 * h, generator=g, device="cuda") * 0.5).to(torch.bfloat16)
        dO = torch.randn(T, h, generator=g, device="cuda").to(torch.bfloat16)
        data.append((QKV, dO, nb, nh))
    ref = []
    for QKV, dO, nb, nh in data:
        O, lse = binding.tp_attn_core_forward(QKV, nb, nh)
        ref.append((O, lse, binding.tp_attn_core_backward(QKV, O, lse, dO, nb, nh)))
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    got = [[], []]
    for _ in range(4):
        for i, (QKV, dO, nb, nh) in enumerate(data):
            with torch.cuda.stream(streams[i]):
                O, lse = binding.tp_attn_core_forward(QKV, nb, nh)
                got[i].append((O, lse, binding.tp_attn_core_backward(QKV, O, lse, dO, nb, nh)))
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    for i in range(2):
        for O, lse, dQKV in got[i]:
            assert torch.equal(O, ref[i][0]) and torch.equal(lse, ref[i][1])
            assert torch.equal(dQKV, ref[i][2])


def test_attention_tile_scheduler_forms_agree_bitwise():
    """The attention block's GEMMs (QKV, output projection with the g sum,
    the weight gradients, dO and dX) give the same bits with static and
    dynamic tile assignment."""
    w = inputs.attn_custom(nb=2, s=257, h=512, nh=4, t=2, seed=31)
    cpu = inputs.make_attn_inputs(w)
    prev = binding.set_tile_scheduler(0)
    try:
        static = run_gpu(w, cpu)
        binding.set_tile_scheduler(1)
        dynamic = run_gpu(w, cpu)
    finally:
        binding.set_tile_scheduler(prev)
    for k in static:
        assert torch.equal(static[k], dynamic[k]), k


def test_attention_graph_replays_beside_eager_calls():
    """A CUDA graph of the core forward and backward, replayed while the same
    calls run eagerly on another stream: each call takes its work items from
    the counters of its own workspace, so every result is the lone call's."""
    nb, s, h, nh = 2, 384, 512, 4
    g = torch.Generator(device="cuda").manual_seed(43)
    QKV = (torch.randn(nb * s, 3 * h, generator=g, device="cuda") * 0.5).to(torch.bfloat16)
    dO = torch.randn(nb * s, h, generator=g, device="cuda").to(torch.bfloat16)
    O_ref, lse_ref = binding.tp_attn_core_forward(QKV, nb, nh)
    dQKV_ref = binding.tp_attn_core_backward(QKV, O_ref, lse_ref, dO, nb, nh)
    O_g, lse_g = torch.empty_like(O_ref), torch.empty_like(lse_ref)
    dQKV_g, delta_g = torch.empty_like(dQKV_ref), torch.empty_like(lse_ref)
    ws_g = torch.empty(int(binding.lib().tp_attn_core_workspace_bytes(nb, s, h, nh)),
                       dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        binding.tp_attn_core_forward(QKV, nb, nh, O=O_g, lse=lse_g, workspace=ws_g)
        binding.tp_attn_core_backward(QKV, O_g, lse_g, dO, nb, nh, dQKV=dQKV_g, delta=delta_g,
                                      workspace=ws_g)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    eager = []
    for _ in range(4):
        graph.replay()
        with torch.cuda.stream(side):
            O, lse = binding.tp_attn_core_forward(QKV, nb, nh)
            eager.append((O, binding.tp_attn_core_backward(QKV, O, lse, dO, nb, nh)))
        torch.cuda.synchronize()
        assert torch.equal(O_g, O_ref) and torch.equal(dQKV_g, dQKV_ref)
    assert binding.device_status() == 0
    for O, dQKV in eager:
        assert torch.equal(O, O_ref) and torch.equal(dQKV, dQKV_ref)


FULL = [inputs.ATTN_GPT2_355M, inputs.ATTN_GPT2_8_3B, inputs.ATTN_MTNLG_530B,
        # h = 12288: dWo and dWqkv from transposed operands, T = 130 ragged
        # (weights drawn as for the MT-NLG block, which has h of this order)
        inputs.attn_custom(nb=1, s=130, h=12288, nh=96, t=8, seed=34,
                           std=inputs.ATTN_MTNLG_530B.std, name="attn-kmajor-ragged")]


def attn_sample_rows(w: inputs.AttnWorkload, total: int = 36) -> np.ndarray:
    """Token rows for the Y / dX comparison: in the first, a middle and the
    last sequence, the first and the last position, one position in each of
    evenly spread 128-token bands (the query and key tiles of the attention
    kernels), and random positions, about `total` rows in all."""
    g = np.random.default_rng(w.seed + 5)
    seqs = sorted({0, w.nb // 2, w.nb - 1})
    per_seq = min(w.s, max(3, total // len(seqs)))
    bands = (w.s + 127) // 128
    rows = set()
    for n in seqs:
        pick = np.unique(np.linspace(0, bands - 1, min(bands, per_seq - 2)).round().astype(int))
        pos = {0, w.s - 1} | {int(g.integers(128 * b, min(w.s, 128 * b + 128))) for b in pick}
        while len(pos) < per_seq:
            pos.add(int(g.integers(0, w.s)))
        rows |= {n * w.s + p for p in pos}
    return np.array(sorted(rows), dtype=np.int64)


@pytest.mark.parametrize("w", FULL, ids=lambda w: w.name)
def test_attention_full_size_sampled_heads(w):
    """Full-size block in the bench's configuration.  The oracle recomputes
    sampled token rows of Y (the g sum over every head's output plus bo and
    the residual) and of dX (the f sum over the Q, K and V shards of every
    head), evaluating the whole block on each sequence that holds a sampled
    row; and two heads (the first and the last) from the bf16 inputs: their O
    columns and their dWqkv columns, dbqkv entries and dWo rows."""
    cpu = inputs.make_attn_inputs(w)
    out = run_gpu(w, cpu)
    rows = attn_sample_rows(w)
    Yr, dXr = oracle.attn_rows(cpu, w.nb, w.nh, w.t, rows)
    ri = torch.as_tensor(rows, device="cuda")
    e = rel(np64(out["Y"][ri]), Yr)
    assert e <= TOL_FWD, ("Y", e)
    e = rel(np64(out["dX"][ri]), dXr)
    assert e <= TOL_BWD, ("dX", e)
    d, h = w.d, w.h
    for j in (0, w.nh - 1):
        Oj = oracle.attn_head(cpu, w.nb, w.nh, j)
        e = rel(np64(out["O"][:, j * d:(j + 1) * d]), Oj)
        assert e <= TOL_FWD, (j, "O", e)
        dW, db, dWo = oracle.attn_head_grads(cpu, w.nb, w.nh, j)
        cols = torch.cat([torch.arange(p * h + j * d, p * h + (j + 1) * d) for p in range(3)]).cuda()
        got_w = np64(out["dWqkv"].index_select(1, cols))  # the head's columns only
        got_b = np64(out["dbqkv"].index_select(0, cols))
        got_o = np64(out["dWo"][j * d:(j + 1) * d])
        for name, got, ref in (("dWqkv", got_w, dW), ("dbqkv", got_b, db), ("dWo", got_o, dWo)):
            e = rel(got, ref)
            assert e <= TOL_BWD, (j, name, e)
