"""CUDA path against the fp64 oracle, element by element, through the C ABI.

Tolerances (fixed by the block's specification: bf16 inputs, fp32
accumulation): max|gpu - ref| / max|ref| <= 1e-2 for the forward outputs
(Y, and the saved Z and H) and <= 2e-2 for every gradient.
"""

import json
import os

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


def run_gpu(inp_cpu, t):
    g = {k: v.cuda() for k, v in inp_cpu.items()}
    Y, Z, H = binding.tp_mlp_forward(g["X"], g["A"], g["b1"], g["B"], g["b2"], g["residual"], t)
    dX, dA, dB, db1, db2 = binding.tp_mlp_backward(g["dY"], g["X"], g["A"], g["B"], Z, H, t)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    return dict(Y=Y, Z=Z, H=H, dX=dX, dA=dA, dB=dB, db1=db1, db2=db2)


def check_full(w: inputs.Workload):
    cpu = inputs.make_inputs(w)
    out = run_gpu(cpu, w.t)
    Y, Z, H = oracle.forward(cpu["X"], cpu["A"], cpu["b1"], cpu["B"], cpu["b2"], cpu["residual"], w.t)
    dX, dA, dB, db1, db2 = oracle.backward(cpu["dY"], cpu["X"], cpu["A"], cpu["b1"], cpu["B"], w.t)
    errs = {}
    for name, ref, tol in (("Y", Y, TOL_FWD), ("Z", Z, TOL_FWD), ("H", H, TOL_FWD),
                           ("dX", dX, TOL_BWD), ("dA", dA, TOL_BWD), ("dB", dB, TOL_BWD),
                           ("db1", db1, TOL_BWD), ("db2", db2, TOL_BWD)):
        errs[name] = (rel(np64(out[name]), ref), tol)
    log_errors({"workload": w.name, "T": w.T, "h": w.h, "F": w.F, "t": w.t, "rows": w.T,
                "cols": w.F, "max_rel_err": {k: v[0] for k, v in errs.items()}})
    bad = {k: v for k, v in errs.items() if not v[0] <= v[1]}
    assert not bad, f"{w}: {errs}"
    return out


# Small problems the oracle finishes in seconds: several tiles in every
# dimension, ragged tails against the 128 x 256 x 64 tiles, every t.
SMALL = [
    inputs.TINY,
    inputs.custom(T=300, h=200, F=1536, t=1, seed=11),
    inputs.custom(T=300, h=200, F=1536, t=2, seed=11),
    inputs.custom(T=300, h=200, F=1536, t=4, seed=11),
    inputs.custom(T=300, h=200, F=1536, t=8, seed=11),
    inputs.custom(T=130, h=136, F=2560, t=5, seed=12),     # odd shard count, f = 512
    inputs.custom(T=257, h=520, F=1600, t=8, seed=13),     # f = 200: ragged shard tail
    inputs.custom(T=77, h=64, F=512, t=64, seed=14),       # f = 8: one sliver per shard
    inputs.custom(T=1, h=8, F=8, t=1, seed=15),            # smallest legal block
    inputs.custom(T=64, h=8, F=16, t=2, seed=16),          # boxes wider than the tensor
    # f = 200 with h a multiple of 64: the row-parallel GEMM's weight operand
    # is read through the one-box (4-D) MN-major view with the shards on k,
    # the weight gradients' X and dY likewise, dZ and H through two boxes
    inputs.custom(T=300, h=256, F=1600, t=8, seed=17),
    inputs.custom(T=200, h=384, F=3072, t=3, seed=18),     # f = 1024: every MN operand one box
]


@pytest.fixture(params=[0, 2], ids=["single_cta", "cta_pairs"])
def pair_mode(request):
    """Runs a test with the single-CTA GEMM kernel, then with CTA pairs."""
    prev = binding.set_cta_pair_mode(request.param)
    yield request.param
    binding.set_cta_pair_mode(prev)


@pytest.mark.parametrize("w", SMALL, ids=lambda w: f"T{w.T}_h{w.h}_F{w.F}_t{w.t}")
def test_small_against_oracle(w, pair_mode):
    check_full(w)


def test_pairs_and_single_cta_agree_bitwise():
    w = inputs.custom(T=600, h=520, F=2048, t=4, seed=20)
    cpu = inputs.make_inputs(w)
    prev = binding.set_cta_pair_mode(0)
    try:
        single = run_gpu(cpu, w.t)
        binding.set_cta_pair_mode(2)
        pairs = run_gpu(cpu, w.t)
    finally:
        binding.set_cta_pair_mode(prev)
    for k in single:
        assert torch.equal(single[k], pairs[k]), k


@pytest.mark.parametrize("w", [
    inputs.custom(T=300, h=200, F=1536, t=4, seed=21),     # ragged rows and columns
    inputs.custom(T=257, h=520, F=1600, t=8, seed=22),     # f = 200: ragged shard tails
    inputs.custom(T=1100, h=1024, F=4096, t=2, seed=23),   # K = 1024: the short-reduction form
    inputs.custom(T=640, h=2176, F=8704, t=1, seed=24),    # K-major weight gradients off, long K
], ids=lambda w: f"T{w.T}_h{w.h}_F{w.F}_t{w.t}")
@pytest.mark.parametrize("pair", [0, 2], ids=["single_cta", "cta_pairs"])
def test_epilogue_warp_forms_agree_bitwise(w, pair):
    """Four and eight epilogue warps (the dZ GEMM's two forms) give every
    output element the same arithmetic: the whole block is bit for bit the
    same in both forms."""
    cpu = inputs.make_inputs(w)
    prev_pair = binding.set_cta_pair_mode(pair)
    prev = binding.set_epilogue_warps(4)
    try:
        four = run_gpu(cpu, w.t)
        binding.set_epilogue_warps(8)
        eight = run_gpu(cpu, w.t)
    finally:
        binding.set_epilogue_warps(prev)
        binding.set_cta_pair_mode(prev_pair)
    for k in four:
        assert torch.equal(four[k], eight[k]), k


def test_dependent_launch_changes_nothing():
    """GEMMs launched as programmatic dependents wait for the kernel before
    them before touching global memory: the block's outputs are the same
    bits with the launch mode on and off, eagerly and replayed from a CUDA
    graph (where the dependencies become programmatic graph edges)."""
    w = inputs.custom(T=1100, h=1024, F=4096, t=2, seed=25)
    cpu = inputs.make_inputs(w)
    prev = binding.set_dependent_launch(0)
    try:
        plain = run_gpu(cpu, w.t)
        binding.set_dependent_launch(3)
        dep = run_gpu(cpu, w.t)
        g = {k: v.cuda() for k, v in cpu.items()}
        outs = {k: torch.empty_like(v) for k, v in dep.items()}
        ws_f = torch.empty(max(16, binding.split_workspace_bytes(w.T, w.h, w.F, w.t)),
                           dtype=torch.uint8, device="cuda")
        ws_b = torch.empty(binding.tp_mlp_backward_workspace_bytes(w.T, w.h, w.F, w.t),
                           dtype=torch.uint8, device="cuda")

        def block():
            binding.tp_mlp_forward(g["X"], g["A"], g["b1"], g["B"], g["b2"], g["residual"], w.t,
                                   Y=outs["Y"], Z=outs["Z"], H=outs["H"], workspace=ws_f)
            binding.tp_mlp_backward(g["dY"], g["X"], g["A"], g["B"], outs["Z"], outs["H"], w.t,
                                    dX=outs["dX"], dA=outs["dA"], dB=outs["dB"], db1=outs["db1"],
                                    db2=outs["db2"], workspace=ws_b)
        block()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            block()
        for v in outs.values():
            v.zero_()
        graph.replay()
        torch.cuda.synchronize()
    finally:
        binding.set_dependent_launch(prev)
    assert binding.device_status() == 0
    for k in plain:
        assert torch.equal(plain[k], dep[k]), k
        assert torch.equal(plain[k], outs[k]), k


@pytest.mark.parametrize("w,pair", [
    (inputs.custom(T=300, h=200, F=1536, t=4, seed=26), 2),       # ragged, CTA pairs
    (inputs.custom(T=300, h=200, F=1536, t=4, seed=26), 0),       # ragged, single CTAs
    (inputs.custom(T=2048, h=12288, F=4096, t=2, seed=27), 1),    # tail split of a3 and a7
    (inputs.custom(T=512, h=4096, F=16384, t=4, seed=28), 1),     # split reduction of a3 and a7
    (inputs.custom(T=1100, h=1024, F=4096, t=2, seed=29), 1),     # dZ with eight epilogue warps
], ids=["pairs", "single_cta", "tail_split", "split_k", "short_k"])
def test_tile_scheduler_forms_agree_bitwise(w, pair):
    """Static and dynamic (cluster launch control) assignment of output
    tiles compute every tile with the same sums: the block's outputs are the
    same bits under both."""
    cpu = inputs.make_inputs(w)
    prev_pair = binding.set_cta_pair_mode(pair)
    prev = binding.set_tile_scheduler(0)
    try:
        static = run_gpu(cpu, w.t)
        binding.set_tile_scheduler(1)
        dynamic = run_gpu(cpu, w.t)
        again = run_gpu(cpu, w.t)
    finally:
        binding.set_tile_scheduler(prev)
        binding.set_cta_pair_mode(prev_pair)
    for k in static:
        assert torch.equal(static[k], dynamic[k]), k
        assert torch.equal(static[k], again[k]), k


@pytest.mark.parametrize("T,h,F,t", [
    (4096, 3072, 4096, 2),    # whole 256 x 512 tiles, shards folded into one k range
    (1000, 1320, 2048, 8),    # ragged rows and columns (1320 = 2.6 wide tiles)
    (2048, 2048, 16384, 4),   # a long reduction: dynamic tile assignment
], ids=["whole", "ragged", "dynamic"])
def test_wide_tiles_agree_bitwise(T, h, F, t):
    """dX on 256 x 512 tiles per CTA pair (two N = 256 MMAs sharing each A
    stage) gives the bits of the 256 x 256 form: every output element is the
    same k-ordered sum, only the columns a pair covers change."""
    w = inputs.custom(T=T, h=h, F=F, t=t, seed=33)
    cpu = inputs.make_inputs(w, keys=("X", "A"))
    A = cpu["A"].cuda()
    dZ = torch.randn(T, F, device="cuda").mul_(0.5).to(torch.bfloat16)
    empty = torch.empty(0, dtype=torch.uint8, device="cuda")  # no split, no tail split
    prev = binding.set_wide_tiles(0)
    try:
        plain = binding.tp_mlp_dx(dZ, A, t, workspace=empty)
        binding.set_wide_tiles(1)
        wide = binding.tp_mlp_dx(dZ, A, t, workspace=empty)
        assert binding.last_launch_count() == 1
        again = binding.tp_mlp_dx(dZ, A, t, workspace=empty)
    finally:
        binding.set_wide_tiles(prev)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    assert torch.equal(plain, wide)
    assert torch.equal(plain, again)


def test_split_reduction_matches_unsplit():
    """The row-parallel GEMMs with and without a split reduction (few output
    tiles: T=512, h=4096 gives 2 x 16 tiles) agree up to the bf16 rounding of
    their outputs; the oracle comparison of the split path is
    test_full_size_sampled[sweep-h4096_T512_t1]."""
    w = inputs.SWEEP.with_shape(T=512, t=4)
    cpu = inputs.make_inputs(w)
    g = {k: v.cuda() for k, v in cpu.items()}
    assert binding.split_workspace_bytes(w.T, w.h, w.F, w.t) > 0
    H = torch.randn(w.T, w.F, device="cuda").mul_(0.5).to(torch.bfloat16)
    y_split = binding.tp_mlp_row_sum(H, g["B"], g["b2"], g["residual"], w.t)
    empty = torch.empty(0, dtype=torch.uint8, device="cuda")
    y_one = binding.tp_mlp_row_sum(H, g["B"], g["b2"], g["residual"], w.t, workspace=empty)
    dx_split = binding.tp_mlp_dx(H, g["A"], w.t)
    dx_one = binding.tp_mlp_dx(H, g["A"], w.t, workspace=empty)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    assert rel(np64(y_split), np64(y_one)) < TOL_FWD  # one bf16 ulp apart at most
    assert rel(np64(dx_split), np64(dx_one)) < TOL_FWD
    assert not torch.equal(dx_split, dx_one)  # the split path really ran


def test_tail_split_matches_one_launch():
    """384 output tiles of 256 x 256 on 76 CTA pairs (5.05 rounds): with a
    workspace the row-parallel GEMMs (a3, also with dropout, and a7) run the
    five whole rounds in one launch and split the last 4 tiles' reduction
    into k ranges (fp32 partial tiles, then a reduce kernel with the fused
    epilogue): three launches.  Without a workspace one launch computes every
    tile.  The two agree bit for bit outside the tail tiles and within one
    bf16 rounding inside them."""
    T, h, F, t = 2048, 12288, 4096, 2
    g = torch.Generator().manual_seed(31)
    bf = lambda *s, std=1.0: (torch.randn(*s, generator=g) * std).to(torch.bfloat16).cuda()  # noqa: E731
    H, B, b2, R = bf(T, F, std=0.5), bf(F, h, std=0.02), bf(h, std=0.02), bf(T, h)
    dZ, A = bf(T, F, std=0.5), bf(h, F, std=0.02)
    assert binding.split_workspace_bytes(T, h, F, t) > 0
    empty = torch.empty(0, dtype=torch.uint8, device="cuda")
    units = torch.cuda.get_device_properties(0).multi_processor_count // 2
    tiles = (T // 256) * (h // 256)
    runs = {
        "row_sum": lambda ws: binding.tp_mlp_row_sum(H, B, b2, R, t, workspace=ws),
        "row_sum_dropout": lambda ws: binding.tp_mlp_row_sum_dropout(H, B, b2, R, t, 0.1, 99, 0,
                                                                     workspace=ws),
        "dx": lambda ws: binding.tp_mlp_dx(dZ, A, t, workspace=ws),
    }
    for name, fn in runs.items():
        tail = fn(None)
        n_tail = binding.last_launch_count()
        one = fn(empty)
        n_one = binding.last_launch_count()
        torch.cuda.synchronize()
        assert binding.device_status() == 0
        assert n_one == 1, name
        if tiles % units == 0 or tiles < units:
            continue  # no partly full round on this GPU
        assert n_tail == 3, name
        assert rel(np64(tail), np64(one)) < TOL_FWD, name
        differ = int((tail != one).sum())
        assert differ <= (tiles % units + 2 * units) * 256 * 256, name


def test_tail_split_never_slower_than_one_launch():
    """The tail split's plan is an estimate (a pair's rate under the power
    cap, DRAM speed, launch cost).  At the MT-NLG row-parallel GEMM, where it
    is taken, the split schedule must not be slower than the one-launch
    schedule: medians of interleaved calls, 5 % margin for noise."""
    import statistics

    T, h, F, t = 2048, 20480, 81920, 8
    g = torch.Generator(device="cuda").manual_seed(33)
    bf = lambda *s, std=1.0: (torch.randn(*s, generator=g, device="cuda") * std).to(torch.bfloat16)  # noqa: E731
    H, B, b2, R = bf(T, F, std=0.5), bf(F, h, std=0.006), bf(h, std=0.01), bf(T, h)
    Y = torch.empty(T, h, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(binding.split_workspace_bytes(T, h, F, t), dtype=torch.uint8, device="cuda")
    empty = torch.empty(0, dtype=torch.uint8, device="cuda")
    runs = {"split": lambda: binding.tp_mlp_row_sum(H, B, b2, R, t, Y=Y, workspace=ws),
            "one": lambda: binding.tp_mlp_row_sum(H, B, b2, R, t, Y=Y, workspace=empty)}
    runs["split"]()
    assert binding.last_launch_count() == 3  # the plan splits this shape
    times = {k: [] for k in runs}
    for rnd in range(6):
        for k in (("split", "one") if rnd % 2 == 0 else ("one", "split")):
            for _ in range(2):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                runs[k]()
                e1.record()
                torch.cuda.synchronize()
                times[k].append(e0.elapsed_time(e1))
    assert binding.device_status() == 0
    split, one = statistics.median(times["split"]), statistics.median(times["one"])
    assert split <= 1.05 * one, (split, one)


def test_empty_batch():
    w = inputs.custom(T=0, h=64, F=256, t=2, seed=17)
    cpu = inputs.make_inputs(w)
    out = run_gpu(cpu, w.t)
    for k in ("dA", "dB", "db1", "db2"):
        assert float(out[k].abs().max()) == 0.0, k
    for k in ("Y", "Z", "H", "dX"):
        assert out[k].numel() == 0


def test_deterministic():
    w = inputs.custom(T=300, h=200, F=1536, t=4, seed=18)
    cpu = inputs.make_inputs(w)
    a = run_gpu(cpu, w.t)
    b = run_gpu(cpu, w.t)
    for k in a:
        assert torch.equal(a[k], b[k]), k


def test_partition_invariant_on_gpu():
    """With every shard width a multiple of the 64-deep k block, the shard
    count changes only the tile boundaries, never a sum's order: all t give
    bit-identical outputs."""
    base = None
    for t in (1, 2, 4, 8):
        w = inputs.custom(T=300, h=200, F=2048, t=t, seed=19)
        out = run_gpu(inputs.make_inputs(w), t)
        if base is None:
            base = out
            continue
        for k in base:
            assert torch.equal(base[k], out[k]), (t, k)


# ---------------------------------------------------------------- full sizes

# Sampled outputs at full size.  The oracle recomputes whole token rows (Y,
# Z, H and dX over every column: every column tile of every shard, the
# row-parallel GEMMs' tail-split tiles among them) and whole FFN columns (dA
# over every row of A, the matching row of dB, db1).  The rows are picked one
# per 128-row tile band (spread evenly when there are more bands than rows),
# plus the first and the last token; the columns are the first and the last
# of every shard, of the first and last 256-column tile of each shard, plus
# random ones.  Sample sizes follow a fixed fp64 budget per case.
ROW_FLOPS_BUDGET = 6e11  # one token row of Y and dX costs 10 h F flops


def sample_rows(T: int, want: int, seed: int) -> np.ndarray:
    g = np.random.default_rng(seed)
    bands = (T + 127) // 128
    pick = np.arange(bands) if bands <= want else np.unique(
        np.linspace(0, bands - 1, want).round().astype(np.int64))
    rows = {0, T - 1}
    for b in pick:
        lo, hi = 128 * b, min(T, 128 * b + 128)
        rows.add(int(g.integers(lo, hi)))
    while len(rows) < min(T, want):
        rows.add(int(g.integers(0, T)))
    return np.array(sorted(rows), dtype=np.int64)


def sample_cols(F: int, t: int, want: int, seed: int) -> np.ndarray:
    g = np.random.default_rng(seed)
    f = F // t
    cols = set()
    for i in range(t):
        a, b = i * f, (i + 1) * f - 1
        cols.update((a, b, min(b, a + 255), max(a, b - 255)))
    while len(cols) < min(F, max(want, len(cols))):
        cols.add(int(g.integers(0, F)))
    return np.array(sorted(cols), dtype=np.int64)


def sample_sizes(w: inputs.Workload):
    nrows = int(min(96, max(32, ROW_FLOPS_BUDGET // (10 * w.h * w.F))))
    return nrows, 64


def log_errors(record: dict):
    """Appends one JSON line of measured errors to the file named by
    TPMLP_PARITY_LOG, if set (the per-configuration table of errors)."""
    path = os.environ.get("TPMLP_PARITY_LOG")
    if path:
        with open(path, "a") as fh:
            fh.write(json.dumps(record) + "\n")


def check_sampled(w: inputs.Workload):
    nrows, ncols = sample_sizes(w)
    cpu = inputs.make_inputs(w)
    out = run_gpu(cpu, w.t)
    rows = sample_rows(w.T, nrows, w.seed + 1)
    cols = sample_cols(w.F, w.t, ncols, w.seed + 2)
    ri = torch.as_tensor(rows, device="cuda")
    ci = torch.as_tensor(cols, device="cuda")
    Yr, Zr, Hr = oracle.forward_rows(cpu, w.t, rows)
    dXr = oracle.backward_rows(cpu, w.t, rows)
    dAc, dBr, db1c = oracle.backward_cols(cpu, w.t, cols)
    db2 = oracle.db2(cpu["dY"])
    errs = {
        "Y": (rel(np64(out["Y"][ri]), Yr), TOL_FWD),
        "Z": (rel(np64(out["Z"][ri]), Zr), TOL_FWD),
        "H": (rel(np64(out["H"][ri]), Hr), TOL_FWD),
        "dX": (rel(np64(out["dX"][ri]), dXr), TOL_BWD),
        "dA": (rel(np64(out["dA"][:, ci]), dAc), TOL_BWD),
        "dB": (rel(np64(out["dB"][ci]), dBr), TOL_BWD),
        "db1": (rel(np64(out["db1"][ci]), db1c), TOL_BWD),
        "db2": (rel(np64(out["db2"]), db2), TOL_BWD),
    }
    log_errors({"workload": w.name, "T": w.T, "h": w.h, "F": w.F, "t": w.t, "rows": len(rows),
                "cols": len(cols), "max_rel_err": {k: v[0] for k, v in errs.items()}})
    bad = {k: v for k, v in errs.items() if not v[0] <= v[1]}
    assert not bad, f"{w.name} t={w.t}: {errs}"


def test_samples_cover_every_band_and_shard_edge():
    rows = sample_rows(16384, 96, 5)
    assert rows[0] == 0 and rows[-1] == 16383 and len(rows) >= 96
    assert len(np.unique(rows // 128)) >= 95  # spread over the 128 bands
    rows = sample_rows(2048, 36, 5)
    assert set(range(16)) <= set((rows // 128).tolist())  # every band of a short batch
    cols = sample_cols(81920, 8, 64, 6)
    f = 81920 // 8
    for i in range(8):
        assert {i * f, (i + 1) * f - 1} <= set(cols.tolist())
    assert len(cols) >= 64


FULL = [
    inputs.custom(T=2048, h=12288, F=4096, t=2, seed=32, name="tail-split"),  # 384 tiles, 76 pairs
    # h >= 8192: dA and dB from transposed operands inside tp_mlp_backward,
    # T = 130 padded to a 136-element row pitch
    inputs.custom(T=130, h=8192, F=32768, t=4, seed=33, name="kmajor-ragged"),
    inputs.GPT2_MEDIUM.with_shape(T=8192, t=1),
    inputs.GPT2_MEDIUM.with_shape(T=8192, t=2),
] + [inputs.MEGATRON_8_3B.with_shape(T=8192, t=t) for t in (1, 2, 4, 8)] + [
    inputs.MTNLG_530B,
] + [inputs.SWEEP.with_shape(T=T, t=t) for T in inputs.SWEEP_TOKENS for t in inputs.SWEEP_SHARDS]


@pytest.mark.parametrize("w", FULL, ids=lambda w: f"{w.name}_T{w.T}_t{w.t}")
def test_full_size_sampled(w):
    check_sampled(w)
