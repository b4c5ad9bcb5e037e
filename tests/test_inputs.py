"""The seeded input generator: reproducible, right shapes and dtypes, and
draws in a fixed order so that a subset equals the full draw's entries."""

import torch

from tensor_transformer_mlp_forward_gb300 import inputs


def test_reproducible_and_typed():
    a = inputs.make_inputs(inputs.TINY)
    b = inputs.make_inputs(inputs.TINY)
    for k in inputs.DRAW_ORDER:
        assert a[k].dtype == torch.bfloat16
        assert tuple(a[k].shape) == inputs.TINY.shape(k)
        assert a[k].is_contiguous()
        assert torch.equal(a[k], b[k])


def test_subset_matches_full_draw():
    full = inputs.make_inputs(inputs.TINY)
    sub = inputs.make_inputs(inputs.TINY, keys=("A", "B"))
    assert set(sub) == {"A", "B"}
    assert torch.equal(sub["A"], full["A"]) and torch.equal(sub["B"], full["B"])


def test_distributions():
    w = inputs.custom(T=512, h=256, F=1024, t=2, seed=5)
    x = inputs.make_inputs(w)
    assert abs(x["X"].float().std().item() - 1.0) < 0.05
    assert abs(x["A"].float().std().item() - 0.02) < 0.002
    z = inputs.make_inputs(inputs.GPT2_MEDIUM.with_shape(T=64), keys=("b1", "b2"))
    assert float(z["b1"].abs().max()) == 0.0 and float(z["b2"].abs().max()) == 0.0


def test_chunked_draw_is_deterministic(monkeypatch):
    monkeypatch.setattr(inputs, "_CHUNK_ELEMS", 1000)
    w = inputs.custom(T=64, h=64, F=128, t=2, seed=6)
    a = inputs.make_inputs(w)
    b = inputs.make_inputs(w)
    assert torch.equal(a["A"], b["A"])


def test_workload_table():
    m = inputs.MTNLG_530B
    assert (m.T, m.h, m.F, m.t, m.f) == (2048, 20480, 81920, 8, 10240)
    assert m.flops_fwd_bwd() == 12 * 2048 * 20480 * 81920
    assert inputs.MEGATRON_8_3B.f == 1536
    idx = inputs.sample_indices(100, 8, 1)
    assert len(set(idx.tolist())) == 8 and 99 in idx.tolist()
