"""The benchmark times the public entry points.

bench.py issues the step's calls one by one so that it can time each kernel
with CUDA events between them.  These tests hold that sequence to the two
public calls a user makes, tp_mlp_forward and tp_mlp_backward: the same
outputs bit for bit and the same number of kernel launches, at the MT-NLG
530B shape the headline is measured on and at a short batch whose
row-parallel GEMMs split their reduction.
"""

import pytest
import torch

import bench
from tensor_transformer_mlp_forward_gb300 import binding, inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("w", [inputs.MTNLG_530B, inputs.SWEEP.with_shape(T=512, t=4)],
                         ids=lambda w: f"{w.name}_T{w.T}_t{w.t}")
def test_bench_step_is_the_public_api(w):
    dev = torch.device("cuda", 0)
    step = bench.Step(w, dev)
    step.launches = 0
    step.run()
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    step_launches = step.launches
    got = {k: getattr(step, k).clone() for k in ("Y", "Z", "H", "dX", "dA", "dB", "db1", "db2")}
    del step
    torch.cuda.empty_cache()

    g = {k: v.to(dev) for k, v in inputs.make_inputs(w).items()}
    Y, Z, H = binding.tp_mlp_forward(g["X"], g["A"], g["b1"], g["B"], g["b2"], g["residual"], w.t)
    n_fwd = binding.last_launch_count()
    dX, dA, dB, db1, db2 = binding.tp_mlp_backward(g["dY"], g["X"], g["A"], g["B"], Z, H, w.t)
    n_bwd = binding.last_launch_count()
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    ref = dict(Y=Y, Z=Z, H=H, dX=dX, dA=dA, dB=dB, db1=db1, db2=db2)
    for k, v in ref.items():
        assert torch.equal(got[k], v), k
    assert step_launches == n_fwd + n_bwd
