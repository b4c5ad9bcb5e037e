"""Host logic of bench.py that needs no GPU: the GEMM source hash that keys
the recorded DRAM-traffic lines ignores comments and blank lines, and
nothing else."""

import bench


def test_code_only_drops_comments_and_blank_lines():
    src = ('int a = 1;  // a comment\n'
           '/* a block\n   comment */ char s[] = "x // not a comment /* nor this */";\n'
           "char q = '\"'; char e = '\\\\';\n"
           '\n'
           '   \n'
           'int b = 2;   \n')
    assert bench.code_only(src) == (
        'int a = 1;\n'
        ' char s[] = "x // not a comment /* nor this */";\n'
        "char q = '\"'; char e = '\\\\';\n"
        'int b = 2;')


def test_comment_edits_keep_the_hash_and_code_edits_change_it():
    a = 'int f(int x) {\n    return x + 1;  // the successor\n}\n'
    b = '// f: the successor\nint f(int x) {\n\n    return x + 1;\n}\n'
    c = 'int f(int x) {\n    return x + 2;  // the successor\n}\n'
    assert bench.code_only(a) == bench.code_only(b)
    assert bench.code_only(a) != bench.code_only(c)



def test_recorded_traffic_is_keyed_by_kernel_workload_and_source(tmp_path, monkeypatch):
    f = tmp_path / "traffic.md"
    f.write_text("notes\n"
                 "traffic: kernel=dB workload=mt-nlg-530b src_sha=aaaa bytes_per_launch=111\n"
                 "traffic: kernel=dB workload=mt-nlg-530b src_sha=bbbb bytes_per_launch=222\n"
                 "traffic: kernel=dA workload=mt-nlg-530b src_sha=bbbb bytes_per_launch=333\n")
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "bbbb")
    assert bench.recorded_traffic("dB", "mt-nlg-530b") == 222
    assert bench.recorded_traffic("dA", "mt-nlg-530b") == 333
    assert bench.recorded_traffic("dB", "megatron-8.3b") is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "cccc")  # a changed kernel: no figure
    assert bench.recorded_traffic("dB", "mt-nlg-530b") is None


def test_reference_arm_prints_one_contract_line():
    """`bench.py --impl reference` (the fp64 oracle on the host cores, a
    bounded sample of the MT-NLG block) needs no GPU: one JSON line with the
    contract's keys, its cpu_baseline and an e2e equal to its own value."""
    import json
    import os
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "1"],
                       cwd=root, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 1
    assert d["value"] > 0 and d["higher_is_better"] is True and d["dtype"] == "f64"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["unit"] == d["unit"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert "workload" in d["config"]


def test_cpu_baseline_states_its_extrapolation():
    """The oracle's timed sample is a few token rows; the whole step's time
    it implies is reported beside it, labelled as an extrapolation."""
    import bench
    from tensor_transformer_mlp_forward_gb300 import inputs

    w = inputs.WORKLOADS["tiny"]
    cb = bench.cpu_baseline(w, inputs.make_inputs(w), budget_s=0.0)
    assert cb["kind"] == "oracle" and cb["value"] > 0
    want = w.flops_fwd_bwd() / (cb["value"] * 1e12)
    assert abs(cb["extrapolated_full_step_s"] - want) <= 0.05 + 1e-3 * want
