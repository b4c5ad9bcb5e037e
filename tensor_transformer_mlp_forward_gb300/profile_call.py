"""Run ONE entry point of the library a few times at a given shape, holding
only that call's operands on the device -- the command a profiler wraps to
capture a single kernel of the block at its full per-launch size:

    python -m tensor_transformer_mlp_forward_gb300.profile_call dB \\
        --T 2048 --h 20480 --F 81920 --t 8 --repeat 4

Operands are seeded device-side normals (the profile depends on shapes, not
values).  Prints one JSON line with the mean CUDA-event time per call.

With --vs-cublas (column_gelu, dx, dA_kmajor, dB_kmajor) the call and the
plain cuBLAS product of the same shapes (torch.matmul, bf16, no epilogue)
alternate in rounds of 5 calls, and the JSON line gives both medians.
"""

from __future__ import annotations

import argparse
import json
import sys

CALLS = ("column_gelu", "column_gelu_h_only", "row_sum", "row_sum_dropout", "dgelu", "dx", "dA",
         "dB", "dA_kmajor", "dB_kmajor", "transpose", "dropout_grad", "ln_forward", "ln_backward")


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    p.add_argument("call", choices=CALLS)
    p.add_argument("--T", type=int, default=2048)
    p.add_argument("--h", type=int, default=20480)
    p.add_argument("--F", type=int, default=81920)
    p.add_argument("--t", type=int, default=8)
    p.add_argument("--repeat", type=int, default=4)
    p.add_argument("--dropout", type=float, default=0.1)
    p.add_argument("--vs-cublas", action="store_true",
                   help="time the call against torch.matmul of the same shapes, interleaved")
    p.add_argument("--rounds", type=int, default=8)
    return p.parse_args(argv)


def main(argv=None) -> int:
    import torch

    from tensor_transformer_mlp_forward_gb300 import binding as b

    a = parse_args(argv)
    T, h, F, t = a.T, a.h, a.F, a.t
    dev = torch.device("cuda", 0)
    gen = torch.Generator(device=dev).manual_seed(1234)

    def bf(*shape, std=1.0):
        return (torch.randn(*shape, generator=gen, device=dev) * std).to(torch.bfloat16)

    c = a.call
    ref = None  # the plain cuBLAS product of the call's shapes (--vs-cublas)
    if c in ("column_gelu", "column_gelu_h_only"):
        X, A, b1 = bf(T, h), bf(h, F, std=0.02), bf(F, std=0.02)
        Z = None if c == "column_gelu_h_only" else bf(T, F)
        H = bf(T, F)
        fn = lambda: b.tp_mlp_column_gelu(X, A, b1, t, Z=Z, H=H, want_z=Z is not None)  # noqa: E731
        C = torch.empty(T, F, dtype=torch.bfloat16, device=dev)
        ref = lambda: torch.matmul(X, A, out=C)  # noqa: E731
    elif c in ("row_sum", "row_sum_dropout"):
        H, B, b2, R, Y = bf(T, F), bf(F, h, std=0.02), bf(h, std=0.02), bf(T, h), bf(T, h)
        ws = torch.empty(max(16, b.split_workspace_bytes(T, h, F, t)), dtype=torch.uint8, device=dev)
        if c == "row_sum":
            fn = lambda: b.tp_mlp_row_sum(H, B, b2, R, t, Y=Y, workspace=ws)  # noqa: E731
        else:
            fn = lambda: b.tp_mlp_row_sum_dropout(H, B, b2, R, t, a.dropout, 7, 0, Y=Y,  # noqa: E731
                                                  workspace=ws)
    elif c == "dgelu":
        dY, B, Z, dZ = bf(T, h), bf(F, h, std=0.02), bf(T, F), bf(T, F)
        db1 = torch.empty(F, device=dev)
        part = torch.empty(max(1, int(b.lib().tp_mlp_dgelu_partial_floats(T, F))), device=dev)
        fn = lambda: b.tp_mlp_dgelu(dY, B, Z, t, dZ=dZ, db1=db1, partial=part)  # noqa: E731
    elif c == "dx":
        dZ, A, dX = bf(T, F), bf(h, F, std=0.02), bf(T, h)
        ws = torch.empty(max(16, b.split_workspace_bytes(T, h, F, t)), dtype=torch.uint8, device=dev)
        fn = lambda: b.tp_mlp_dx(dZ, A, t, dX=dX, workspace=ws)  # noqa: E731
        C = torch.empty(T, h, dtype=torch.bfloat16, device=dev)
        ref = lambda: torch.matmul(dZ, A.t(), out=C)  # noqa: E731
    elif c == "dA":
        X, dZ, dA = bf(T, h), bf(T, F), bf(h, F)
        fn = lambda: b.tp_mlp_dA(X, dZ, t, dA=dA)  # noqa: E731
    elif c == "dB":
        H, dY, dB = bf(T, F), bf(T, h), bf(F, h)
        fn = lambda: b.tp_mlp_dB(H, dY, t, dB=dB)  # noqa: E731
    elif c == "dA_kmajor":  # from X^T [h, ldT] and dZ^T [F, ldT]
        ld = b.pitch(T)
        Xt, dZt, dA = bf(h, ld), bf(F, ld), bf(h, F)
        fn = lambda: b.tp_mlp_dA_kmajor(Xt, dZt, T, t, dA=dA)  # noqa: E731
        C = torch.empty(h, F, dtype=torch.bfloat16, device=dev)
        ref = lambda: torch.matmul(Xt[:, :T], dZt[:, :T].t(), out=C)  # noqa: E731
    elif c == "dB_kmajor":  # from H^T [F, ldT] and dY^T [h, ldT]
        ld = b.pitch(T)
        Ht, dYt, dB = bf(F, ld), bf(h, ld), bf(F, h)
        fn = lambda: b.tp_mlp_dB_kmajor(Ht, dYt, T, t, dB=dB)  # noqa: E731
        C = torch.empty(F, h, dtype=torch.bfloat16, device=dev)
        ref = lambda: torch.matmul(Ht[:, :T], dYt[:, :T].t(), out=C)  # noqa: E731
    elif c == "transpose":  # dZ [T, F] -> dZ^T [F, ldT]
        dZ = bf(T, F)
        dZt = torch.empty(F, b.pitch(T), dtype=torch.bfloat16, device=dev)
        fn = lambda: b.tp_transpose(dZ, out=dZt)  # noqa: E731
    elif c == "dropout_grad":
        dY, dP = bf(T, h), bf(T, h)
        fn = lambda: b.tp_mlp_dropout_grad(dY, a.dropout, 7, 0, dP=dP)  # noqa: E731
    else:
        x, r, gam, bet = bf(T, h), bf(T, h), bf(h, std=0.1), bf(h, std=0.1)
        X, s = torch.empty_like(x), torch.empty_like(x)
        mean, rstd = torch.empty(T, device=dev), torch.empty(T, device=dev)
        b.tp_ln_residual_forward(x, r, gam, bet, 1e-5, X=X, s=s, mean=mean, rstd=rstd)
        if c == "ln_forward":
            fn = lambda: b.tp_ln_residual_forward(x, r, gam, bet, 1e-5, X=X, s=s,  # noqa: E731
                                                  mean=mean, rstd=rstd)
        else:
            dX, dres, ds = bf(T, h), bf(T, h), torch.empty_like(x)
            dg, dbt = torch.empty(h, device=dev), torch.empty(h, device=dev)
            part = torch.empty(max(1, int(b.lib().tp_ln_residual_backward_workspace_floats(T, h))),
                               device=dev)
            fn = lambda: b.tp_ln_residual_backward(dX, dres, x, r, gam, mean, rstd, ds=ds,  # noqa: E731
                                                   dgamma=dg, dbeta=dbt, partial=part)
    if a.vs_cublas:
        if ref is None:
            raise SystemExit(f"--vs-cublas is not defined for {c}")
        return compare(c, fn, ref, a, 2.0 * T * h * F)
    ms = []
    for _ in range(a.repeat):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        ms.append(e0.elapsed_time(e1))
    status = b.device_status()
    print(json.dumps({"call": c, "T": T, "h": h, "F": F, "t": t, "repeat": a.repeat,
                      "launches_per_call": b.last_launch_count(),
                      "ms_mean_after_first": sum(ms[1:]) / max(1, len(ms) - 1), "ms": ms,
                      "device_status": status}))
    return 0 if status == 0 else 1


def compare(call, fn, ref, a, flops) -> int:
    """The call and cuBLAS alternating in rounds (the order flips each round),
    5 calls a round, the first of each round dropped; medians of the rest."""
    import statistics

    import torch

    from tensor_transformer_mlp_forward_gb300 import binding as b

    for f in (fn, ref, fn, ref):
        f()
    torch.cuda.synchronize()
    res = {"ours": [], "cublas": []}
    for rnd in range(a.rounds):
        order = (("ours", fn), ("cublas", ref)) if rnd % 2 == 0 else (("cublas", ref), ("ours", fn))
        for tag, f in order:
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
            ev[0].record()
            for k in range(5):
                f()
                ev[k + 1].record()
            torch.cuda.synchronize()
            res[tag] += [ev[k].elapsed_time(ev[k + 1]) for k in range(1, 5)]
    mo, mc = statistics.median(res["ours"]), statistics.median(res["cublas"])
    status = b.device_status()
    print(json.dumps({"call": call, "ours_ms": mo, "cublas_ms": mc, "ours_over_cublas": mo / mc,
                      "ours_tflops": flops / mo / 1e9, "cublas_tflops": flops / mc / 1e9,
                      "samples": len(res["ours"]), "device_status": status}))
    return 0 if status == 0 else 1


if __name__ == "__main__":
    sys.exit(main())
