"""The C-ABI library on a host without a GPU: it builds, loads, exports every
function include/tpmlp.h declares, and rejects bad arguments with the
documented status codes before touching CUDA."""

import ctypes

import pytest

from tensor_transformer_mlp_forward_gb300 import binding, build


@pytest.fixture(scope="module")
def L():
    build.build()
    return binding.lib()


def test_every_declared_symbol_is_exported(L):
    names = binding.declared_functions()
    assert len(names) >= 15
    for name in names:
        assert hasattr(L, name), name
    assert set(names) == set(binding._SIGNATURES)


def test_status_strings(L):
    for code in range(0, 8):
        assert binding.status_string(code)
    assert binding.status_string(99) == "unknown status"


# fake device addresses: never dereferenced, because every check below fails
# before the library calls into CUDA
P = ctypes.c_void_p(0x10000)
Q = ctypes.c_void_p(0x10008)  # 8-byte aligned only
N = None


def fwd(L, *, X=P, T=128, h=256, F=1024, t=2, Y=P):
    return L.tp_mlp_forward(X, P, P, P, P, P, T, h, F, t, Y, P, P, N, 0, N)


@pytest.mark.parametrize("kw", [
    dict(t=0), dict(t=3), dict(h=12), dict(F=1000, t=8), dict(T=-1), dict(h=0), dict(F=4),
    dict(t=65, F=65 * 8),
])
def test_shape_errors(L, kw):
    assert fwd(L, **kw) == binding.TPMLP_ERR_SHAPE


def test_null_and_alignment_errors(L):
    assert fwd(L, X=N) == binding.TPMLP_ERR_NULL
    assert fwd(L, Y=N) == binding.TPMLP_ERR_NULL
    assert fwd(L, X=Q) == binding.TPMLP_ERR_ALIGN
    assert L.tp_mlp_dx(P, Q, 128, 256, 1024, 2, P, N, 0, N) == binding.TPMLP_ERR_ALIGN
    assert L.tp_mlp_dx(P, P, 128, 256, 1024, 2, P, Q, 1 << 20, N) == binding.TPMLP_ERR_ALIGN
    assert L.tp_mlp_row_sum(P, P, P, P, 128, 256, 1024, 2, P, Q, 1 << 20, N) == binding.TPMLP_ERR_ALIGN
    assert L.tp_mlp_dA(P, P, 128, 256, 1024, 2, N, N) == binding.TPMLP_ERR_NULL
    assert L.tp_mlp_bias_grad(P, 128, 12, P, P, N) == binding.TPMLP_ERR_SHAPE


def test_workspace_errors(L):
    T, h, F, t = 300, 200, 1536, 4
    need = L.tp_mlp_backward_workspace_bytes(T, h, F, t)
    # dZ (bf16) + db1 partials (4 rows per 128-token tile) + db2 partials
    assert need >= 2 * T * F + 4 * 4 * 3 * F + 4 * h
    args = [P] * 6 + [T, h, F, t] + [P] * 5
    assert L.tp_mlp_backward(*args, N, need, N) == binding.TPMLP_ERR_WORKSPACE
    assert L.tp_mlp_backward(*args, P, need - 1, N) == binding.TPMLP_ERR_WORKSPACE
    assert L.tp_mlp_backward(*args, Q, need, N) == binding.TPMLP_ERR_ALIGN
    assert L.tp_mlp_backward_workspace_bytes(T, h, 1000, 8) == 0


def test_weight_grad_form_rule(L):
    # extents that are multiples of 64: the row-major (MN-major) operands
    # are read in one box per stage, no transposes
    assert L.tp_weight_grad_kmajor(20480, 10240) == 0   # MT-NLG dA_i / dB_i (F/t = 10240)
    assert L.tp_weight_grad_kmajor(20480, 81920) == 0
    assert L.tp_weight_grad_kmajor(20480, 20480) == 0   # MT-NLG dWo
    assert L.tp_weight_grad_kmajor(4096, 16384) == 0
    assert L.tp_weight_grad_kmajor(3072, 9216) == 0     # GPT-2 8.3B dWqkv
    # a ragged extent: K-major (transposed operands) where M N / (M + N) >= 6144
    assert L.tp_weight_grad_kmajor(12320, 12288) == 1 and L.tp_weight_grad_kmajor(12296, 12288) == 1
    assert L.tp_weight_grad_kmajor(20480, 20488) == 1 and L.tp_weight_grad_kmajor(4104, 16384) == 0
    assert L.tp_weight_grad_kmajor(0, 81920) == 0 and L.tp_weight_grad_kmajor(-5, 81920) == 0


def test_backward_workspace_holds_the_transposes(L):
    # with the K-major weight gradients (a large block of ragged width): dZ,
    # then X^T and dY^T [h, ldT] and dZ^T and H^T [F, ldT], ldT = T rounded
    # up to 8; without them (extents multiples of 64, or small), none
    T, ldT = 300, 304
    h, F, t = 20488, 81920, 8
    assert L.tp_weight_grad_kmajor(h, F // t) == 1
    big = L.tp_mlp_backward_workspace_bytes(T, h, F, t)
    assert big >= 2 * T * F + 2 * ldT * (2 * h + 2 * F)
    # the same block at h = 20480 (multiples of 64) holds no transposed
    # buffers (its split partials differ a little from the ragged block's)
    assert L.tp_weight_grad_kmajor(20480, F // t) == 0
    assert big - L.tp_mlp_backward_workspace_bytes(T, 20480, F, t) >= 0.5 * 2 * ldT * (2 * h + 2 * F)
    h, F, t = 200, 1536, 4
    assert L.tp_weight_grad_kmajor(h, F // t) == 0
    assert L.tp_mlp_backward_workspace_bytes(T, h, F, t) < 2 * T * F + 2 * ldT * (2 * h + 2 * F)


def test_transpose_argument_errors(L):
    S, NU, AL = binding.TPMLP_ERR_SHAPE, binding.TPMLP_ERR_NULL, binding.TPMLP_ERR_ALIGN
    assert L.tp_transpose(P, 130, 70, P, 136, N) == S    # cols % 8
    assert L.tp_transpose(P, 130, 72, P, 128, N) == S    # ld_out < 136
    assert L.tp_transpose(P, 130, 72, P, 140, N) == S    # ld_out % 8
    assert L.tp_transpose(P, -1, 72, P, 136, N) == S
    assert L.tp_transpose(N, 130, 72, P, 136, N) == NU
    assert L.tp_transpose(P, 130, 72, Q, 136, N) == AL
    assert L.tp_transpose(N, 0, 72, N, 0, N) == binding.TPMLP_OK  # nothing to do
    assert L.tp_transpose(N, 130, 0, N, 136, N) == binding.TPMLP_OK


def test_kmajor_weight_grad_argument_errors(L):
    S = binding.TPMLP_ERR_SHAPE
    for fn in (L.tp_mlp_dA_kmajor, L.tp_mlp_dB_kmajor):
        assert fn(P, P, 130, 128, 256, 1024, 2, P, N) == S   # ldT < 136
        assert fn(P, P, 130, 140, 256, 1024, 2, P, N) == S   # ldT % 8
        assert fn(P, P, 130, 136, 256, 1000, 8, P, N) == S   # F / t % 8
        assert fn(N, P, 130, 136, 256, 1024, 2, P, N) == binding.TPMLP_ERR_NULL
        assert fn(P, P, 130, 136, 256, 1024, 2, N, N) == binding.TPMLP_ERR_NULL
        assert fn(P, Q, 130, 136, 256, 1024, 2, P, N) == binding.TPMLP_ERR_ALIGN


def test_split_workspace_sizes(L):
    # few output tiles (T=512, h=4096: 2 x 16 tiles of 256 x 256): the
    # row-parallel GEMMs split their reduction, and the scratch covers it
    n = L.tp_mlp_split_workspace_bytes(512, 4096, 16384, 8)
    assert n > 0 and n % (4 * 512 * 4096) == 0
    assert L.tp_mlp_forward_workspace_bytes(512, 4096, 16384, 8) == n
    # many tiles (MT-NLG 530B, 640 of them): no whole split, but the last
    # round's 32 tiles are split 7 ways into 256 x 256 fp32 partial tiles
    assert L.tp_mlp_split_workspace_bytes(2048, 20480, 81920, 8) == 32 * 7 * 256 * 256 * 4
    # a multiple of 76 tiles, or too short a reduction to repay a split: nothing
    assert L.tp_mlp_split_workspace_bytes(2048, 19456, 81920, 8) == 0
    assert L.tp_mlp_split_workspace_bytes(8192, 1024, 4096, 2) == 0
    assert L.tp_mlp_split_workspace_bytes(0, 4096, 16384, 8) == 0
    # the backward workspace includes the dX split scratch
    assert (L.tp_mlp_backward_workspace_bytes(512, 4096, 16384, 8)
            >= n + 2 * 512 * 16384)


def test_weight_grad_split_workspace(L):
    # 256 x 256 output tiles of an M x N weight gradient against 76 SM pairs:
    # dWo at h = 1024 has 16 tiles -> 4 k ranges; dWqkv (1024 x 3072) 48 ->
    # 3; 64 tiles (h = 1920) or a 2048-token MT-NLG gradient: none
    assert L.tp_weight_grad_workspace_bytes(8192, 1024, 1024) == 4 * 1024 * 1024 * 4
    assert L.tp_weight_grad_workspace_bytes(8192, 1024, 3072) == 3 * 1024 * 3072 * 4
    assert L.tp_weight_grad_workspace_bytes(8192, 1920, 1920) == 0
    assert L.tp_weight_grad_workspace_bytes(2048, 20480, 81920) == 0
    assert L.tp_weight_grad_workspace_bytes(256, 1024, 1024) == 0  # 4 k-blocks: too short
    assert L.tp_weight_grad_workspace_bytes(0, 1024, 1024) == 0
    # the attention backward workspace holds dWo's and dWqkv's partials
    assert (L.tp_attn_backward_workspace_bytes(8, 1024, 1024, 16, 2)
            >= 3 * 1024 * 3072 * 4)
    assert L.tp_mlp_dA_ws(P, P, 128, 256, 1024, 1, P, Q, 1 << 20, N) == binding.TPMLP_ERR_ALIGN
    assert L.tp_mlp_dB_ws(P, P, 128, 256, 1024, 1, P, Q, 1 << 20, N) == binding.TPMLP_ERR_ALIGN
    assert L.tp_mlp_dA_ws(P, P, 128, 256, 1024, 1, N, P, 1 << 20, N) == binding.TPMLP_ERR_NULL
    assert L.tp_mlp_dB_ws(P, P, 128, 12, 1024, 1, P, P, 1 << 20, N) == binding.TPMLP_ERR_SHAPE


def test_scratch_sizes(L):
    assert L.tp_mlp_dgelu_partial_floats(300, 1536) == 4 * 3 * 1536
    assert L.tp_mlp_dgelu_partial_floats(0, 1536) == 0
    assert L.tp_mlp_bias_grad_workspace_floats(2048, 20480) >= 20480
    assert L.tp_mlp_bias_grad_workspace_floats(8, 64) == 64


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="missing"):
        binding.lib(str(tmp_path / "nope.so"))


def test_no_cpu_fallback_in_binding():
    src = open(binding.__file__).read()
    assert "import oracle" not in src and "from oracle" not in src
    for forbidden in ("torch.matmul", "torch.nn.functional", "torch.mm(", ".cpu()"):
        assert forbidden not in src, forbidden


def test_dropout_argument_errors(L):
    rs = lambda p, off, Y=P: L.tp_mlp_row_sum_dropout(P, P, P, P, 128, 256, 1024, 2, p, 7, off,
                                                      Y, N, 0, N)
    assert rs(1.0, 0) == binding.TPMLP_ERR_SHAPE   # p must be < 1
    assert rs(-0.1, 0) == binding.TPMLP_ERR_SHAPE
    assert rs(float("nan"), 0) == binding.TPMLP_ERR_SHAPE
    assert rs(0.1, 6) == binding.TPMLP_ERR_SHAPE   # offset a multiple of 4
    assert rs(0.1, 8, Y=N) == binding.TPMLP_ERR_NULL
    assert L.tp_mlp_dropout_grad(P, 128, 12, 0.1, 7, 0, P, N) == binding.TPMLP_ERR_SHAPE
    assert L.tp_mlp_dropout_grad(Q, 128, 256, 0.1, 7, 0, P, N) == binding.TPMLP_ERR_ALIGN
    fd = [P] * 6 + [128, 256, 1024, 2, 0.1, 7, 0] + [P] * 3 + [N, 0, N]
    assert L.tp_mlp_forward_dropout(*fd[:10], 0.1, 7, 2, *fd[13:]) == binding.TPMLP_ERR_SHAPE
    # an empty batch is valid and launches nothing
    assert L.tp_mlp_dropout_grad(N, 0, 256, 0.1, 7, 0, N, N) == binding.TPMLP_OK


def test_dropout_backward_workspace(L):
    T, h, F, t = 300, 200, 1536, 4
    base = L.tp_mlp_backward_workspace_bytes(T, h, F, t)
    need = L.tp_mlp_backward_dropout_workspace_bytes(T, h, F, t)
    assert need >= base + 2 * T * h       # plus the bf16 dP
    args = [P] * 6 + [T, h, F, t, 0.1, 7, 0] + [P] * 5
    assert L.tp_mlp_backward_dropout(*args, P, need - 1, N) == binding.TPMLP_ERR_WORKSPACE
    assert L.tp_mlp_backward_dropout(*args, N, need, N) == binding.TPMLP_ERR_WORKSPACE


def test_recompute_workspace(L):
    T, h, F, t = 300, 200, 1536, 4
    fwd_need = L.tp_mlp_forward_recompute_workspace_bytes(T, h, F, t)
    assert fwd_need >= 2 * T * F                  # H lives in the workspace
    bwd_need = L.tp_mlp_backward_recompute_workspace_bytes(T, h, F, t)
    assert bwd_need >= 4 * T * F + L.tp_mlp_backward_workspace_bytes(T, h, F, t)
    fargs = [P] * 6 + [T, h, F, t, P]
    assert L.tp_mlp_forward_recompute(*fargs, N, fwd_need, N) == binding.TPMLP_ERR_WORKSPACE
    assert L.tp_mlp_forward_recompute(*fargs, P, 2 * T * F - 1, N) == binding.TPMLP_ERR_WORKSPACE
    assert L.tp_mlp_forward_recompute(*fargs, Q, fwd_need, N) == binding.TPMLP_ERR_ALIGN
    bargs = [P] * 5 + [T, h, F, t] + [P] * 5
    assert L.tp_mlp_backward_recompute(*bargs, P, bwd_need - 1, N) == binding.TPMLP_ERR_WORKSPACE
    bargs_nob1 = [P] * 3 + [N, P] + [T, h, F, t] + [P] * 5
    assert L.tp_mlp_backward_recompute(*bargs_nob1, P, bwd_need, N) == binding.TPMLP_ERR_NULL
    # Z may be NULL in a2 (H only), H may not
    assert L.tp_mlp_column_gelu(P, P, P, T, h, F, t, N, N, N) == binding.TPMLP_ERR_NULL


def test_launch_mode_setters(L):
    """The process-wide GEMM launch modes: each setter returns the previous
    mode, rejects a mode outside its range with -1 (leaving the mode as it
    was), and touches no device."""
    cases = [  # setter, default, valid modes, invalid modes
        (L.tpmlp_set_cta_pair_mode, 1, (0, 1, 2), (-1, 3)),
        (L.tpmlp_set_epilogue_warps, 0, (0, 4, 8), (2, 16)),
        (L.tpmlp_set_dependent_launch, 3, (0, 1, 2, 3), (-1, 4)),
        (L.tpmlp_set_tile_scheduler, 2, (0, 1, 2), (-1, 3)),
        (L.tpmlp_set_wide_tiles, 0, (0, 1), (-1, 2)),
    ]
    for setter, default, valid, invalid in cases:
        prev = setter(default)
        try:
            for bad in invalid:
                assert setter(bad) == -1
            assert setter(default) == default  # unchanged by the rejected calls
            last = default
            for m in valid:
                assert setter(m) == last
                last = m
        finally:
            setter(prev)
