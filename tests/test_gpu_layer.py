"""GPU parity of w4a16_gemv and w4a16_gemm against the FP64 oracle on small
shapes that span several tiles and ragged tails, plus bit-exact special cases,
determinism, guard bands around the output and host-side rejections."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import weight_only_int4_gb300 as w4  # noqa: E402
from gpu_util import (TORCH_DTYPE, DeviceCase, act_to_torch, assert_within_tol, check_guards,  # noqa: E402
                      guarded_out, torch_to_f64)
from oracle import w4a16_oracle as O  # noqa: E402
from w4a16_inputs import make_case  # noqa: E402

pytestmark = pytest.mark.gpu

OPS = {"gemv": w4.gemv, "gemm": w4.gemm}


def run(op, dc, out=None):
    return OPS[op](dc.x, dc.qw, dc.s, dc.qz, dc.g, out=out)


def parity(op, M, N, K, g, act, sym, scales="uniform", seed=0):
    dc = DeviceCase(make_case(M, N, K, g, act, sym, seed=seed, scales=scales))
    buf, y, pad = guarded_out(M, N, TORCH_DTYPE[act])
    run(op, dc, out=y)
    torch.cuda.synchronize()
    check_guards(buf, pad)
    assert_within_tol(y, dc.reference(), act, f"{op} M={M} N={N} K={K} g={g} {act} sym={sym}")
    assert w4.device_status() == w4.OK


GEMV_SHAPES = [(8, 64), (264, 256), (776, 1024), (2048, 384)]


@pytest.mark.parametrize("act", ["f16", "bf16"])
@pytest.mark.parametrize("g", [32, 128])
@pytest.mark.parametrize("sym", [False, True])
@pytest.mark.parametrize("M", [1, 2, 3, 4, 7, 8, 16])
def test_gemv_parity(act, g, sym, M):
    for (N, K) in GEMV_SHAPES:
        if K % g:
            K = g * max(1, K // g)
        parity("gemv", M, N, K, g, act, sym, seed=M + N + K)


# One row with more 256-column blocks than SMs but at most one 288-column block
# per SM: 9 columns a lane, three 96-column tensor copies per row set, every CTA
# one whole block. Ragged last block, N % 32 != 0 (zero-point words read per
# lane; a lane's 3-column group can cross a word), and N = 152 x 288.
WIDE_BLOCK_LAYERS = [(43000, 512, 128, "f16", False), (39936, 256, 32, "bf16", True),
                     (43776, 256, 64, "f16", False), (42024, 384, 32, "bf16", False)]


@pytest.mark.parametrize("N,K,g,act,sym", WIDE_BLOCK_LAYERS)
def test_gemv_wide_blocks(N, K, g, act, sym):
    parity("gemv", 1, N, K, g, act, sym, seed=N + K)


# Layers just above 4 Mi weights: 2..16 rows run the GEMV's tensor-core MMA
# conversion (smaller layers keep FP32 FMAs up to 2 rows). One with N % 32 != 0
# (zero-point words read per lane, ragged last column block), one with N % 32 == 0
# (zero-point words by tensor copy).
MMA_LAYERS = [(2056, 2304), (2304, 2048)]


@pytest.mark.parametrize("act", ["f16", "bf16"])
@pytest.mark.parametrize("g", [32, 128, 256])
@pytest.mark.parametrize("sym", [False, True])
@pytest.mark.parametrize("M", [2, 3, 4, 5, 8, 9, 13, 16])
def test_gemv_mma_parity(act, g, sym, M):
    for (N, K) in MMA_LAYERS:
        assert N * K > 4 << 20
        parity("gemv", M, N, K, g, act, sym, seed=3 * M + g + N)


@pytest.mark.parametrize("g", [64, 256])
@pytest.mark.parametrize("M", [1, 5, 11])
def test_gemv_other_groups(g, M):
    parity("gemv", M, 520, 2 * g * 3, g, "bf16", False, seed=g + M)
    parity("gemv", M, 520, 2 * g * 3, g, "f16", True, seed=g + M + 1)


@pytest.mark.parametrize("act", ["f16", "bf16"])
@pytest.mark.parametrize("M", [1, 2, 3, 4])
def test_gemv_precomputed_chunk_sums(act, M):
    """Shapes with at least 8 chunks per warp take the GEMV variant whose chunk
    sums of x are computed once per CTA (8192 columns, 640 chunks of K: 20480
    column-block x chunk items for M = 1, 40960 for M = 2..4, against 8 x 16
    warps x 152 or 304 CTAs); smaller shapes form them in each chunk."""
    parity("gemv", M, 8192, 20480, 32, act, False, seed=90 + M)


@pytest.mark.parametrize("act", ["f16", "bf16"])
@pytest.mark.parametrize("M", [1, 4])
def test_gemv_signed_scales(act, M):
    parity("gemv", M, 776, 1024, 32, act, False, scales="signed", seed=3)


GEMM_SHAPES = [(256, 256), (520, 384), (8, 128), (1032, 640)]


@pytest.mark.parametrize("act", ["bf16", "f16"])
@pytest.mark.parametrize("g", [32, 128])
@pytest.mark.parametrize("sym", [False, True])
@pytest.mark.parametrize("M", [1, 17, 128, 255, 256, 300])
def test_gemm_parity(act, g, sym, M):
    for (N, K) in GEMM_SHAPES:
        if K % g:
            K = g * max(1, K // g)
        parity("gemm", M, N, K, g, act, sym, seed=M + N + K)


@pytest.mark.parametrize("M", [32, 33, 64, 65, 127, 129])
@pytest.mark.parametrize("act", ["bf16", "f16"])
def test_gemm_row_buckets(M, act):
    """Both sides of every padding step of the operand-swapped kernel (32, 64, 128
    rows of x) and of its hand-over to the CTA-pair kernel above 128 rows."""
    parity("gemm", M, 776, 384, 32, act, False, seed=M)
    parity("gemm", M, 264, 256, 128, act, True, seed=M + 1)


@pytest.mark.parametrize("g", [64, 256])
def test_gemm_other_groups(g):
    parity("gemm", 200, 520, 2 * g * 3, g, "bf16", False, seed=g)


@pytest.mark.parametrize("act", ["bf16", "f16"])
def test_gemm_signed_scales(act):
    parity("gemm", 384, 776, 1024, 32, act, False, scales="signed", seed=5)


@pytest.mark.parametrize("act", ["f16", "bf16"])
@pytest.mark.parametrize("op,M", [("gemv", 1), ("gemv", 4), ("gemv", 16), ("gemm", 64), ("gemm", 384)])
def test_q4_0_arithmetic(act, op, M):
    """q4_0 weights ("qsa_prompt_attn: Q4_0 KV on tensor cores", section What):
    blocks of 32, w = (code - 8) * d with a scale d of either sign -- the
    symmetric layer at g = 32 with signed scales."""
    parity(op, M, 776, 1024, 32, act, True, scales="signed", seed=40 + M)


def test_gemm_k_tail_half_step():
    # K = 96 with g = 32: the last 64-deep step is half outside K
    parity("gemm", 130, 264, 96, 32, "bf16", False, seed=1)
    parity("gemm", 130, 264, 160, 32, "f16", True, seed=2)


@pytest.mark.parametrize("M", [17, 64, 100])
@pytest.mark.parametrize("K", [96, 160, 224, 288])
def test_gemm_few_rows_k_tail(M, K):
    """The few-row kernel steps 128 deep for up to 64 padded rows of x (64 deep
    above): K = 96 .. 288 leaves the last step 1/4 to 3/4 outside K."""
    parity("gemm", M, 520, K, 32, "bf16", M % 2 == 0, seed=K + M)


def test_gemm_many_tiles_multiple_waves():
    # more tiles than SMs: every CTA loops over several tiles and both accumulators
    parity("gemm", 1024, 8192, 256, 128, "bf16", False, seed=9)


@pytest.mark.parametrize("op", ["gemv", "gemm"])
@pytest.mark.parametrize("act", ["f16", "bf16"])
@pytest.mark.parametrize("sym", [False, True])
def test_onehot_bit_exact(op, act, sym):
    """x = e_k selects one dequantised weight row: y = RN((q - z) * s), bit for bit."""
    M, N, K, g = (5 if op == "gemv" else 130), 264, 256, 32
    case = make_case(M, N, K, g, act, sym, seed=17)
    ks = [(37 * m + 5) % K for m in range(M)]
    x = np.zeros((M, K), dtype=np.float32)
    for m, k in enumerate(ks):
        x[m, k] = 1.0
    case.x = x.astype(np.float16) if act == "f16" else (x.view(np.uint32) >> 16).astype(np.uint16)
    dc = DeviceCase(case)
    y = torch_to_f64(run(op, dc))
    s = O.widen(case.s, act)
    for m, k in enumerate(ks):
        z = 8 if sym else case.z[k // g].astype(np.int64)
        want = O.round_to_act((case.q[k].astype(np.int64) - z) * s[k // g], act)
        assert np.array_equal(y[m], want), (op, act, sym, m)


@pytest.mark.parametrize("op,M", [("gemv", 6), ("gemv", 16), ("gemm", 200)])
@pytest.mark.parametrize("act", ["f16", "bf16"])
def test_q_equals_z_is_exactly_zero(op, M, act):
    """Paths that subtract z from each nibble in 16-bit arithmetic give exact zeros."""
    case = make_case(M, 264, 256, 32, act, False, seed=23)
    case.q = np.repeat(case.z, 32, axis=0)
    y = run(op, DeviceCase(case))
    assert torch.count_nonzero(y).item() == 0


@pytest.mark.parametrize("M", [1, 2, 3, 4])
@pytest.mark.parametrize("act", ["f16", "bf16"])
def test_q_equals_z_gemv_chunk_sums(M, act):
    """For M <= 4 the GEMV applies z once per 32-row chunk as (magic + z) * sum(x):
    q == z then gives zero up to FP32 rounding of two sums of size magic * sum|x|.
    Bound: 64 FP32 half-ulps of magic * sum|x| per chunk (32 additions into two sums
    and their difference), times max|s|, summed over the chunks."""
    K = 1024
    case = make_case(M, 264, K, 32, act, False, seed=29)
    ref_scale = np.abs(DeviceCase(case).reference()).max()
    case.q = np.repeat(case.z, 32, axis=0)
    y = torch_to_f64(run("gemv", DeviceCase(case)))
    x = O.widen(case.x, act)
    magic = 1024.0 if act == "f16" else 128.0
    s_max = np.abs(O.widen(case.s, act)).max()
    chunk_abs = np.abs(x).reshape(M, K // 32, 32).sum(axis=2)          # [M, chunks]
    bound = 64 * 2.0 ** -23 * magic * s_max * chunk_abs.sum(axis=1).max()
    assert np.abs(y).max() <= bound, (np.abs(y).max(), bound)
    assert np.abs(y).max() <= 1e-3 * ref_scale


@pytest.mark.parametrize("op,M", [("gemv", 4), ("gemm", 300), ("gemm", 17), ("gemm", 128)])
def test_deterministic(op, M):
    dc = DeviceCase(make_case(M, 2056, 2048, 128, "bf16", False, seed=31))
    a = run(op, dc).clone()
    b = run(op, dc).clone()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_gemv_and_gemm_agree():
    dc = DeviceCase(make_case(16, 776, 1024, 32, "bf16", False, seed=41))
    a = torch_to_f64(w4.gemv(dc.x, dc.qw, dc.s, dc.qz, 32))
    b = torch_to_f64(w4.gemm(dc.x, dc.qw, dc.s, dc.qz, 32))
    ref = dc.reference()
    assert np.abs(a - b).max() <= 2 * 1.6e-2 * np.abs(ref).max()


def test_gemm_stream_k_workspace_reuse():
    """The few-row GEMM splits column blocks between CTAs and settles them
    through workspace tickets: one zeroed workspace serves calls of different
    shapes (every call leaves its tickets at zero), split and whole blocks both
    match the oracle, and a shape whose every block is split (fewer K-step
    units than SMs) too."""
    cases = [DeviceCase(make_case(M, N, K, 32, act, False, seed=M + N))
             for (M, N, K, act) in ((17, 43008, 512, "bf16"), (64, 4104, 2048, "f16"), (128, 1032, 4096, "bf16"),
                                    (5, 264, 256, "f16"))]
    need = max(w4.workspace_bytes(w4.OP_GEMM, dc.case.M, dc.case.N, dc.case.K, 32) for dc in cases)
    ws = w4.new_workspace(need)
    for _ in range(2):
        for dc in cases:
            y = w4.gemm(dc.x, dc.qw, dc.s, dc.qz, 32, workspace=ws)
            torch.cuda.synchronize()
            assert_within_tol(y, dc.reference(), dc.act, f"gemm {dc.case.M}x{dc.case.N}x{dc.case.K}")
    assert w4.device_status() == w4.OK


def test_gemv_workspace_reuse_across_shapes():
    """One workspace serves calls of different shapes: every call leaves its tickets at zero."""
    ws = w4.new_workspace(32 << 20)
    cases = [DeviceCase(make_case(M, N, K, 32, "f16", False, seed=M + N))
             for (M, N, K) in ((1, 4104, 2048), (3, 1032, 4096), (1, 43008, 512), (7, 264, 256))]
    for _ in range(2):
        for dc in cases:
            need = w4.workspace_bytes(w4.OP_GEMV, dc.case.M, dc.case.N, dc.case.K, 32)
            assert 0 < need <= ws.numel()
            y = w4.gemv(dc.x, dc.qw, dc.s, dc.qz, 32, workspace=ws)
            assert_within_tol(y, dc.reference(), "f16", "reuse")


def test_gemv_workspace_shared_by_templates():
    """Calls of different row templates (MMA conversion with 16 rows x 64
    columns and 8 rows x 128 columns, FMA conversion with 1 row x 256 columns
    and 6 rows x 64 columns), alternating on one workspace: partial sums of
    one never land on the ticket words another relies on."""
    cases = [DeviceCase(make_case(M, N, K, 32, "bf16", False, seed=M + N))
             for (M, N, K) in ((16, 10248, 1024), (1, 4104, 2048), (8, 43008, 896), (6, 1032, 2048))]
    need = max(w4.workspace_bytes(w4.OP_GEMV, dc.case.M, dc.case.N, dc.case.K, 32) for dc in cases)
    ws = w4.new_workspace(need)
    for _ in range(3):
        for dc in cases:
            y = w4.gemv(dc.x, dc.qw, dc.s, dc.qz, 32, workspace=ws)
            assert_within_tol(y, dc.reference(), "bf16", f"shared workspace M={dc.case.M} N={dc.case.N}")
    assert w4.device_status() == w4.OK


def test_gemv_workspace_too_small():
    dc = DeviceCase(make_case(1, 2048, 2048, 128, "f16", False, seed=0))
    need = w4.workspace_bytes(w4.OP_GEMV, 1, 2048, 2048, 128)
    small = w4.new_workspace(max(16, need - 256))
    with pytest.raises(w4.W4A16Error) as e:
        w4.gemv(dc.x, dc.qw, dc.s, dc.qz, 128, workspace=small)
    assert e.value.status == w4.ERR_WORKSPACE


def test_binding_rejections():
    dc = DeviceCase(make_case(2, 64, 128, 32, "f16", False, seed=0))
    z_act = torch.zeros(4, 64, dtype=torch.float16, device="cuda")
    with pytest.raises(TypeError):
        w4.gemv(dc.x, dc.qw, dc.s, z_act, 32)                       # zero-points in the activation dtype
    with pytest.raises(TypeError):
        w4.gemv(dc.x, dc.qw, dc.s.to(torch.bfloat16), dc.qz, 32)   # scales dtype differs from x
    with pytest.raises(ValueError):
        w4.gemv(dc.x, dc.qw, dc.s, dc.qz, 64)                       # scales shape vs g
    big = torch.zeros(2 * 128 + 8, dtype=torch.float16, device="cuda")
    x_mis = big[1:1 + 256].view(2, 128)                               # 2-byte offset: not 16-byte aligned
    with pytest.raises(w4.W4A16Error) as e:
        w4.gemv(x_mis, dc.qw, dc.s, dc.qz, 32)
    assert e.value.status == w4.ERR_ALIGN
    x17 = act_to_torch(make_case(17, 64, 128, 32, "f16", False).x, "f16")
    with pytest.raises(w4.W4A16Error) as e:
        w4.gemv(x17, dc.qw, dc.s, dc.qz, 32)
    assert e.value.status == w4.ERR_SHAPE


@pytest.mark.parametrize("M,N,K,g,act", [(5, 16392, 4096, 32, "f16"), (8, 9216, 4096, 128, "bf16"),
                                         (16, 2056, 5120, 64, "f16"), (12, 43008, 640, 32, "bf16"),
                                         (2, 4104, 4096, 64, "bf16"), (7, 776, 8192, 128, "f16"),
                                         (3, 10248, 4352, 64, "bf16"), (8, 41000, 1280, 128, "f16")])
def test_gemv_mma_rows(M, N, K, g, act):
    """3..16 rows (2 rows above 4 Mi weights) go through the GEMV's tensor-core
    MMA conversion: 8 x-rows x 64 columns where those blocks give a
    block-aligned grid, x 128 columns otherwise (the last two cases: more
    narrow blocks than SMs), 16 x 64 from M = 9; ragged column blocks
    included. Parity with the oracle, and two calls bit-identical."""
    dc = DeviceCase(make_case(M, N, K, g, act, False, seed=M * 3 + g))
    need = w4.workspace_bytes(w4.OP_GEMV, M, N, K, g)
    assert need > w4.workspace_bytes(w4.OP_GEMM, M, N, K, g)   # both kernels' partial regions
    ws = w4.new_workspace(need)
    y1 = w4.gemv(dc.x, dc.qw, dc.s, dc.qz, g, workspace=ws)
    y2 = w4.gemv(dc.x, dc.qw, dc.s, dc.qz, g, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
    assert_within_tol(y1, dc.reference(), act, f"gemv {M}x{N}x{K} g{g} (tensor cores)")
    assert w4.device_status() == w4.OK
