"""C-ABI checks that need no GPU: the library builds and loads, exports every
entry point the header declares, and rejects bad arguments on the host
before touching the device (nothing here launches a kernel)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8q.h")


@pytest.fixture(scope="module")
def lib():
    from fp8_fine_grained_21_b300 import build as b

    b.build()
    import fp8_fine_grained_21_b300 as fq

    return fq.load()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"FP8Q_API\s+[\w\s\*]+?\b(fp8q_\w+)\s*\(", text)


def test_header_declares_expected_calls():
    names = set(declared_functions())
    for n in ("fp8q_quant_act_1x128", "fp8q_quant_act_128x1", "fp8q_quant_w_128x128",
              "fp8q_gemm", "fp8q_gemm_ex", "fp8q_gemm_grouped", "fp8q_get_device_status",
              "fp8q_status_string", "fp8q_version"):
        assert n in names, n


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n
        assert ctypes.cast(getattr(lib, n), ctypes.c_void_p).value


def test_binding_names_match_header():
    import fp8_fine_grained_21_b300 as fq

    for n in declared_functions():
        assert callable(getattr(fq, n)), n


def test_status_strings_and_version(lib):
    assert lib.fp8q_status_string(0) == b"ok"
    assert lib.fp8q_status_string(5) == b"device pipeline wait timed out"
    assert lib.fp8q_status_string(99) == b"unknown status"
    assert lib.fp8q_version() == 100


P = ctypes.c_void_p
A16 = P(0x10000)          # fake, 16-byte aligned device addresses: never dereferenced,
A16b = P(0x20000)         # the calls below all fail argument checks first
A16c = P(0x30000)
MIS = P(0x10004)


def test_quant_argument_checks(lib):
    f = lib.fp8q_quant_act_1x128
    assert f(None, 1, 128, 128, A16b, A16c, None) == 1        # null input
    assert f(A16, 7, 128, 128, A16b, A16c, None) == 1         # bad dtype
    assert f(A16, 1, 0, 128, A16b, A16c, None) == 1           # empty
    assert f(A16, 1, 128, 200, A16b, A16c, None) == 2         # ragged K
    assert f(MIS, 1, 128, 128, A16b, A16c, None) == 3         # misaligned input
    g = lib.fp8q_quant_act_128x1
    assert g(A16, 1, 100, 64, A16b, A16c, None) == 2          # T not multiple of 128
    assert g(A16, 1, 128, 96, A16b, A16c, None) == 2          # C not multiple of 64
    h = lib.fp8q_quant_w_128x128
    assert h(A16, 1, 130, 128, A16b, A16c, None) == 2
    assert h(A16, 0, 128, 128, MIS, A16c, None) == 3


def test_rmsnorm_quant_argument_checks(lib):
    f = lib.fp8q_rmsnorm_quant_1x128
    f.argtypes = [P, P, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_float, P, P, P]
    assert f(A16, None, 1, 64, 256, 1e-6, A16b, A16c, None) == 1       # null weight
    assert f(A16, A16, 1, 64, 256, 0.0, A16b, A16c, None) == 1         # eps must be > 0
    assert f(A16, A16, 1, 64, 256, float("nan"), A16b, A16c, None) == 1
    assert f(A16, A16, 1, 64, 200, 1e-6, A16b, A16c, None) == 2        # K not a multiple of 128
    assert f(A16, A16, 1, 64, 16384 + 128, 1e-6, A16b, A16c, None) == 2   # K above 16384
    assert f(MIS, A16, 1, 64, 256, 1e-6, A16b, A16c, None) == 3        # misaligned input


def test_swiglu_quant_argument_checks(lib):
    f = lib.fp8q_swiglu_quant_1x128
    assert f(None, A16, 1, 64, 256, 512, A16b, A16c, None) == 1     # null gate
    assert f(A16, A16, 5, 64, 256, 512, A16b, A16c, None) == 1      # bad dtype
    assert f(A16, A16, 1, 0, 256, 512, A16b, A16c, None) == 1       # empty
    assert f(A16, A16, 1, 64, 256, 128, A16b, A16c, None) == 1      # ld < I
    assert f(A16, A16, 1, 64, 200, 512, A16b, A16c, None) == 2      # I not a multiple of 128
    assert f(A16, MIS, 1, 64, 256, 512, A16b, A16c, None) == 3      # misaligned up
    assert f(A16, A16, 1, 64, 256, 260, A16b, A16c, None) == 3      # row stride not 16-byte


def test_gemm_argument_checks(lib):
    g = lib.fp8q_gemm_ex
    ok = (A16, A16b, A16c, P(0x40000), P(0x50000))
    assert g(None, *ok[1:], 128, 128, 128, 0, 0, None) == 1
    assert g(*ok, 128, 128, 128, 3, 0, None) == 1               # bad out dtype
    assert g(*ok, 128, 128, 128, 0, 9, None) == 1               # bad scale mode
    assert g(*ok, 100, 128, 128, 0, 0, None) == 2               # ragged M
    assert g(*ok, 128, 136, 128, 0, 0, None) == 2               # ragged N
    assert g(*ok, 128, 128, 64, 0, 0, None) == 2                # ragged K
    assert g(*ok, -128, 128, 128, 0, 0, None) == 1
    assert g(MIS, *ok[1:], 128, 128, 128, 0, 0, None) == 3
    assert g(*ok, 1 << 30, 1 << 24, 128, 0, 0, None) == 2       # 2^37 output tiles
    gg = lib.fp8q_gemm_grouped
    assert gg(*ok, None, 4, 512, 128, 128, 1, None) == 1       # no offsets
    assert gg(*ok, A16, 0, 512, 128, 128, 1, None) == 2        # no groups
    assert gg(*ok, A16, 513, 512, 128, 128, 1, None) == 2      # too many groups
    assert gg(*ok, P(0x10002), 4, 512, 128, 128, 1, None) == 3  # misaligned offsets


def test_workspace_and_noalloc_argument_checks(lib):
    ok = (A16, A16b, A16c, P(0x40000), P(0x50000))
    w = lib.fp8q_gemm_ws
    assert w(None, *ok[1:], 128, 128, 128, 0, 0, A16, 1 << 30, None) == 1
    assert w(*ok, 128, 128, 64, 0, 0, A16, 1 << 30, None) == 2          # ragged K
    na = lib.fp8q_gemm_noalloc
    assert na(None, *ok[1:], 128, 128, 128, 0, 0, None) == 1
    assert na(*ok, 128, 128, 128, 5, 0, None) == 1                       # bad out dtype
    assert na(*ok, 128, 136, 128, 0, 0, None) == 2                       # ragged N
    assert na(MIS, *ok[1:], 128, 128, 128, 0, 0, None) == 3
    gw = lib.fp8q_gemm_grouped_ws
    assert gw(*ok, None, 4, 512, 128, 128, 1, A16, 1 << 30, None) == 1


def test_noalloc_checks_every_limit_before_launching(lib):
    """fp8q_gemm_noalloc clears its counters with an asynchronous memset before
    the GEMM; every shape limit of the workspace GEMM must be checked before
    that.  2^30 x 2^24 passes the per-dimension limits but has 2^40 output
    tiles: the call must answer FP8Q_ERR_UNSUPPORTED_SHAPE before it looks for
    a device (without a GPU, reaching the device set-up answers
    FP8Q_ERR_CUDA instead).  The pointers are fake and never dereferenced."""
    ok = (A16, A16b, A16c, P(0x40000), P(0x50000))
    na = lib.fp8q_gemm_noalloc
    assert na(*ok, 1 << 30, 1 << 24, 128, 0, 0, None) == 2
    assert na(*ok, 1 << 30, 1 << 24, 128, 1, 1, None) == 2


def test_selftest_wait_limit_checks(lib):
    assert lib.fp8q_selftest_wait(0, None) == 1
    assert lib.fp8q_selftest_wait(-5, None) == 1
    assert lib.fp8q_selftest_wait(100000001, None) == 1


def test_python_binding_refuses_cpu_tensors(lib):
    import torch

    import fp8_fine_grained_21_b300 as fq

    x = torch.zeros(128, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        fq.quant_act_1x128(x)


def test_python_binding_checks_buffer_sizes(lib):
    """The binding checks every buffer's size against the shapes it passes to
    the library (which trusts them), before any device pointer is taken."""
    import torch

    import fp8_fine_grained_21_b300 as fq

    u8, f32 = torch.uint8, torch.float32
    M, N, K = 256, 384, 512
    A8, B8 = torch.zeros(M, K, dtype=u8), torch.zeros(N, K, dtype=u8)
    sA, sB = torch.zeros(K // 128, M, dtype=f32), torch.zeros(N // 128, K // 128, dtype=f32)
    C = torch.zeros(M, N, dtype=f32)
    for bad, what in (
        (dict(C=torch.zeros(M, N + 128, dtype=f32)), "C must have shape"),
        (dict(C=torch.zeros(M - 128, N, dtype=f32)), "C must have shape"),
        (dict(B8=torch.zeros(N, K + 128, dtype=u8)), "same K"),
        (dict(sA=torch.zeros(K // 128 - 1, M, dtype=f32)), "sA must hold"),
        (dict(sB=torch.zeros(N // 128, K // 128 - 1, dtype=f32)), "sB must hold"),
    ):
        args = dict(A8=A8, sA=sA, B8=B8, sB=sB, C=C)
        args.update(bad)
        for fn in (fq.fp8q_gemm, fq.fp8q_gemm_ex, fq.fp8q_gemm_ws, fq.fp8q_gemm_noalloc):
            with pytest.raises(ValueError, match=what):
                fn(args["A8"], args["sA"], args["B8"], args["sB"], args["C"])
    # 1x128 B scales are [K/128][N]: the block-scale count is refused
    with pytest.raises(ValueError, match="sB must hold"):
        fq.fp8q_gemm_ex(A8, sA, B8, sB, C, fq.BSCALE_ROW1x128)
    # grouped: B8 [G][N][K], sB [G][N/128][K/128], m_offsets G + 1 entries
    G = 3
    Bg = torch.zeros(G, N, K, dtype=u8)
    sBg = torch.zeros(G, N // 128, K // 128, dtype=f32)
    offs = torch.zeros(G + 1, dtype=torch.int32)
    with pytest.raises(ValueError, match="sB must hold"):
        fq.fp8q_gemm_grouped(A8, sA, Bg, sB, C, offs)
    with pytest.raises(ValueError, match="m_offsets must hold"):
        fq.fp8q_gemm_grouped_ws(A8, sA, Bg, sBg, C, offs[:G])
    # quantizer outputs
    x = torch.zeros(M, K, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="q must have shape"):
        fq.fp8q_quant_act_1x128(x, torch.zeros(M, K - 16, dtype=u8), sA)
    with pytest.raises(ValueError, match="s must hold"):
        fq.fp8q_quant_act_1x128(x, A8, torch.zeros(K // 128, M - 1, dtype=f32))
    with pytest.raises(ValueError, match="qT must have shape"):
        fq.fp8q_quant_act_128x1(x, A8, torch.zeros(M // 128, K, dtype=f32))
    with pytest.raises(ValueError, match="s must hold"):
        fq.fp8q_quant_w_128x128(x, A8, torch.zeros(M // 128, K // 128 + 1, dtype=f32))
    with pytest.raises(ValueError, match="q must have shape"):
        fq.fp8q_rmsnorm_quant_1x128(x, torch.zeros(K, dtype=torch.bfloat16),
                                    torch.zeros(M + 128, K, dtype=u8), sA)


def test_fused_quant_gemm_argument_checks(lib):
    f = lib.fp8q_gemm_quant_a
    f.argtypes = [P, P, P, P, P, P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                  P, ctypes.c_size_t, P]
    bufs = (A16, A16b, A16c, P(0x40000))
    assert f(None, *bufs[1:], None, None, 256, 256, 256, 0, None, 0, None) == 1      # no A
    assert f(*bufs, A16, None, 256, 256, 256, 0, None, 0, None) == 1               # A8 without sA
    assert f(*bufs, None, None, 256, 384, 256, 0, None, 0, None) == 2              # N % 256
    assert f(*bufs, None, None, 200, 256, 256, 0, None, 0, None) == 2              # ragged M
    assert f(MIS, *bufs[1:], None, None, 256, 256, 256, 0, None, 0, None) == 3      # misaligned A
    assert f(*bufs, P(0x50008), P(0x60000), 256, 256, 256, 0, None, 0, None) == 3  # misaligned A8
    assert f(*bufs, None, None, 1 << 30, 1 << 24, 128, 0, None, 0, None) == 2       # 2^37 tiles


def test_ep_argument_checks(lib):
    I64, I = ctypes.c_int64, ctypes.c_int
    assert lib.fp8q_ep_row_bytes(7168) == 7168 + 224
    assert lib.fp8q_ep_row_bytes(1024) == 1024 + 32
    assert lib.fp8q_ep_row_bytes(128) == 128 + 16          # 4 bytes of scale, padded to 16
    assert lib.fp8q_ep_row_bytes(100) == -1
    r = lib.fp8q_ep_route
    assert r(A16, 10, 2, 0, A16b, A16c, None) == 1           # no experts
    assert r(A16, 10, 2, 257, A16b, A16c, None) == 2         # more than 256 experts
    assert r(A16, 10, 0, 8, A16b, A16c, None) == 1           # k = 0
    assert r(P(0x10002), 10, 2, 8, A16b, A16c, None) == 3    # misaligned ids
    p = lib.fp8q_ep_pack
    assert p(A16, A16b, A16c, 10, 2, 200, P(0x40000), None) == 2       # H % 128
    assert p(MIS, A16b, A16c, 10, 2, 256, P(0x40000), None) == 3
    assert p(None, None, None, 0, 2, 256, None, None) == 0             # no tokens: nothing to do
    u = lib.fp8q_ep_unpack
    args = (A16, 10, 256, A16b, A16c, 2, P(0x40000), P(0x50000), 2, P(0x60000), P(0x70000))
    assert u(*args, 200, None) == 2                                     # Mp % 128
    assert u(*args[:2], 200, *args[3:], 256, None) == 2                 # H % 128
    c = lib.fp8q_ep_combine
    assert c(A16, A16b, A16c, 4, 2, 12, P(0x40000), None) == 2         # N % 8
    assert c(None, None, None, 0, 2, 16, None, None) == 0               # no tokens
    g = lib.fp8q_ep_gather
    assert g(A16, 256, 4, 12, A16b, A16c, 2, P(0x40000), None) == 2    # N % 8
