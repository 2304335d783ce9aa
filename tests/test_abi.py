"""The C-ABI library loads without a GPU and exports every symbol its header declares;
host-side argument checks answer before any CUDA call (CPU only: no compute calls)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "split_switched_decode.h")


@pytest.fixture(scope="module")
def ssd():
    import split_switched_decode_gb300 as m
    m.build()
    return m


def _declared():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"^DEC_API [^(]*?\b([a-z0-9_]+)\(", src, re.M)))


def test_header_declares_the_documented_entry_points():
    names = _declared()
    for n in ["dec_gemv", "dec_splitk_gemm", "dec_linear", "moe_front", "moe_experts",
              "l2_prefetch"]:
        assert n in names


def test_library_exports_every_declared_symbol(ssd):
    lib = ctypes.CDLL(ssd.LIB_PATH)
    for n in _declared():
        assert hasattr(lib, n), n
    assert sorted(ssd.EXPORTS) == _declared()


def test_library_has_no_libcuda_link_dependency(ssd):
    import subprocess
    out = subprocess.run(["ldd", ssd.LIB_PATH], capture_output=True, text=True).stdout
    assert "libcuda.so" not in out and "libcudart.so" not in out


def test_static_strings(ssd):
    lib = ssd.lib()
    assert lib.dec_status_string(0) == b"ok"
    assert lib.dec_status_string(6) == b"device wait timed out"
    assert lib.dec_variant_name(0) == b"tiny"
    assert lib.dec_variant_name(2) == b"splitk_tc"
    assert lib.dec_variant_name(3) == b"front_one_launch"
    assert lib.dec_variant_name(4) == b"splitk_tc_pair"
    assert lib.dec_version() == 100
    assert lib.dec_last_variant() == -1
    assert lib.moe_route_map_ints(64, 384, 8) == 3 * 384 + 2 + 2 * 64 * 8


def test_host_argument_checks_need_no_device(ssd):
    lib = ssd.lib()
    A = ctypes.c_void_p(0x1000)  # never dereferenced: every call below fails its checks
    U = ctypes.c_void_p(0x1001)  # misaligned
    N0 = None
    s = None
    assert lib.dec_gemv(N0, A, N0, A, 1, 8, 8, s) == ssd.DEC_ERR_INVALID_ARG
    assert lib.dec_gemv(A, A, N0, A, 0, 8, 8, s) == ssd.DEC_ERR_INVALID_ARG
    assert lib.dec_gemv(A, A, N0, A, 65, 8, 8, s) == ssd.DEC_ERR_UNSUPPORTED_SHAPE
    assert lib.dec_gemv(A, A, N0, A, 1, 8, 12, s) == ssd.DEC_ERR_MISALIGNED
    assert lib.dec_gemv(U, A, N0, A, 1, 8, 8, s) == ssd.DEC_ERR_MISALIGNED
    assert lib.dec_gemv(A, A, N0, A, 5, 8, 8, s) == ssd.DEC_ERR_UNSUPPORTED_SHAPE
    assert lib.dec_splitk_gemm(A, A, N0, A, 4, 8, 8, -1, 0, A, 0, s) == ssd.DEC_ERR_INVALID_ARG
    assert lib.dec_splitk_gemm(A, A, N0, A, 4, 8, 8, 0, 2, A, 0, s) == ssd.DEC_ERR_INVALID_ARG
    assert lib.dec_linear(A, N0, N0, A, 4, 8, 8, A, 0, s) == ssd.DEC_ERR_INVALID_ARG
    args = [A, A, 4, 64, 384, 512, 8, A, A, A, N0, N0, A, 1 << 30, s]
    bad = list(args)
    bad[6] = 17  # topk > 16
    assert lib.moe_front(*bad) == ssd.DEC_ERR_UNSUPPORTED_SHAPE
    bad = list(args)
    bad[4] = 513  # E > 512
    assert lib.moe_front(*bad) == ssd.DEC_ERR_UNSUPPORTED_SHAPE
    bad = list(args)
    bad[7] = N0  # latent missing with L > 0
    assert lib.moe_front(*bad) == ssd.DEC_ERR_INVALID_ARG
    e_args = [A, A, A, N0, A, A, 384, A, N0, 4, 7168, 2048, 8, A, A, 1 << 30, s, s, 0]
    assert lib.moe_experts(*e_args) == ssd.DEC_ERR_INVALID_ARG  # shared Wgu without Wd
    bad = list(e_args)
    bad[8] = A
    bad[10] = 7000  # H % 128 != 0
    assert lib.moe_experts(*bad) == ssd.DEC_ERR_UNSUPPORTED_SHAPE
    assert lib.l2_prefetch(U, 64, 0, s) == ssd.DEC_ERR_MISALIGNED
    assert lib.l2_prefetch(N0, 64, 0, s) == ssd.DEC_ERR_INVALID_ARG
    assert lib.l2_prefetch(A, 15, 0, s) == ssd.DEC_OK  # rounds down to nothing: no launch
    assert lib.dec_set_force_variant(7) == ssd.DEC_ERR_INVALID_ARG
    assert lib.dec_set_wait_limit_ns(10) == ssd.DEC_ERR_INVALID_ARG
    assert lib.dec_debug_wait_timeout(10, s) == ssd.DEC_ERR_INVALID_ARG
    assert lib.dec_sim_comm_wait(999, s) == ssd.DEC_ERR_INVALID_ARG
    l_args = [N0, A, 384, 512, 8, A, A, A, A, 4, 7168, 2048, A, A, A, N0, A, A, 1 << 30, s, s, 0]
    assert lib.moe_layer(*l_args) == ssd.DEC_ERR_INVALID_ARG  # X missing
    bad = list(l_args)
    bad[0], bad[12] = A, N0  # latent missing with L > 0
    assert lib.moe_layer(*bad) == ssd.DEC_ERR_INVALID_ARG
    assert lib.dec_sim_comm_wait(1000000001, s) == ssd.DEC_ERR_INVALID_ARG
    assert lib.dec_read_stream(N0, 1 << 20, s) == ssd.DEC_ERR_INVALID_ARG
    assert lib.dec_read_stream(U, 1 << 20, s) == ssd.DEC_ERR_MISALIGNED
    # tile-packed weights: whole 128-row tiles and 64-wide k-blocks only
    assert lib.dec_pack_weight(A, 256, 128, A, s) == ssd.DEC_ERR_INVALID_ARG  # W and Wp overlap
    assert lib.dec_pack_weight(A, 200, 128, ctypes.c_void_p(0x100000), s) == \
        ssd.DEC_ERR_UNSUPPORTED_SHAPE
    assert lib.dec_pack_weight(A, 256, 96, ctypes.c_void_p(0x100000), s) == \
        ssd.DEC_ERR_UNSUPPORTED_SHAPE
    assert lib.dec_pack_weight(U, 256, 128, ctypes.c_void_p(0x100000), s) == ssd.DEC_ERR_MISALIGNED
    assert lib.dec_pack_weight(N0, 256, 128, A, s) == ssd.DEC_ERR_INVALID_ARG
    assert lib.dec_gemv_packed(A, A, N0, A, 1, 200, 128, s) == ssd.DEC_ERR_UNSUPPORTED_SHAPE
    assert lib.dec_gemv_packed(A, A, N0, A, 1, 256, 96, s) == ssd.DEC_ERR_UNSUPPORTED_SHAPE
    assert lib.dec_splitk_gemm_packed(A, A, N0, A, 4, 8, 64, 0, 1, A, 0, s) == \
        ssd.DEC_ERR_UNSUPPORTED_SHAPE
    assert lib.dec_linear_packed(A, A, N0, A, 4, 128, 72, A, 0, s) == ssd.DEC_ERR_UNSUPPORTED_SHAPE
    assert lib.dec_linear_packed(A, N0, N0, A, 4, 128, 64, A, 0, s) == ssd.DEC_ERR_INVALID_ARG
    B1, B2, B3 = (ctypes.c_void_p(0x1000000 * i) for i in (2, 3, 4))
    assert lib.dec_pack_expert_weights(A, B1, 2, 256, 128, A, B3, s) == ssd.DEC_ERR_INVALID_ARG
    assert lib.dec_pack_expert_weights(A, B1, 2, 200, 128, B2, B3, s) == \
        ssd.DEC_ERR_UNSUPPORTED_SHAPE
    assert lib.dec_pack_expert_weights(A, B1, 2, 256, 96, B2, B3, s) == \
        ssd.DEC_ERR_UNSUPPORTED_SHAPE
    assert lib.dec_pack_expert_weights(U, B1, 2, 256, 128, B2, B3, s) == ssd.DEC_ERR_MISALIGNED
    assert lib.dec_pack_expert_weights(N0, B1, 2, 256, 128, B2, B3, s) == ssd.DEC_ERR_INVALID_ARG
    # a source bank overlapping the other bank's destination
    assert lib.dec_pack_expert_weights(A, B1, 2, 256, 128, B2, A, s) == ssd.DEC_ERR_INVALID_ARG
    assert lib.dec_pack_expert_weights(A, B1, 2, 256, 128, B1, B3, s) == ssd.DEC_ERR_INVALID_ARG
    assert lib.dec_set_fault_inject(-1) == ssd.DEC_ERR_INVALID_ARG
