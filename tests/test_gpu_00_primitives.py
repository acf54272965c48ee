"""Single-CTA checks of the TMA + tcgen05 building blocks of the prefill kernel
(libgqa_selftest.so), run before the full-kernel tests so that a failure
points at the primitive rather than at the pipeline."""
import ctypes

import pytest
import torch

from grouped_query_attention_08_b300 import build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def st():
    build.build()
    lib = ctypes.CDLL(build.lib_path("libgqa_selftest.so"))
    lib.gqa_selftest_qk.restype = ctypes.c_int
    lib.gqa_selftest_qk.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int]
    lib.gqa_selftest_pv.restype = ctypes.c_int
    lib.gqa_selftest_pv.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int, ctypes.c_uint, ctypes.c_uint]
    return lib


@pytest.mark.parametrize("use_cp", [0, 1], ids=["a_from_smem", "a_copied_to_tmem"])
def test_tma_swizzle_and_kmajor_mma(st, use_cp):
    g = torch.Generator().manual_seed(use_cp)
    A = torch.randn(128, 64, generator=g).to(torch.bfloat16)
    B = torch.randn(128, 64, generator=g).to(torch.bfloat16)
    S = torch.zeros(128, 128, device="cuda")
    dA, dB = A.cuda(), B.cuda()          # keep the device copies alive across the call
    rc = st.gqa_selftest_qk(dA.data_ptr(), dB.data_ptr(), S.data_ptr(), use_cp)
    assert rc == 0
    ref = A.double() @ B.double().T
    err = (S.cpu().double() - ref).abs().max().item()
    assert err < 1e-3, "QK^T via tcgen05 differs by %g" % err


@pytest.mark.parametrize("N", [64, 128])
def test_tmem_a_operand_and_mn_major_b(st, N):
    g = torch.Generator().manual_seed(N)
    P = torch.rand(128, 128, generator=g)
    V = torch.randn(128, N, generator=g).to(torch.bfloat16)
    O = torch.zeros(128, N, device="cuda")
    dP, dV = P.cuda(), V.cuda()          # keep the device copies alive across the call
    rc = st.gqa_selftest_pv(dP.data_ptr(), dV.data_ptr(), O.data_ptr(), N, 128 * 128, 1024)
    assert rc == 0
    ref = P.to(torch.bfloat16).double() @ V.double()
    err = (O.cpu().double() - ref).abs().max().item()
    if err >= 1e-3:  # diagnostic: try the other reading of the descriptor offsets
        O2 = torch.zeros(128, N, device="cuda")
        st.gqa_selftest_pv(dP.data_ptr(), dV.data_ptr(), O2.data_ptr(), N, 1024, 128 * 128)
        err2 = (O2.cpu().double() - ref).abs().max().item()
        pytest.fail("P.V via tcgen05 differs by %g (swapped LBO/SBO: %g)" % (err, err2))
