"""GPU probes of the tcgen05 / TMA building blocks: operand layouts,
descriptors, the instruction descriptor and the TMEM lane mapping, checked
against a host fp64 matmul (and a host slice for TMA)."""
import ctypes

import pytest
import torch

from linear_attention_recurrence_fwd_gb300 import binding, build

pytestmark = pytest.mark.gpu

SW128, SW64, SW32 = 2, 4, 6


@pytest.fixture(scope="module")
def probe(cuda_device):
    build.build()
    return binding.load_probe()


def _run(probe, M, N, K, a_mn, a_sw, a_bc, b_mn, b_sw, b_bc, b_row0=0, NB=None, neg=0, acc=1,
         seed=0, tf32=0):
    NB = NB or (b_row0 + N)
    g = torch.Generator().manual_seed(seed)
    A = torch.randn(M, K, generator=g).bfloat16()
    B = torch.randn(NB, K, generator=g).bfloat16()
    Ad, Bd = A.cuda(), B.cuda()
    D = torch.full((128, N), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = probe.kda_probe_umma(Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), M, N, K, NB, a_mn, a_sw,
                              a_bc, b_mn, b_sw, b_bc, b_row0, neg, acc, tf32, st.data_ptr(),
                              torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert st.item() == 0, "MMA completion wait timed out"
    exp = (A.double() @ B[b_row0:b_row0 + N].double().T) * acc * (-1.0 if neg else 1.0)
    return D.cpu().double(), exp


def _close(a, b):
    return torch.allclose(a, b, rtol=1e-3, atol=1e-3)


CASES = [
    # M, N, K, a_mn, a_sw, a_bc, b_mn, b_sw, b_bc, b_row0, NB
    (128, 64, 128, 0, SW128, 0, 0, SW128, 0, 0, None),
    (128, 256, 64, 0, SW128, 0, 0, SW128, 0, 0, None),
    (128, 64, 128, 1, SW128, 0, 0, SW128, 0, 0, None),
    (128, 64, 128, 1, SW128, 1, 0, SW128, 0, 0, None),
    (128, 64, 128, 0, SW128, 0, 1, SW128, 0, 0, None),
    (128, 128, 64, 0, SW128, 0, 1, SW128, 1, 0, None),
    (128, 128, 64, 0, SW128, 0, 1, SW128, 0, 0, None),
    (128, 128, 128, 0, SW128, 0, 1, SW128, 0, 0, None),  # two N blocks one LBO apart, K = 128
    (128, 16, 128, 0, SW128, 0, 1, SW128, 0, 16, 64),
    (128, 16, 128, 0, SW128, 0, 1, SW128, 0, 48, 64),
    (128, 32, 64, 0, SW128, 0, 1, SW128, 0, 32, 64),
    (128, 16, 128, 0, SW128, 0, 1, SW32, 0, 0, None),
    (128, 16, 128, 0, SW128, 0, 1, SW32, 0, 16, 32),
    (128, 32, 64, 0, SW64, 0, 0, SW64, 0, 0, None),
    (128, 32, 64, 1, SW64, 0, 1, SW64, 0, 0, None),
    (128, 64, 64, 0, SW128, 0, 0, SW128, 0, 16, 128),
    # the state pass: N = 192 as three MN-major blocks one LBO apart, K = 128
    (128, 192, 128, 0, SW128, 0, 1, SW128, 0, 0, None),
    # the state pass's value term: A MN-major (a raw v tile), B K-major N = 192
    (128, 192, 64, 1, SW128, 0, 0, SW128, 0, 0, None),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_umma_m128_layouts(probe, case):
    M, N, K, a_mn, a_sw, a_bc, b_mn, b_sw, b_bc, b_row0, NB = case
    D, exp = _run(probe, M, N, K, a_mn, a_sw, a_bc, b_mn, b_sw, b_bc, b_row0, NB)
    assert _close(D, exp), f"max err {(D - exp).abs().max().item():.3e}"


def test_umma_negate_and_accumulate(probe):
    D, exp = _run(probe, 128, 64, 64, 0, SW128, 0, 1, SW128, 0, neg=1, acc=3)
    assert _close(D, exp)


def test_umma_m64_lane_mapping(probe):
    """Where the 64 rows of an M=64 accumulator land among the 128 TMEM lanes."""
    D, exp = _run(probe, 64, 32, 64, 0, SW128, 0, 0, SW128, 0)
    found = {}
    for m in range(64):
        lanes = [l for l in range(128) if torch.allclose(D[l], exp[m], rtol=1e-3, atol=1e-3)]
        found[m] = lanes
    expected = {m: [32 * (m // 16) + m % 16] for m in range(64)}
    assert found == expected, f"lane mapping: {found}"


@pytest.mark.parametrize("N,K,b_mn", [(64, 64, 0), (128, 128, 1), (192, 128, 1), (128, 64, 0)])
def test_umma_a_from_tmem(probe, N, K, b_mn):
    """A read from tensor memory: row m in lane m, two consecutive K elements
    per 32-bit column, the lower half the even one."""
    g = torch.Generator().manual_seed(N + K)
    A = torch.randn(128, K, generator=g).bfloat16()
    B = torch.randn(N, K, generator=g).bfloat16()
    Ad, Bd = A.cuda(), B.cuda()  # held: the device copies must outlive the call
    D = torch.full((128, N), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = probe.kda_probe_umma_ta(Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), 128, N, K,
                                 N, 0, SW128, 0, b_mn, SW128, 0, 0, 0, 1, 0, 1, st.data_ptr(),
                                 torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert st.item() == 0
    exp = A.double() @ B.double().T
    assert _close(D.cpu().double(), exp), f"max err {(D.cpu().double() - exp).abs().max().item():.3e}"


def test_umma_m64_mn_major_a(probe):
    """M = 64 with an MN-major A operand (the A_qk image read as A): rows land
    on lanes 32 (m // 16) + m % 16."""
    D, exp = _run(probe, 64, 64, 64, 1, SW128, 0, 1, SW128, 0)
    lanes = [32 * (m // 16) + m % 16 for m in range(64)]
    assert _close(D[lanes], exp), f"max err {(D[lanes] - exp).abs().max().item():.3e}"


@pytest.mark.parametrize("d,t0", [(128, 0), (128, 64), (64, 32)])
def test_tma_tile_matches_layout(probe, d, t0):
    T, H, h = 100, 3, 1
    src = torch.randn(T, H, d).bfloat16().cuda()
    out = torch.full((64, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = probe.kda_probe_tma(src.data_ptr(), out.data_ptr(), T, H, d, h, t0, st.data_ptr(),
                             torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert st.item() == 0
    exp = torch.zeros(64, d, dtype=torch.bfloat16)
    n = min(64, T - t0)
    exp[:n] = src[t0:t0 + n, h].cpu()
    assert torch.equal(out.cpu(), exp)


# Only K-major operands: with MN-major fp32 operands (laid out like the 16-bit
# MN-major atoms, 32 fp32 per 128-byte row) kind::tf32 did not reproduce the
# matmul on GB300, so the kernels keep tf32 out of the MN-major products.
TF32_CASES = [
    # M, N, K, a_mn, a_sw, b_mn, b_sw, b_row0, NB
    (128, 64, 32, 0, SW128, 0, SW128, 0, None),
    (128, 64, 64, 0, SW128, 0, SW128, 0, None),
]


@pytest.mark.parametrize("case", TF32_CASES, ids=lambda c: "-".join(map(str, c)))
def test_umma_tf32_layouts(probe, case):
    """kind::tf32 with fp32 operands (bf16-valued inputs, so products are exact)."""
    M, N, K, a_mn, a_sw, b_mn, b_sw, b_row0, NB = case
    D, exp = _run(probe, M, N, K, a_mn, a_sw, 0, b_mn, b_sw, 0, b_row0, NB, tf32=1)
    assert _close(D, exp), f"max err {(D - exp).abs().max().item():.3e}"
