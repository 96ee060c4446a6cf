"""GPU self-test of the tcgen05 building blocks: shared-memory descriptors
(K-major and MN-major operands), the kind::f16 instruction descriptor (bf16
and fp16) and the TMEM accumulator layout for M = 64 and M = 128, against a
float64 matmul of the same 16-bit values."""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def _lanes_m64():
    """Accumulator rows of an M = 64 MMA by TMEM lane: 16 rows in each of the
    four 32-lane sub-partitions."""
    return [32 * (r // 16) + r % 16 for r in range(64)]


@pytest.mark.parametrize("M,N,K,a_mn,b_mn,bf16", [
    (128, 128, 64, 0, 0, 1), (128, 256, 64, 0, 1, 1), (128, 64, 128, 0, 0, 0), (128, 128, 32, 0, 1, 0),
    (64, 64, 64, 0, 0, 1), (64, 256, 64, 0, 1, 1), (64, 128, 128, 0, 1, 0),
    (64, 64, 64, 1, 1, 0), (64, 128, 64, 1, 1, 0), (128, 64, 64, 1, 0, 1),
])
def test_mma_layouts(gpu_lib, M, N, K, a_mn, b_mn, bf16):
    import torch
    lib = gpu_lib.load()
    lib.atlas_mem_selftest_mma.argtypes = [ctypes.c_int] * 6 + [ctypes.c_void_p] * 5
    lib.atlas_mem_selftest_mma.restype = ctypes.c_int
    g = torch.Generator().manual_seed(M * 1000 + N + K)
    dt = torch.bfloat16 if bf16 else torch.float16
    A = torch.randn(M, K, generator=g).to(dt)
    Bm = torch.randn(N, K, generator=g).to(dt)
    ref = A.double() @ Bm.double().T
    Bdev = (Bm.T.contiguous() if b_mn else Bm).cuda()
    Adev = (A.T.contiguous() if a_mn else A).cuda()
    raw = torch.full((128, N), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = lib.atlas_mem_selftest_mma(M, N, K, a_mn, b_mn, bf16, Adev.data_ptr(), Bdev.data_ptr(), raw.data_ptr(),
                                    st.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert st.item() == 0, "bounded wait gave up"
    raw = raw.double().cpu()
    lanes = list(range(128)) if M == 128 else _lanes_m64()
    got = raw[lanes]
    err = (got - ref).abs().max().item() / ref.abs().max().item()
    if err > 1e-6:
        # report where the rows landed to help read the layout
        hits = {}
        for r in range(M):
            d = (raw - ref[r]).abs().max(dim=1).values
            hits[r] = int(d.argmin())
        print("row -> lane", hits)
    assert err < 1e-6, err


def test_tmem_ld_16x32bx2_layout(gpu_lib):
    """Thread t of warp w gets accumulator row 16 w + t % 16, columns
    col + 16 (t // 16) + j.  D[r][c] = 256 r + c exactly, so every loaded
    value names its own row and column.  Lanes 16-31 of each sub-partition,
    marked before the M = 64 MMA, must come back unchanged."""
    import torch
    lib = gpu_lib.load()
    lib.atlas_mem_selftest_ld16x2.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    lib.atlas_mem_selftest_ld16x2.restype = ctypes.c_int
    N, K, col = 128, 16, 32
    A = torch.zeros(64, K)
    A[:, 0] = torch.arange(64, dtype=torch.float32)
    A[:, 1] = 1.0
    Bm = torch.zeros(N, K)
    Bm[:, 0] = 256.0
    Bm[:, 1] = torch.arange(N, dtype=torch.float32)
    A, Bm = A.to(torch.bfloat16), Bm.to(torch.bfloat16)
    raw = torch.full((128, 16), -1.0, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    Adev, Bdev = A.cuda(), Bm.cuda()          # keep the device copies alive during the launch
    rc = lib.atlas_mem_selftest_ld16x2(N, K, Adev.data_ptr(), Bdev.data_ptr(), raw.data_ptr(), col,
                                       st.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert st.item() != 1, "bounded wait gave up"
    assert st.item() == 0, "an M = 64 MMA changed TMEM lanes 16-31"
    raw = raw.cpu().numpy().astype(np.int64)
    got = {(w, t, j): (int(raw[32 * w + t, j]) // 256, int(raw[32 * w + t, j]) % 256)
           for w in range(4) for t in range(32) for j in range(16)}
    want = {(w, t, j): (16 * w + t % 16, col + 16 * (t // 16) + j) for w in range(4) for t in range(32) for j in range(16)}
    if got != want:
        for t in range(32):
            print("warp 0 thread", t, [got[(0, t, j)] for j in (0, 1, 2, 15)])
        print("warp 1 thread 0", [got[(1, 0, j)] for j in (0, 1, 15)])
    assert got == want


def test_bounded_wait_gives_up_and_the_context_stays_usable(gpu_lib):
    """Failure detection without a GPU fault: a kernel waits on an mbarrier
    that nothing arrives at, with the library's bounded wait limited to about
    a millisecond.  It gives up, reports ATLAS_ERR_TIMEOUT in its status
    word and returns; a memory-layer forward afterwards still matches the
    oracle."""
    import torch

    import test_learned_neural_gb300 as tln
    from harness import WORKLOADS
    from tests.gpu_common import TOL, compare
    lib = gpu_lib.load()
    lib.atlas_mem_selftest_wait_timeout.argtypes = [ctypes.c_longlong, ctypes.c_void_p, ctypes.c_void_p,
                                                    ctypes.c_void_p]
    lib.atlas_mem_selftest_wait_timeout.restype = ctypes.c_int
    assert lib.atlas_mem_selftest_wait_timeout(0, None, None, None) == tln.ATLAS_ERR_INVALID_ARG
    budget = 2_000_000                                   # SM cycles, about 1 ms
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    waited = torch.zeros(1, dtype=torch.int64, device="cuda")
    rc = lib.atlas_mem_selftest_wait_timeout(budget, st.data_ptr(), waited.data_ptr(),
                                             torch.cuda.current_stream().cuda_stream)
    assert rc == tln.ATLAS_OK
    torch.cuda.synchronize()
    assert int(st.item()) == tln.ATLAS_ERR_TIMEOUT
    assert budget <= int(waited.item()) < 100 * budget
    w = WORKLOADS["titans_mlp"].scaled(B=1, H=2, T=128)
    errs = compare(w)
    assert errs["y"] <= TOL["bf16"] and errs["W0"] <= TOL["bf16"]
