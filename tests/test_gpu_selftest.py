"""tcgen05 building blocks on the GPU: the three operand forms of the
backward kernel's MMAs against a float64 matmul of the same 16-bit inputs,
and the bounded semaphore wait."""
import time

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("N", [64, 128])
@pytest.mark.parametrize("K", [64, 128])
def test_umma_forms(fa, cuda_device, mode, N, K, dtype):
    g = torch.Generator().manual_seed(1000 * mode + 10 * N + K)
    if mode == 0:       # C = A B^T, A [128, K], B [N, K]
        A = torch.randn((128, K), generator=g).to(dtype)
        B = torch.randn((N, K), generator=g).to(dtype)
        ref = A.double() @ B.double().T
    elif mode == 1:     # C = A B, A [128, K] (in tensor memory), B [K, N]
        A = torch.randn((128, K), generator=g).to(dtype)
        B = torch.randn((K, N), generator=g).to(dtype)
        ref = A.double() @ B.double()
    else:               # C = A^T B, A [K, 128], B [K, N]
        A = torch.randn((K, 128), generator=g).to(dtype)
        B = torch.randn((K, N), generator=g).to(dtype)
        ref = A.double().T @ B.double()
    C, err = fa.selftest_umma(mode, A.cuda(), B.cuda(), N, K)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    diff = (C.double().cpu() - ref).abs().max().item()
    assert diff <= 1e-4 * max(1.0, ref.abs().max().item()), diff


def test_semaphore_wait_that_cannot_succeed_times_out(fa, cuda_device):
    sem = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.time()
    err = fa.selftest_semaphore(sem, target=1, budget_ns=50_000_000)   # nothing ever adds 1
    torch.cuda.synchronize()
    assert time.time() - t0 < 10.0
    assert int(err.item()) != 0
    assert int(sem.item()) == 0
    # the context is still usable
    x = torch.ones(4, device="cuda") * 2
    assert float(x.sum().item()) == 8.0


def test_semaphore_wait_that_succeeds(fa, cuda_device):
    sem = torch.full((1,), 5, dtype=torch.int32, device="cuda")
    err = fa.selftest_semaphore(sem, target=3, budget_ns=50_000_000)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert int(sem.item()) == 6


def test_tmem_16x256b_load_layout(fa, cuda_device):
    """Register 4k + e of thread t, lane offset h: lane 32 w + 16 h + t/4 + 8 (e/2),
    column 8k + 2 (t%4) + e%2 (w = warp, t = thread in the warp)."""
    out = fa.selftest_tmem_layout(0)
    bad = []
    for r in range(128):
        w, t = divmod(r, 32)
        for h in range(2):
            for reg in range(16):
                k, e = divmod(reg, 4)
                lane = 32 * w + 16 * h + t // 4 + 8 * (e // 2)
                col = 8 * k + 2 * (t % 4) + e % 2
                got = int(out[r, 16 * h + reg])
                if got != (lane << 8 | col):
                    bad.append((r, h, reg, got >> 8, got & 255, lane, col))
    assert not bad, bad[:8]


def test_tmem_16x128b_store_layout(fa, cuda_device):
    """Register 2k + e of thread t, lane offset h goes to lane 32 w + 16 h + t/4 + 8e,
    column 4k + t%4; columns 16..31 stay untouched."""
    out = fa.selftest_tmem_layout(1)
    want = torch.zeros((128, 32), dtype=torch.int64)
    for r in range(128):
        w, t = divmod(r, 32)
        for h in range(2):
            for reg in range(8):
                k, e = divmod(reg, 2)
                lane = 32 * w + 16 * h + t // 4 + 8 * e
                col = 4 * k + t % 4
                want[lane, col] = 0x80000000 | r << 8 | h << 4 | reg
    bad = (out != want).nonzero().tolist()
    assert not bad, [(l, c, hex(int(out[l, c])), hex(int(want[l, c]))) for l, c in bad[:8]]
