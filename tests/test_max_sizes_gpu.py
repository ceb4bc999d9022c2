"""GPU: the dense GEMM at the largest M and N the C ABI accepts (M, N < 2^31).

A problem with M = 2^31 - 1 (or N = 2^31 - 8, the largest multiple of 8) and the other two
extents 8 holds 32 GiB in each of its long operand and C.  The long operand is written on the
device in chunks by plain torch arithmetic from an integer formula, and the oracle rebuilds the
rows (or columns) it checks from the same formula on the host, so no input or expected value
comes from the kernels.  Integer entries keep every sum exact in fp32: the sampled outputs must
equal the oracle bit for bit, among them the last row (column) and the rows around tile edges
near 2^31.  Skipped when the device lacks the memory.
"""

import numpy as np
import pytest
import torch

import persistent_warp_specialized_gb300 as tg
from persistent_warp_specialized_gb300 import workloads as wl
from oracle import gemm as ogemm, mx

from gpu_helpers import VARIANTS, ensure_library

pytestmark = pytest.mark.gpu

BIG = 2 ** 31 - 1
CHUNK = 1 << 26


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_library()


def need_gib(n):
    free, _ = torch.cuda.mem_get_info()
    if free < n * (1 << 30):
        pytest.skip(f"needs {n} GiB of free device memory, {free >> 30} GiB free")


def formula(i, k, a, b, mod):
    """((i * a + k * b) mod mod) - mod // 2, elementwise on int64 arrays or tensors."""
    return (i * a + k * b) % mod - mod // 2


def fill_long(t, along_rows, a, b, mod):
    """t[i, k] (along_rows) or t[k, j] = formula(index along the long side, short index)."""
    long_n = t.shape[0] if along_rows else t.shape[1]
    short = torch.arange(t.shape[1] if along_rows else t.shape[0], device=t.device,
                         dtype=torch.int64)
    for s in range(0, long_n, CHUNK):
        e = min(long_n, s + CHUNK)
        idx = torch.arange(s, e, device=t.device, dtype=torch.int64)
        if along_rows:
            t[s:e] = formula(idx[:, None], short[None, :], a, b, mod).to(t.dtype)
        else:
            t[:, s:e] = formula(idx[None, :], short[:, None], a, b, mod).to(t.dtype)


def sample_indices(n, tile):
    """First, last and tile-edge indices near the end of a long extent of n, plus a few more."""
    picks = {0, 1, n - 1, n - 2, n // 2}
    last_tile = (n - 1) // tile * tile
    picks.update({last_tile, last_tile - 1, last_tile + 127, last_tile - tile})
    gen = np.random.default_rng(n)
    picks.update(int(x) for x in gen.integers(0, n, 8))
    return sorted(p for p in picks if 0 <= p < n)


@pytest.mark.parametrize("variant", ["auto"] + VARIANTS)
def test_largest_m(variant):
    need_gib(80)
    M, N, K = BIG, 8, 8
    dt = torch.bfloat16
    a = torch.empty((M, K), dtype=dt, device="cuda")
    fill_long(a, True, 37, 11, 7)
    b_cpu = wl.small_int_inputs(8, N, K, "bf16", lo=-2, hi=2, seed=5)[1]
    b = b_cpu.cuda()
    c = torch.empty((M, N), dtype=dt, device="cuda")
    c.view(torch.int16).fill_(-1)
    tg.tg_gemm_persistent_ex(a, b, c, M, N, K, "bf16", variant=variant)
    torch.cuda.synchronize()
    assert tg.tg_device_status() == 0
    rows = sample_indices(M, 256)
    got = wl.bits(c[rows].cpu())
    a_rows = torch.from_numpy(formula(np.array(rows, dtype=np.int64)[:, None],
                                      np.arange(K, dtype=np.int64)[None, :], 37, 11, 7)
                              .astype(np.float64)).to(dt)
    want = ogemm.gemm_ref(wl.bits(a_rows), wl.bits(b_cpu), "bf16")
    assert np.array_equal(got, want), rows
    del a, c
    torch.cuda.empty_cache()


@pytest.mark.parametrize("variant", ["auto"] + VARIANTS)
def test_largest_n(variant):
    need_gib(80)
    M, N, K = 8, BIG - 7, 8          # 2^31 - 8: the largest multiple of 8 below 2^31
    dt = torch.bfloat16
    b = torch.empty((K, N), dtype=dt, device="cuda")
    fill_long(b, False, 13, 5, 9)
    a_cpu = wl.small_int_inputs(M, 8, K, "bf16", lo=-2, hi=2, seed=6)[0]
    a = a_cpu.cuda()
    c = torch.empty((M, N), dtype=dt, device="cuda")
    c.view(torch.int16).fill_(-1)
    tg.tg_gemm_persistent_ex(a, b, c, M, N, K, "bf16", variant=variant)
    torch.cuda.synchronize()
    assert tg.tg_device_status() == 0
    cols = sample_indices(N, 512)
    got = wl.bits(c[:, cols].cpu())
    b_cols = torch.from_numpy(formula(np.array(cols, dtype=np.int64)[None, :],
                                      np.arange(K, dtype=np.int64)[:, None], 13, 5, 9)
                              .astype(np.float64)).to(dt)
    want = ogemm.gemm_ref(wl.bits(a_cpu), wl.bits(b_cols.contiguous()), "bf16")
    assert np.array_equal(got, want), cols
    del b, c
    torch.cuda.empty_cache()


def test_largest_k():
    # K = 2^31 - 8 with M = N = 8: one tile walks 2^25 k-blocks, the last one partial.  A and B
    # are zero except at a few k spread over the range (both sides of the last k-block's start
    # among them), so C is their exact sum: a k-block skipped, repeated or loaded at a wrong
    # coordinate changes it.
    need_gib(80)
    M, N, K = 8, 8, BIG - 7
    dt = torch.bfloat16
    ks = [0, 63, 64, 1 << 30, K - 72, K - 64 - 1, K - 57, K - 9, K - 1]
    gen = torch.Generator().manual_seed(9)
    a_cols = torch.randint(-3, 4, (M, len(ks)), generator=gen).to(dt)
    b_rows = torch.randint(-3, 4, (len(ks), N), generator=gen).to(dt)
    a = torch.zeros((M, K), dtype=dt, device="cuda")
    b = torch.zeros((K, N), dtype=dt, device="cuda")
    idx = torch.tensor(ks, dtype=torch.int64, device="cuda")
    a[:, idx] = a_cols.cuda()
    b[idx, :] = b_rows.cuda()
    c = torch.empty((M, N), dtype=dt, device="cuda")
    c.view(torch.int16).fill_(-1)
    tg.tg_gemm_persistent(a, b, c, M, N, K, "bf16")
    torch.cuda.synchronize()
    assert tg.tg_device_status() == 0
    want = ogemm.gemm_ref(wl.bits(a_cols), wl.bits(b_rows), "bf16")
    assert np.array_equal(wl.bits(c.cpu()), want)
    del a, b, c
    torch.cuda.empty_cache()


def test_mxfp8_beyond_one_pass_of_the_pack_grid():
    # 524297 k-blocks of 128: 65538 groups of 8, more than the 65535 a grid's y extent holds, so
    # the scale pack strides over them.  Sampled atoms (the last among them) against the
    # documented layout, then the GEMM at that K: A and B are zero except at a few k, one per
    # 32-element block and spread over the range, so C is their exact scaled sum, which the
    # oracle computes on the same entries with the same block scales gathered into a short K.
    need_gib(8)
    M = N = 8
    kb = 8 * 65535 + 17
    K = 128 * kb
    gen = torch.Generator().manual_seed(12)
    # scales 2^-3 .. 2^3: the six terms of a sum stay within 18 bits, exact in fp32
    sfa = torch.randint(124, 131, (M, K // 32), generator=gen).to(torch.uint8)
    sfb = torch.randint(124, 131, (N, K // 32), generator=gen).to(torch.uint8)
    pa = tg.mxfp8_pack(sfa.cuda(), K)
    pb = tg.mxfp8_pack(sfb.cuda(), K)
    torch.cuda.synchronize()
    row_blocks = 2                               # 8 rows pad to 256: two blocks of 128
    for k in [0, 7, 8, 65535 * 8 - 1, 65535 * 8, kb - 1]:
        for b in range(row_blocks):
            atom = pa[(k * row_blocks + b) * 512:(k * row_blocks + b + 1) * 512].cpu().numpy()
            want = np.zeros(512, np.uint8)
            for r in range(128):
                if b * 128 + r < M:
                    off = (r % 32) * 16 + (r // 32) * 4
                    want[off:off + 4] = sfa[b * 128 + r, 4 * k:4 * k + 4].numpy()
            assert np.array_equal(atom, want), (k, b)
    ks = [5, 32 * 1000 + 3, K // 2 + 7, 128 * (65535 * 8) - 32 + 1, K - 33, K - 1]
    e4m3 = lambda v: v.to(torch.float32).to(torch.float8_e4m3fn).view(torch.uint8)
    a_vals = torch.randint(-3, 4, (M, len(ks)), generator=gen).float()
    b_vals = torch.randint(-3, 4, (N, len(ks)), generator=gen).float()
    a = torch.zeros((M, K), dtype=torch.uint8, device="cuda")
    b = torch.zeros((N, K), dtype=torch.uint8, device="cuda")
    idx = torch.tensor(ks, dtype=torch.int64, device="cuda")
    a[:, idx] = e4m3(a_vals).cuda()
    b[:, idx] = e4m3(b_vals).cuda()
    c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    c.view(torch.int16).fill_(-1)
    tg.tg_gemm_mxfp8(a, pa, b, pb, c, M, N, K, "bf16")
    torch.cuda.synchronize()
    assert tg.tg_device_status() == 0
    # the same entries in a K of 32 per position, each block with its original scale
    blocks = [k // 32 for k in ks]
    assert len(set(blocks)) == len(blocks)
    a_c = torch.zeros((M, 32 * len(ks)), dtype=torch.uint8)
    b_c = torch.zeros((N, 32 * len(ks)), dtype=torch.uint8)
    a_c[:, 32 * torch.arange(len(ks)) + torch.tensor([k % 32 for k in ks])] = e4m3(a_vals)
    b_c[:, 32 * torch.arange(len(ks)) + torch.tensor([k % 32 for k in ks])] = e4m3(b_vals)
    want = mx.gemm_mxfp8_ref(a_c.numpy(), sfa[:, blocks].numpy(), b_c.numpy(),
                             sfb[:, blocks].numpy(), "bf16")
    assert np.array_equal(wl.bits(c.cpu()), want)
    del a, b, c, pa, pb
    torch.cuda.empty_cache()
