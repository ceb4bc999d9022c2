"""GPU parity: tg_gemm_persistent against the CPU oracle, element by element.

Small shapes span several tiles and ragged tails in M, N and K (the kernel tiles
128 x 256 x 64), integer-valued inputs must be bit-exact (every fp32 partial sum is an
exact integer, so any accumulation order gives the same bits: a wrong slot, phase or
accumulator shows up as a wrong value), and the degenerate cases have closed forms.
"""

import numpy as np
import pytest
import torch

import persistent_warp_specialized_gb300 as tg
from persistent_warp_specialized_gb300 import workloads as wl
from oracle import formats

from gpu_helpers import (VARIANTS, assert_within_tolerance, ensure_library, nan_filled, oracle_bits,
                         run_gpu)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_library()


SHAPES = [
    (128, 256, 64),     # exactly one tile, one k-block
    (1, 8, 8),          # smallest legal problem
    (300, 520, 200),    # 3 x 3 tiles, ragged M, N and K
    (129, 264, 72),     # one row / one 8-column strip past a tile, K tail of 8
    (257, 776, 136),
    (640, 1024, 320),   # 5 x 4 tiles, full
    (1000, 8, 16),      # a single column strip
    (8, 4000, 1032),
]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("shape", SHAPES)
def test_small_shapes_match_oracle(shape, dtype, variant):
    M, N, K = shape
    a, b = wl.make_inputs(M, N, K, dtype, "uniform", seed=M + N + K)
    assert_within_tolerance(run_gpu(a, b, dtype, variant=variant), oracle_bits(a, b, dtype),
                            dtype, f"{shape} {variant}")


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("dtype,K", [("f16", 512), ("bf16", 64), ("f16", 200), ("bf16", 40)])
def test_integer_inputs_are_bit_exact(dtype, K, variant):
    # entries in [-2, 2]: |C| <= 4K, exact in the output type (f16: 2048, bf16: 256)
    M, N = 300, 776
    a, b = wl.small_int_inputs(M, N, K, dtype, seed=K)
    assert np.array_equal(run_gpu(a, b, dtype, variant=variant), oracle_bits(a, b, dtype))


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_many_tiles_per_cta_with_short_k(dtype, variant):
    # 32 x 16 = 512 tiles (> 3 per SM); k_blocks = 3 is not a multiple of the 4 stages, the
    # case where indexing the consumer's slot by k instead of the phase goes wrong
    M, N, K = 4096, 4096, 192
    a, b = wl.small_int_inputs(M, N, K, dtype, lo=-1, hi=1, seed=9)
    assert np.array_equal(run_gpu(a, b, dtype, variant=variant), oracle_bits(a, b, dtype))


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_k_shorter_than_one_block_many_tiles(dtype, variant):
    M, N, K = 2048, 2048, 8          # k_blocks = 1: every phase is a new tile
    a, b = wl.small_int_inputs(M, N, K, dtype, seed=4)
    assert np.array_equal(run_gpu(a, b, dtype, variant=variant), oracle_bits(a, b, dtype))


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_identity_reproduces_operand(dtype, variant):
    n = 384
    eye = torch.eye(n, dtype=wl.TORCH_DTYPES[dtype])
    x, _ = wl.make_inputs(n, 8, 520, dtype, "uniform", seed=2)      # [384, 520]
    assert np.array_equal(run_gpu(eye, x, dtype, variant=variant), wl.bits(x))   # I . X = X
    y, _ = wl.make_inputs(300, 8, n, dtype, "uniform", seed=3)       # [300, 384]
    assert np.array_equal(run_gpu(y, eye, dtype, variant=variant), wl.bits(y))   # Y . I = Y


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("dtype,K", [("f16", 2048), ("bf16", 8192)])
def test_all_ones_give_k(dtype, K, variant):
    M, N = 384, 512
    t = wl.TORCH_DTYPES[dtype]
    c = run_gpu(torch.ones((M, K), dtype=t), torch.ones((K, N), dtype=t), dtype, variant=variant)
    assert np.array_equal(formats.decode(c, dtype), np.full((M, N), float(K)))


@pytest.mark.parametrize("plain", [False, True])
@pytest.mark.parametrize("variant", VARIANTS)
def test_split_tail_after_full_waves_is_bit_exact(variant, plain):
    # 2560 x 2560: 200 single tiles (152 + a last wave of 48) or 100 pair tiles (76 + 24);
    # 5120 x 2560: 100 wide pair tiles (76 + 24).  The last wave runs as half-width units
    # unless the plain page order is asked for
    M, N, K = (5120, 2560, 448) if variant == "wide" else (2560, 2560, 448)
    shape = tg.tg_gemm_launch_shape(M, N, K, variant, plain)
    assert (shape["units"] > shape["split_from"]) == (not plain)
    a, b = wl.small_int_inputs(M, N, K, "bf16", lo=-1, hi=1, seed=11)
    M_, K_ = a.shape
    a_d, b_d = a.cuda(), b.cuda()
    c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    c.view(torch.int16).fill_(-1)
    tg.tg_gemm_persistent_ex(a_d, b_d, c, M, N, K, "bf16", variant=variant, plain=plain)
    torch.cuda.synchronize()
    assert tg.tg_device_status() == 0
    assert np.array_equal(wl.bits(c.cpu()), oracle_bits(a, b, "bf16"))


@pytest.mark.parametrize("variant", VARIANTS)
def test_column_major_order_is_bit_exact(variant):
    M, N, K = 3000, 2304, 320
    a, b = wl.small_int_inputs(M, N, K, "f16", seed=13)
    a_d, b_d = a.cuda(), b.cuda()
    c = torch.empty((M, N), dtype=torch.float16, device="cuda")
    c.view(torch.int16).fill_(-1)
    tg.tg_gemm_persistent_ex(a_d, b_d, c, M, N, K, "f16", variant=variant, column_major=True)
    torch.cuda.synchronize()
    assert tg.tg_device_status() == 0
    assert np.array_equal(wl.bits(c.cpu()), oracle_bits(a, b, "f16"))


def test_k_zero_gives_zeros():
    c = torch.full((64, 64), 7.0, dtype=torch.bfloat16, device="cuda")
    a = torch.empty((64, 0), dtype=torch.bfloat16, device="cuda")
    b = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    tg.tg_gemm_persistent(a, b, c, 64, 64, 0, "bf16")
    torch.cuda.synchronize()
    assert bool((c == 0).all())


def test_runs_on_a_side_stream():
    M, N, K = 500, 600, 264
    a, b = wl.make_inputs(M, N, K, "bf16", "uniform", seed=21)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        got = run_gpu(a, b, "bf16", stream=s)
    assert_within_tolerance(got, oracle_bits(a, b, "bf16"), "bf16", "side stream")


def test_repeated_calls_are_deterministic():
    M, N, K = 1024, 1024, 1024
    a, b = wl.make_inputs(M, N, K, "bf16", "normal", seed=5)
    first = run_gpu(a, b, "bf16")
    for _ in range(3):
        assert np.array_equal(run_gpu(a, b, "bf16"), first)


def test_host_entry_point_round_trip():
    M, N, K = 700, 1032, 520
    a, b = wl.make_inputs(M, N, K, "f16", "uniform", seed=17)
    a_h, b_h = a.pin_memory(), b.pin_memory()
    c_h = torch.empty((M, N), dtype=torch.float16).pin_memory()
    a_d = torch.empty_like(a_h, device="cuda")
    b_d = torch.empty_like(b_h, device="cuda")
    c_d = torch.empty((M, N), dtype=torch.float16, device="cuda")
    tg.tg_gemm_persistent_host(a_h, b_h, c_h, a_d, b_d, c_d, M, N, K, "f16")
    torch.cuda.synchronize()
    assert_within_tolerance(wl.bits(c_h), oracle_bits(a, b, "f16"), "f16", "host entry")


def test_rejections_with_a_gpu():
    a = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    b = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    host = torch.zeros((64, 64), dtype=torch.bfloat16)
    with pytest.raises(tg.TgError) as e:                  # host memory where device is required
        tg.tg_gemm_persistent(host, b, a, 64, 64, 64, "bf16")
    assert e.value.code == tg.TG_ERR_ARG
    with pytest.raises(tg.TgError) as e:                  # C aliases A
        tg.tg_gemm_persistent(a, b, a, 64, 64, 64, "bf16")
    assert e.value.code == tg.TG_ERR_ARG
    big = torch.zeros(64 * 64 + 8, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(tg.TgError) as e:                  # misaligned by 2 bytes
        tg.tg_gemm_persistent(big.data_ptr() + 2, b, a, 64, 64, 64, "bf16")
    assert e.value.code == tg.TG_ERR_ALIGN
    torch.cuda.synchronize()


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("M,N,K", [(1000, 520, 384), (4000, 7000, 512), (300, 2056, 136),
                                   (8192, 8192, 256)])
def test_direct_store_epilogue_is_bit_exact(M, N, K, variant):
    # TG_EPILOGUE_DIRECT: 16-byte stores from registers, clipped at M and N by the kernel
    a, b = wl.small_int_inputs(M, N, K, "bf16", seed=M + K)
    c = nan_filled(M, N, "bf16")
    tg.tg_gemm_persistent_ex(a.cuda(), b.cuda(), c, M, N, K, "bf16", variant=variant, direct=True)
    torch.cuda.synchronize()
    assert tg.tg_device_status() == 0
    assert np.array_equal(wl.bits(c.cpu()), oracle_bits(a, b, "bf16"))


@pytest.mark.parametrize("variant", VARIANTS)
def test_direct_store_epilogue_fp16_within_tolerance(variant):
    M, N, K = 1024, 1024, 1024
    a, b = wl.make_inputs(M, N, K, "f16", "uniform", seed=2)
    c = nan_filled(M, N, "f16")
    tg.tg_gemm_persistent_ex(a.cuda(), b.cuda(), c, M, N, K, "f16", variant=variant, direct=True)
    torch.cuda.synchronize()
    assert_within_tolerance(wl.bits(c.cpu()), oracle_bits(a, b, "f16"), "f16", "direct epilogue")


def _two_term(pairs, dtype, M=256, N=512, K=64, w=0.5):
    """A, B with C[i, j] = x_i + w y_i for (x_i, y_i) = pairs[i % len(pairs)]: A holds x in
    column 0 and y in column 1, B holds ones in row 0 and w in row 1, zeros elsewhere.
    Every product and the one non-trivial sum are exact in fp32, so the kernel's output must
    be the oracle's rounding of the exact sum, bit for bit."""
    tdt = wl.TORCH_DTYPES[dtype]
    a = torch.zeros((M, K), dtype=torch.float64)
    for i in range(M):
        a[i, 0], a[i, 1] = pairs[i % len(pairs)]
    b = torch.zeros((K, N), dtype=torch.float64)
    b[0, :] = 1.0
    b[1, :] = w
    a16, b16 = a.to(tdt), b.to(tdt)
    assert torch.equal(a16.double(), a) and torch.equal(b16.double(), b), "inputs must be exact"
    return a16.contiguous(), b16.contiguous()


@pytest.mark.parametrize("variant", VARIANTS)
def test_fp16_outputs_overflow_to_inf_as_rne_does(variant):
    # 65504 is the largest finite fp16; sums below the midpoint 65520 stay 65504, the midpoint
    # itself ties to even (the infinity), beyond it is inf, and the same on the negative side
    big = 65504.0
    pairs = [(big, 0.0), (big, 16.0), (big, 30.0), (big, 32.0), (big, 64.0), (big, big),
             (32768.0, big), (-big, -30.0), (-big, -32.0), (-big, -big), (60000.0, 10000.0),
             (1.0, 2.0)]
    a, b = _two_term(pairs, "f16")
    got = run_gpu(a, b, "f16", variant=variant)
    want = oracle_bits(a, b, "f16")
    assert np.array_equal(got, want)
    vals = formats.decode(want, "f16")
    assert np.isposinf(vals).any() and np.isneginf(vals).any() and (vals == big).any()


@pytest.mark.parametrize("variant", VARIANTS)
def test_fp16_subnormal_outputs_round_to_nearest_even(variant):
    # u = 2^-24 is the least fp16 subnormal; x + y/2 with y = u puts the exact sum half an ulp
    # between two subnormals: 0.5 u -> 0, 1.5 u -> 2u, 2.5 u -> 2u, 3.5 u -> 4u (ties to even)
    u = 2.0 ** -24
    pairs = [(0.0, u), (u, u), (2 * u, u), (3 * u, u), (2.0 ** -14, -u), (-u, -u), (1000 * u, u),
             (2.0 ** -15, 2 * u),
             # normal inputs whose sum cancels into the subnormal range: 2^-13 - (2^-13 - u) = u
             (2.0 ** -13, -(2.0 ** -12 - 2.0 ** -23))]
    a, b = _two_term(pairs, "f16")
    got = run_gpu(a, b, "f16", variant=variant)
    want = oracle_bits(a, b, "f16")
    assert np.array_equal(got, want)
    vals = formats.decode(want, "f16")
    assert ((vals != 0) & (np.abs(vals) < 2.0 ** -14)).any()


@pytest.mark.parametrize("variant", VARIANTS)
def test_bf16_outputs_at_the_top_of_the_range(variant):
    # the largest finite bf16 is (2 - 2^-7) 2^127; sums that stay below the rounding midpoint to
    # 2^128 keep it, sums beyond the fp32 range are inf in the accumulator and in the oracle
    top = (2.0 - 2.0 ** -7) * 2.0 ** 127
    pairs = [(2.0 ** 127, 2.0 ** 127), (top, 0.0), (top, top * 2.0 ** -8), (top, top),
             (-top, -top), (2.0 ** 126, 2.0 ** 127), (1.0, 2.0)]
    a, b = _two_term(pairs, "bf16")
    got = run_gpu(a, b, "bf16", variant=variant)
    want = oracle_bits(a, b, "bf16")
    assert np.array_equal(got, want)
    vals = formats.decode(want, "bf16")
    assert np.isposinf(vals).any() and np.isneginf(vals).any() and (vals == top).any()


@pytest.mark.parametrize("variant", VARIANTS)
def test_bf16_subnormals_are_kept(variant):
    # bf16 has fp32's exponent range, so its subnormals (multiples of s = 2^-133) are fp32
    # subnormals too: the tensor core keeps them (no flush to zero) in the inputs, in products
    # and in the fp32 sum, and the output rounds to nearest even among them
    s = 2.0 ** -133
    w = 2.0 ** -60
    pairs = [(2.0 ** -127, 0.0), (s, 0.0), (0.0, 2.0 ** -70),          # copies and a product
             (2.0 ** -127, 2.0 ** -70), (64 * s, 2.0 ** -74),            # 72 s; 64.5 s -> 64 s
             (65 * s, 2.0 ** -74), (-3 * s, -(2.0 ** -74)),                # 66 s; -4 s
             (2.0 ** -126, -(2.0 ** -67))]                              # normal - half: 64 s
    a, b = _two_term(pairs, "bf16", w=w)
    got = run_gpu(a, b, "bf16", variant=variant)
    want = oracle_bits(a, b, "bf16")
    assert np.array_equal(got, want)
    vals = formats.decode(want, "bf16")
    assert ((vals != 0) & (np.abs(vals) < 2.0 ** -126)).sum() > vals.size // 2
