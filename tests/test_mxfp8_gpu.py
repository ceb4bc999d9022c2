"""GPU: the block-scaled MXFP8 GEMM against the oracle (oracle.mx).

* integer elements with power-of-two scales: every partial sum is exact in fp32, so the
  CUDA path must equal the oracle bit for bit -- this is what catches a scale read from the
  wrong row, column, k-block or pipeline stage;
* MX-quantized normal draws: the acceptance bound |C - C_ref| <= 5e-3 + 1e-2 |C_ref| and the
  tighter fp32 accumulation bound 2 ulp(C_ref) + gamma_K (|A| . |B|);
* the debug trace against the oracle's schedule; the watchdog; empty and K = 0 problems;
* the full 8192^3 workload on sampled rows and columns.
"""

import numpy as np
import pytest
import torch

import persistent_warp_specialized_gb300 as tg
from persistent_warp_specialized_gb300 import workloads as wl
from oracle import formats, mx, schedule

from gpu_helpers import ATOL, RTOL, ensure_library, nan_filled

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_library()


def device_inputs(a, sa, b, sb):
    """Device copies of A and B and the packed device scales of SA and SB."""
    K = a.shape[1]
    return a.cuda(), tg.mxfp8_pack(sa.cuda(), K), b.cuda(), tg.mxfp8_pack(sb.cuda(), K)


MX_VARIANTS = ["single", "pair"]


def run_mx(a, sa, b, sb, out="bf16", debug=False, variant="auto", **kw):
    M, K = a.shape
    N = b.shape[0]
    c = nan_filled(M, N, out)
    dev = device_inputs(a, sa, b, sb)
    if debug:
        tg.tg_gemm_mxfp8_debug(*dev, c, M, N, K, out, variant=variant, **kw)
    elif variant == "auto":
        tg.tg_gemm_mxfp8(*dev, c, M, N, K, out)
    else:
        tg.tg_gemm_mxfp8_ex(*dev, c, M, N, K, out, variant=variant)
    torch.cuda.synchronize()
    assert tg.tg_device_status() == 0
    return wl.bits(c.cpu())


def ref_bits(a, sa, b, sb, out="bf16"):
    return mx.gemm_mxfp8_ref(a.numpy(), sa.numpy(), b.numpy(), sb.numpy(), out)


def check_tolerance(c_bits, r_bits, a, sa, b, sb, out, what, gate=True):
    """The acceptance gate (unless ``gate`` is False) and the fp32 accumulation bound."""
    c = formats.decode(c_bits, out)
    r = formats.decode(r_bits, out)
    assert np.isfinite(c).all(), f"{what}: non-finite outputs"
    err = np.abs(c - r)
    if gate:
        bad = err > ATOL + RTOL * np.abs(r)
        assert not bad.any(), f"{what}: {int(bad.sum())} outside the gate, first {np.argwhere(bad)[:4].tolist()}"
    s = np.abs(mx.scaled(a.numpy(), sa.numpy())) @ np.abs(mx.scaled(b.numpy(), sb.numpy())).T
    K = a.shape[1]
    u = 2.0 ** -23
    bound = 2.0 * formats.ulp(r_bits, out) + K * u / (1 - K * u) * s
    bad = err > bound
    assert not bad.any(), f"{what}: {int(bad.sum())} outside the fp32 accumulation bound"


def packed_layout(sf, K):
    """The packed layout as the C header defines it, written out element by element."""
    rows = sf.shape[0]
    row_blocks = 2 * ((rows + 255) // 256)
    out = np.zeros((K // 128) * row_blocks * 512, np.uint8)
    for k in range(K // 128):
        for b in range(row_blocks):
            for r in range(128):
                if b * 128 + r < rows:
                    for j in range(4):
                        out[(k * row_blocks + b) * 512 + (r % 32) * 16 + (r // 32) * 4 + j] = \
                            sf[b * 128 + r, 4 * k + j]
    return out


@pytest.mark.parametrize("rows,K", [(1, 128), (128, 256), (300, 384), (513, 512), (256, 128)])
def test_pack_scales_is_the_documented_layout(rows, K):
    gen = torch.Generator().manual_seed(rows + K)
    sf = torch.randint(0, 256, (rows, K // 32), generator=gen).to(torch.uint8)
    packed = torch.full((tg.tg_mxfp8_scale_bytes(rows, K),), 0xAB, dtype=torch.uint8,
                        device="cuda")
    tg.tg_mxfp8_pack_scales(sf.cuda(), packed, rows, K)
    torch.cuda.synchronize()
    assert np.array_equal(packed.cpu().numpy(), packed_layout(sf.numpy(), K))


@pytest.mark.parametrize("variant", MX_VARIANTS)
@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (512, 768, 512), (1000, 520, 384),
                                   (4096, 4096, 128), (2560, 2560, 256), (8, 8, 128),
                                   (384, 640, 256)])
def test_integer_inputs_are_bit_exact(M, N, K, variant):
    a, sa, b, sb = wl.mx_int_inputs(M, N, K, seed=M + N + K)
    assert np.array_equal(run_mx(a, sa, b, sb, variant=variant), ref_bits(a, sa, b, sb))


@pytest.mark.parametrize("variant", MX_VARIANTS)
@pytest.mark.parametrize("out", ["bf16", "f16"])
@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (1024, 1024, 1024), (1000, 520, 2048),
                                   (4000, 7000, 2048)])
def test_quantized_normal_inputs_within_tolerance(M, N, K, out, variant):
    a, sa, b, sb = wl.make_mx_inputs(M, N, K, seed=7 * M + K)
    check_tolerance(run_mx(a, sa, b, sb, out, variant=variant), ref_bits(a, sa, b, sb, out), a, sa,
                    b, sb, out, f"{M}x{N}x{K} {out} {variant}")


@pytest.mark.parametrize("variant", MX_VARIANTS)
def test_scales_span_the_e8m0_range(variant):
    # element blocks scaled from 2^-60 to 2^+60 (all products stay normal in fp32).  Here an
    # output can be the small residue of block terms 10^7 .. 10^13 times larger that cancel,
    # and no fp32 accumulation order meets the relative gate there (an in-order fp32 sum of
    # the exact block terms misses it on 8 of these 65536 outputs), so only the fp32
    # accumulation bound is asserted.
    M, N, K = 256, 256, 256
    a, _, b, _ = wl.mx_int_inputs(M, N, K, seed=3)
    gen = torch.Generator().manual_seed(11)
    sa = torch.randint(127 - 30, 127 + 31, (M, K // 32), generator=gen).to(torch.uint8)
    sb = torch.randint(127 - 30, 127 + 31, (N, K // 32), generator=gen).to(torch.uint8)
    check_tolerance(run_mx(a, sa, b, sb, variant=variant), ref_bits(a, sa, b, sb), a, sa, b, sb,
                    "bf16", "scales", gate=False)


@pytest.mark.parametrize("variant", MX_VARIANTS)
@pytest.mark.parametrize("plain,column_major", [(False, False), (True, False), (False, True)])
@pytest.mark.parametrize("M,N,K", [(4096, 4096, 128), (4000, 7000, 128), (256, 256, 256),
                                   (8192, 8192, 128)])
def test_kernel_followed_the_schedule(M, N, K, plain, column_major, variant):
    shape = tg.tg_gemm_launch_shape(M, N, K, variant, plain, mxfp8=True)
    units = shape["units"]
    trace = torch.full((units, 5), -7, dtype=torch.int32, device="cuda")
    a, sa, b, sb = wl.mx_int_inputs(M, N, K, seed=5)
    got_c = run_mx(a, sa, b, sb, debug=True, variant=variant, trace=trace, plain=plain,
                   column_major=column_major)
    want = schedule.enumerate_units(shape["m_tiles"], shape["n_tiles"], shape["workers"],
                                    tg.tg_gemm_config()["group"], split_tail=not plain,
                                    column_major=column_major)
    assert len(want) == units
    by_unit = {worker + w * shape["workers"]: (worker, w, bx, by, part)
               for (worker, w, bx, by, part) in want}
    got = trace.cpu().numpy()
    for u in range(units):
        assert tuple(int(v) for v in got[u]) == by_unit[u], u
    assert np.array_equal(got_c, ref_bits(a, sa, b, sb))


@pytest.mark.parametrize("variant,cta", [(v, 0) for v in MX_VARIANTS] + [("pair", 1)])
def test_watchdog_fires_and_context_survives(variant, cta):
    # CTA ``cta``'s producer skips phase 2; in the pair, CTA 1 (odd) leaves a phase that only
    # the even CTA armed, which the abort path must still see land
    M, N, K = 512, 512, 1024
    a, sa, b, sb = wl.mx_int_inputs(M, N, K, seed=1)
    dev = device_inputs(a, sa, b, sb)
    c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(tg.TgError) as e:
        # phase 2 exists in both kernels (single: k-blocks 0..7; pair: stages of 2 k-blocks)
        tg.tg_gemm_mxfp8_debug(*dev, c, M, N, K, "bf16", variant=variant, watchdog_ns=20_000_000,
                               inject_skip_phase=(cta << 32) + 2)
    assert e.value.code == tg.TG_ERR_TIMEOUT
    assert tg.tg_device_status() == 0
    assert np.array_equal(run_mx(a, sa, b, sb, variant=variant), ref_bits(a, sa, b, sb))


def test_empty_and_zero_k():
    c = nan_filled(64, 64, "bf16")
    z = torch.zeros(16, dtype=torch.uint8, device="cuda")   # K = 0: nothing is read
    assert tg.tg_gemm_mxfp8(z, z, z, z, c, 64, 64, 0, "bf16") == 0
    torch.cuda.synchronize()
    assert (c.float() == 0).all()
    assert tg.tg_gemm_mxfp8(None, None, None, None, None, 0, 64, 128, "bf16") == 0


@pytest.mark.parametrize("variant", MX_VARIANTS)
def test_full_size_workload_sampled_entries(variant):
    M, N, K, seed = wl.MX_WORKLOADS["mxfp8_8192"]
    a, sa, b, sb = wl.make_mx_inputs(M, N, K, seed)
    c = run_mx(a, sa, b, sb, variant=variant)
    rng = np.random.default_rng(0)
    rows = np.concatenate([[0, M - 1], rng.choice(M, 62, replace=False)])
    cols = np.concatenate([[0, N - 1], rng.choice(N, 62, replace=False)])
    want = mx.gemm_mxfp8_ref_entries(a.numpy(), sa.numpy(), b.numpy(), sb.numpy(), rows, cols)
    got = c[np.ix_(rows, cols)]
    cv, rv = formats.decode(got, "bf16"), formats.decode(want, "bf16")
    assert np.isfinite(cv).all()
    assert (np.abs(cv - rv) <= ATOL + RTOL * np.abs(rv)).all()


@pytest.mark.parametrize("variant", MX_VARIANTS)
def test_group_width_option_followed(variant):
    M, N, K, group = 4096, 4096, 128, 12
    shape = tg.tg_gemm_launch_shape(M, N, K, variant, mxfp8=True)
    units = shape["units"]
    trace = torch.full((units, 5), -7, dtype=torch.int32, device="cuda")
    a, sa, b, sb = wl.mx_int_inputs(M, N, K, seed=12)
    got_c = run_mx(a, sa, b, sb, debug=True, variant=variant, trace=trace, group=group)
    want = schedule.enumerate_units(shape["m_tiles"], shape["n_tiles"], shape["workers"], group,
                                    split_tail=True)
    by_unit = {worker + w * shape["workers"]: (worker, w, bx, by, part)
               for (worker, w, bx, by, part) in want}
    got = trace.cpu().numpy()
    for u in range(units):
        assert tuple(int(v) for v in got[u]) == by_unit[u], u
    assert np.array_equal(got_c, ref_bits(a, sa, b, sb))


def test_mxfp8_gemm_convenience_matches_the_oracle():
    M, N, K = 300, 520, 256
    a, sa, b, sb = wl.mx_int_inputs(M, N, K, seed=4)
    c = tg.mxfp8_gemm(a.cuda(), sa.cuda(), b.cuda(), sb.cuda())
    torch.cuda.synchronize()
    assert c.shape == (M, N) and c.dtype == torch.bfloat16
    assert np.array_equal(wl.bits(c.cpu()), ref_bits(a, sa, b, sb))


@pytest.mark.parametrize("M,N,K", [(512, 512, 8192), (256, 1024, 4096)])
def test_auto_long_k_below_a_wave(M, N, K):
    # tg_gemm_mxfp8 takes the CTA-pair kernel here (fewer pair tiles than a wave, K >= 4096):
    # the same gate and bound as every other MXFP8 parity case
    assert tg.tg_gemm_launch_shape(M, N, K, mxfp8=True)["variant"] == tg.TG_VARIANT_PAIR
    a, sa, b, sb = wl.make_mx_inputs(M, N, K, seed=M + K)
    check_tolerance(run_mx(a, sa, b, sb), ref_bits(a, sa, b, sb), a, sa, b, sb, "bf16",
                    "auto long K")


def _block_terms(rows, out_rows=256, N=256, K=128):
    """A, SFA, B, SFB with C[i, j] = sum_t x_t 2^(e_t) over the terms (x_t, e_t) of
    rows[i % len(rows)] (at most K / 32 terms, one per 32-element block): A holds x_t at the first
    element of block t with scale 2^(e_t); B holds 1.0 there with scale 1.  Every partial sum in
    the cases below is exact in fp32, in any order."""
    a = torch.zeros((out_rows, K), dtype=torch.float32)
    sa = torch.full((out_rows, K // 32), 127, dtype=torch.uint8)
    for i in range(out_rows):
        for t, (x, e) in enumerate(rows[i % len(rows)]):
            a[i, 32 * t] = x
            sa[i, t] = 127 + e
    b = torch.zeros((N, K), dtype=torch.float32)
    b[:, 0::32] = 1.0
    sb = torch.full((N, K // 32), 127, dtype=torch.uint8)
    a8 = a.to(torch.float8_e4m3fn)
    assert torch.equal(a8.float(), a), "elements must be exact in E4M3"
    return (a8.view(torch.uint8).contiguous(), sa, b.to(torch.float8_e4m3fn).view(torch.uint8)
            .contiguous(), sb)


@pytest.mark.parametrize("variant", MX_VARIANTS)
def test_output_rounding_at_the_edges_of_fp16_and_bf16(variant):
    u = -24                                   # 2^-24: the least fp16 subnormal
    f16_rows = [
        [(448.0, 7)],                         # 57344: finite
        [(448.0, 7), (1.0, 13), (-1.0, 4)],   # 65520: the midpoint above 65504, ties to inf
        [(448.0, 7), (1.0, 13)],              # 65536: inf
        [(-448.0, 7), (-1.0, 13), (1.0, 4)],  # -65520: -inf
        [(448.0, 7), (1.75, 12), (-1.0, 4)],  # 64496: halfway to 64512, ties to it (finite)
        [(1.5, u)],                           # 1.5 u: ties to 2u
        [(0.5, u)],                           # 0.5 u: ties to 0
        [(1.0, u), (1.0, u - 2)],             # 1.25 u: u
        [(1.0, -14), (-1.0, u)],              # 2^-14 - u: the largest subnormal
    ]
    a, sa, b, sb = _block_terms(f16_rows)
    got = run_mx(a, sa, b, sb, "f16", variant=variant)
    want = ref_bits(a, sa, b, sb, "f16")
    assert np.array_equal(got, want)
    vals = formats.decode(want, "f16")
    assert np.isposinf(vals).any() and np.isneginf(vals).any()
    assert ((vals != 0) & (np.abs(vals) < 2.0 ** -14)).any()
    bf16_rows = [
        [(448.0, 120)],                       # 5.96e38: past the fp32 range, inf
        [(-448.0, 120)],                      # -inf
        [(1.0, 127), (1.0, 126)],             # 1.5 x 2^127: finite, exact
        [(1.75, 127)],                        # 2.98e38: finite
    ]
    a, sa, b, sb = _block_terms(bf16_rows)
    got = run_mx(a, sa, b, sb, "bf16", variant=variant)
    want = ref_bits(a, sa, b, sb, "bf16")
    assert np.array_equal(got, want)
    vals = formats.decode(want, "bf16")
    assert np.isposinf(vals).any() and np.isneginf(vals).any() and np.isfinite(vals).any()
