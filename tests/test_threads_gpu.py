"""GPU: the C ABI called from several host threads at once.

The library's host state is the per-device facts (set up once under a lock), the tensor-map
encoder's entry point (looked up once) and a thread-local error message.  ctypes releases the
interpreter lock for the duration of each call, so these threads are inside the library
concurrently: each issues repeated GEMMs on a stream of its own (the dense kernels and the MXFP8
GEMM with its scale packs), one more makes calls that fail, and every thread's outputs and
messages must be its own.
"""

import threading

import numpy as np
import pytest
import torch

import persistent_warp_specialized_gb300 as tg
from persistent_warp_specialized_gb300 import workloads as wl
from oracle import mx

from gpu_helpers import ensure_library, nan_filled, oracle_bits

pytestmark = pytest.mark.gpu

DENSE = [(512, 768, 256, "bf16", "single"), (1024, 512, 384, "f16", "pair"),
         (768, 1024, 512, "bf16", "wide"), (300, 520, 1000, "bf16", "auto")]
REPEATS = 12


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_library()


def test_concurrent_calls_from_host_threads():
    inputs = [wl.small_int_inputs(M, N, K, dt, seed=M + K) for (M, N, K, dt, _) in DENSE]
    a_mx, sa_mx, b_mx, sb_mx = wl.mx_int_inputs(384, 512, 512, seed=4)
    results, errors, messages = {}, [], {}
    start = threading.Barrier(len(DENSE) + 2, timeout=120)   # a thread that fails early breaks it

    # every thread allocates and works on a stream of its own, so that a block the caching
    # allocator hands out again is never still in use on another thread's stream
    def dense(t):
        try:
            M, N, K, dt, v = DENSE[t]
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                a, b = (x.cuda() for x in inputs[t])
                c = nan_filled(M, N, dt)
                start.wait()
                for _ in range(REPEATS):
                    tg.tg_gemm_persistent_ex(a, b, c, M, N, K, dt, stream=s, variant=v)
                s.synchronize()
                results[t] = wl.bits(c.cpu())
        except Exception as e:          # reported by the main thread
            errors.append((t, repr(e)))

    def block_scaled():
        try:
            M, N, K = 384, 512, 512
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                a, b = a_mx.cuda(), b_mx.cuda()
                c = nan_filled(M, N, "bf16")
                start.wait()
                for _ in range(REPEATS):
                    sa = tg.mxfp8_pack(sa_mx.cuda(), K, stream=s)
                    sb = tg.mxfp8_pack(sb_mx.cuda(), K, stream=s)
                    tg.tg_gemm_mxfp8(a, sa, b, sb, c, M, N, K, "bf16", stream=s)
                s.synchronize()
                results["mx"] = wl.bits(c.cpu())
        except Exception as e:
            errors.append(("mx", repr(e)))

    def failing():
        # a size error whose message names this call's M, different on every call
        start.wait()
        for i in range(REPEATS):
            try:
                tg.tg_gemm_persistent(None, None, None, -1 - i, 64, 64, "bf16")
                messages[i] = None
            except tg.TgError as e:
                messages[i] = (i, e.code, str(e), tg.tg_last_error())

    threads = [threading.Thread(target=dense, args=(t,)) for t in range(len(DENSE))]
    threads += [threading.Thread(target=block_scaled), threading.Thread(target=failing)]
    for th in threads:
        th.start()
    for th in threads:
        th.join(timeout=300)
    assert not any(th.is_alive() for th in threads)
    assert not errors, errors
    torch.cuda.synchronize()
    assert tg.tg_device_status() == 0
    for t, (a, b) in enumerate(inputs):
        assert np.array_equal(results[t], oracle_bits(a, b, DENSE[t][3])), DENSE[t]
    assert np.array_equal(results["mx"], mx.gemm_mxfp8_ref(a_mx.numpy(), sa_mx.numpy(),
                                                          b_mx.numpy(), sb_mx.numpy(), "bf16"))
    # each failing call saw its own message, not another thread's (which succeeded meanwhile)
    assert len(messages) == REPEATS and None not in messages.values()
    for i, code, text, last in messages.values():
        assert code == tg.TG_ERR_ARG
        assert f"M={-1 - i} " in last and last in text, (i, last)
