"""CPU oracle for the persistent warp-specialized GEMM -- test infrastructure only.

This package is the plain, slow, obviously correct statement of what the GPU path
computes.  It is NOT part of the product: only ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py`` (its ``cpu_baseline`` leg and its ``--impl reference`` arm) may
import it.  The CUDA library (``persistent_warp_specialized_gb300``) never imports,
links or calls anything here, and nothing here imports the CUDA library: the two
share no code.  Inputs reach both sides from ``persistent_warp_specialized_gb300.workloads``,
which only draws seeded random numbers.

What it computes, and where the pages define it
-----------------------------------------------
* ``formats``  -- IEEE-754 binary16 and bfloat16: decoding of the 16-bit patterns and
  round-to-nearest-even from binary64.  The GEMM's input/output/accumulator roles
  (``in_dtype``, ``out_dtype``, ``accum_dtype``) are the kernel parameters of
  ``gemm_persistent`` in "[Feature] Introduce tile scheduler #2441"
  (examples/gemm_sm100/gemm_tcgen5mma_ws_persistent.py, ``main`` benchmark call);
  the final cast of the fp32 accumulator to the output type is the epilogue store of
  the generated kernel in "tilelang" (Generated Kernel Source, the ``half_t`` cast).
* ``gemm``     -- C = A.B with exact products and binary64 accumulation, then one
  rounding to the output type (the plain definition of the contraction the kernel in
  "[Feature] Introduce tile scheduler #2441", ``gemm_persistent``, accumulates tile by
  tile in ``C_tmem_0``/``C_tmem_1``).
* ``schedule`` -- the persistent tile schedule: worker ``c`` takes linear tiles
  ``c, c+P, c+2P, ...`` and decodes each with the grouped (swizzled) order of the
  ``tile_id`` decode in ``gemm_persistent`` ("[Feature] Introduce tile scheduler
  #2441", the removed ``for w in T.unroll(waves)`` form, and the
  ``PersistentTileScheduler(..., swizzle_size=group_size)`` that replaces it).

* ``mx``       -- the block-scaled MXFP8 GEMM of the same PR
  (examples/blockscaled_gemm_sm100/gemm_mxfp8_blockscaled_1d1d.py): E4M3 elements, one
  E8M0 scale per 32 K-elements of each A row and each B column, exact scaled products,
  binary64 sum, one rounding to the output type.

Pins (tests that tie the oracle to something other than itself): see
``tests/test_oracle_formats.py``, ``tests/test_oracle_gemm.py``,
``tests/test_oracle_schedule.py`` and ``tests/test_oracle_mx.py``.  Every function here is pinned; none is
"parity unpinned".
"""
