"""CPU fp64 oracle for the shape-fused Muon update.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library and
its Python binding) imports, calls or links this package; only the tests,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` use it.  It shares no code with the CUDA path.

Sources (the method is only described in words on these pages; where a page is
silent the reading taken is stated next to the code that takes it):

* «MindSpore HyperParallel X 盘古,Muon优化器实现6倍性能跃升» (jinguxun.com
  article), sections 三大性能挑战 (5-10 Newton-Schulz iterations),
  Muon亲和的专家切分 (Fig. 4: an [E,M,N] expert tensor is E independent
  matrices) and 矩阵融合优化 (Fig. 6-7: parameters with equal trailing two dims
  are stacked into one [B,M,N] batch).
* «关于分布式Muon的想法整合及讨论» (gtnt.cn blog), §1 (momentum of the gradient,
  then approximate orthogonalisation of M), §2 (normalise M, Gram matrix, a
  series of matmuls) and §6 (the normaliser is a sum of squares; the Gram
  matrix is recomputed every iteration).
* HyperParallel-FSDP abstract (arXiv 2609.21594), contribution (3):
  shape-fused Newton-Schulz iterations.

Pins (checked in ``tests/test_oracle_pins.py`` against things other than the
oracle itself): the singular-value closed form of the polynomial iteration,
brute-force SVD on tiny matrices, an exact 1-row case, transpose symmetry,
batch independence, a pure-Python loop implementation, and the bucketing
examples the pages print.  Parity unpinned: the values of eps and of the
shape-dependent scale s are readings (the pages give neither); they are pinned
only to the stated reading.
"""
from .muon_ref import (  # noqa: F401
    NS_COEFFS_QUINTIC,
    SCALE_MODES,
    bucket_shapes,
    frobenius_normalize,
    momentum,
    muon_step_ref,
    muon_update_ref,
    nesterov_input,
    newton_schulz,
    newton_schulz_sharded,
    ns_polynomial,
    orthogonalize,
    scale_factor,
    sharded_frobenius_normalize,
    step_coefficients,
)
