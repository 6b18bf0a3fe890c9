"""fp64 CPU oracle for the CODA GEMM-epilogue hot path.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check in
``__graft_entry__`` and the ``cpu_baseline`` / reference leg of ``bench.py``
may import this package.  The product (the CUDA library and its binding)
never calls it, and it shares no code with the CUDA path.

Source of truth: "CODA: Rewriting Transformer Blocks as GEMM-Epilogue
Programs" as reported in the Synced article (page "还在手写CUDA内核?CODA来了!",
sections 尾声 and 五种积木; same text on the KuCoin page, sections 尾聲 and
五種積木).  Every function here is the plain, unfused, obviously-correct
definition of one quantity, written in float64 with numpy.  numpy's matmul is
used as the only library primitive.

All functions take numpy float64 arrays (exact widenings of the bf16 inputs)
and never round to bf16: the oracle computes the exact-arithmetic result (up
to fp64 rounding order).

Parity status: every function is pinned by the CPU tests in
``tests/test_oracle_pins.py`` (closed forms, brute force, finite differences,
hand-worked fixtures under ``tests/golden``).  The pages print no numeric
example, so nothing is pinned against the authors' own outputs.
"""
from .coda_oracle import *  # noqa: F401,F403
from .coda_oracle import __all__  # noqa: F401
