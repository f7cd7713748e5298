"""CPU oracle for the block-quantized MoE gather-qmm path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import this package.  The
library in ``block_quantized_moe_gather_gb300`` never imports it and has no
CPU fallback: the CUDA kernels are the only implementation of the path.

The oracle is a plain, slow, fp64 restatement of what the path computes,
written from the pages' formulas.  It shares no code with the CUDA path.
See ``oracle/bq_oracle.py`` for the functions and the passages each follows.
"""
from .bq_oracle import *  # noqa: F401,F403
