"""CPU oracle for the dropless MoE expert-MLP path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import
this package.  The product path (``dropless_grouped_gemm_gb300``) never
imports it and has no CPU fallback.

The oracle is plain numpy in float64 (per-expert loops around ``@``), written
from the pages' definitions.  It shares no code with the CUDA library.  Every
function cites the page passage it follows; the pages are cited by title and
section:

* [CuTe] "NVIDIA CuTe DSL 융합 커널은 MoE 학습의 CPU·메모리 병목을 지운다"
* [Sonic] "SonicMoE로 보는 GPU 커널 최적화"
* [TE] "NVIDIA Transformer Engine JAX dropless MoE 105→1,025 TFLOPs"

Parity status: the pages print no numeric fixture for any floating-point
result, so the floating-point functions are pinned by closed forms,
brute force on tiny inputs, finite differences and invariants (see
``tests/test_oracle_*.py``).  The routing functions are also pinned by
the pages' worked examples (``tests/golden/``).
"""
from .moe import *  # noqa: F401,F403
from .mx import *  # noqa: F401,F403
