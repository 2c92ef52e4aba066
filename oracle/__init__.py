"""CPU oracle for causal GQA attention. TEST INFRASTRUCTURE, not product code.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its
``cpu_baseline`` leg and its ``--impl reference`` arm) may import, call or run
anything in this package.  The product path (the C-ABI library and its Python
binding) never imports it and has no CPU fallback.

The oracle shares no code with the CUDA path.  Both are fed the same seeded
inputs from ``attn_workloads``, a module that holds no attention arithmetic.

Modules:
  * ``attn``  -- the plain definition in float64 numpy: explicit RoPE, explicit
    GQA head repetition, explicit T x T scores, additive -inf mask, row softmax,
    weighted sum of V; plus the decode form and the split log-sum-exp merge.
  * ``naive`` -- an independently written scalar-loop version (Python floats and
    ``math`` only), used to brute-force-check ``attn`` on tiny inputs.

Every function here is pinned by ``tests/test_oracle_pins.py``; none is
"parity unpinned".
"""
from . import attn, naive  # noqa: F401
