"""CPU oracle for the NVFP4 MoE router gate -- TEST INFRASTRUCTURE ONLY.

This package is a plain, slow, obviously-correct NumPy restatement of what the
router hot path computes.  It exists so that the CUDA path can be checked
against something written independently of it.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference arm may
import it.  The product package (``nvfp4_router_gate_gb300``) never imports it
and never falls back to it.

It shares no code with the CUDA path: no kernels, headers, helpers, tables or
constant generators.  The only module both sides use is ``workloads`` (seeded
synthetic inputs), which holds none of the method's arithmetic.

Sources (the web pages this project is built from, cited by page title and
section):

* "nvfp4-megamoe-kernel commit 04cf8ca: dsv4/layers/router.py" -- runtime
  global activation scale section (gsa = max|x| / (6 * 448), so that
  x / gsa <= 2688), and the NVFP4 gate / activation_topk two-kernel section.
* "nvfp4-megamoe-kernel commit e0f60b9: dsv4/kernels/router/__init__.py" --
  the activation_topk section (single-pass fused six-step epilogue) and the
  fused decode kernel notes (row-level top-k across N-subtiles).
* "nvfp4-megamoe-kernel commit df05289: dsv4/layers/grouped_linear.py" --
  zero-sync fused quantize section (one flattened (G*T, D) tensor, GPU-only
  gsa), and the repeated runtime-gsa section.

Where the pages leave a step open the module docstrings state the reading
taken.  Modules:

* ``formats``  -- E2M1 / E4M3 decode tables and round-to-nearest-even encoders.
* ``quantize`` -- runtime gsa, 16-element E4M3 block scales, E2M1 codes,
  nibble packing and the 128x4 scale-factor tile layout.
* ``gemm``     -- logits of the dequantized operands in float64.
* ``router``   -- sigmoid, bias-corrected top-k, renormalised routed weights.
* ``compare``  -- the tolerance rules used by the parity tests.

Parity status: every function here is pinned by a ``-m "not gpu"`` test in
``tests/test_oracle_*.py`` except the GPU tensor-core accumulation order,
which is "parity unpinned" beyond the floating-point error bound used in
``compare`` (the hardware's internal accumulation precision is not
documented).
"""

from . import formats, quantize, gemm, router, compare, pipeline, hash_router, moe  # noqa: F401
