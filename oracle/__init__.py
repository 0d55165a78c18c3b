"""CPU oracle for the Flint-style W4A16 (NVFP4) MoE decode layer.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports, calls or
executes this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may. It shares no
code with the CUDA library (no kernels, headers, helpers, tables or constant
generators) and does not import it; its inputs come from ``synth`` (random
draws only) or from the tests themselves.

Everything here is the plain definition, written out in float64 with numpy;
a matrix-vector product and a sort are the only library steps. Sources are
the pages on the method:

* "Day-0 Support for Flint on vLLM" (vLLM blog; Chinese, Japanese, French
  and Korean versions), section "Model architecture": 256 experts, sigmoid
  top-6 plus one always-on shared expert; the NVFP4 checkpoint runs weight-only
  (W4A16) with BF16 activations, following the reference implementation's
  rounding points.
* Same post, section "Optimisation": the small-batch MoE kernels make the
  router and expert GEMVs read only the selected experts' weights; the SiLU
  kernel follows the reference rounding; routing and the expert combine are
  fused into the adjacent GEMVs.

Where the pages are silent, each function states the plain reading it takes
(the NVFP4 bit layout from its public definition, renormalised routing
weights, FP32 accumulation with BF16 rounding after SiLU*up and at the
output, an unweighted shared expert of the routed intermediate size).

Pins (tests in ``tests/test_oracle_pins.py``) tie every function to
something other than itself: the E2M1 and E4M3 code tables, torch's own
float8_e4m3fn and bfloat16 conversions, brute-force nearest-value search,
quantise/dequantise round-trip bounds and idempotence, brute-force top-k
over all expert subsets, a dense all-experts formulation of the layer, and
the textbook dense SwiGLU special case.
"""
from . import nvfp4, moe  # noqa: F401
