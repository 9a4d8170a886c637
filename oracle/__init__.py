"""Float64 CPU oracle of the greedy block-verify step.

TEST INFRASTRUCTURE.  This package is the slow, plain definition that the
CUDA library is checked against.  Only the tests, the smoke check and the
CPU-baseline leg of the bench may import or run it; the CUDA library neither
imports it nor shares any code, table or helper with it, and it imports
nothing from the library.  Inputs come from the seeded generators in
`workload/`, which hold no arithmetic of the method.

Modules:
  formats  -- BF16 / E4M3 / E2M1 bit-field decoders and nearest-even encoders
  quant    -- round-to-nearest FP8 per-channel and NVFP4 quantisers, exact dequant
  model    -- float64 decoder forward, prefill, autoregressive greedy decode,
              greedy block verification with prefix accept and KV commit
  weights  -- canonical (quantised) weight entries from BF16 master weights
  loop     -- slot scheduling of the device-resident draft / verify loop
  sampling -- stochastic (temperature) block verification, random numbers as inputs
"""
from . import formats, quant, model, weights, loop, sampling  # noqa: F401
