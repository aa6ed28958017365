"""CPU oracle for the KVarN codec and its decode attention.

TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the CPU-baseline
leg of the benchmark may import anything under this package; the library's
product path never does. It shares no code with the CUDA path: it has its own
statement of the page layout and its own arithmetic, all in float64 numpy.

Modules:
  codec      rotation, variance normalisation, asymmetric RTN, dequantisation
  layout     byte layout of a cache page (the library's documented format)
  attention  decode attention over a paged cache, fp16 tail, fp16 bypass
  mla        the MLA latent-cache codec and decode
  affine     the per-token affine comparison codec (groups of 64 channels,
             fp16 scale and offset), its page layout and decode
"""
from . import codec, layout, attention, mla, affine  # noqa: F401
