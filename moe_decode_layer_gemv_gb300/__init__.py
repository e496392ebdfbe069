"""GB300-native Mixture-of-Experts decode layer (sm_103a).

The layer -- router GEMV, fp32 softmax + top-k, stable grouping of the routes
by expert, grouped gate_up/SiLU*up and down projections and the weighted
combine -- runs in hand-written CUDA kernels behind the C ABI of
``include/moe.h`` (``libmoe.so``, built in-tree by ``build.build()``).

Submodules:
  api         ctypes binding of libmoe.so (importing it fails loudly when the
              library is missing; there is no CPU fallback)
  synth       seeded synthetic inputs (shared with the tests' oracle)
  accounting  byte / reuse formulas used by the benchmark
  build       nvcc build of libmoe.so
"""
__all__ = ["api", "synth", "accounting", "build"]
