"""GB300-native finite-automaton constrained sampling for diffusion language models.

The product is the C-ABI library libfa.so (include/fa.h) built from csrc/ for
sm_103a; `native` is its thin Python binding and `synth` the seeded workload
generators.  Importing the package does not load the library; the first call
through `native` does, and raises if it has not been built.
"""
__all__ = ["native", "synth", "build"]
