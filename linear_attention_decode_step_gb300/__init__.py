"""GB300-native Kimi Delta Attention (KDA): fused decode step and chunked
prefill as hand-written sm_103a CUDA kernels behind a C ABI (include/kda.h).

Submodules:
  build   compiles csrc/*.cu into libkda_gb300.so (in-tree)
  kda     ctypes binding of the C ABI (argument marshalling only)
  inputs  seeded synthetic inputs shaped like the GLM-5.3-Flash workload

Importing the package loads nothing; ``kda`` loads the compiled library on
first use and raises if it has not been built.
"""

__all__ = ["build", "kda", "inputs"]
