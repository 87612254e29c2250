"""GB300-native hot path of dropless Mixture-of-Experts training.

The compute lives in libmoe.so (C ABI, include/moe.h; hand-written sm_103a
kernels).  This package is its thin Python face:

* ``grouped_gemm_top_gb300.ops``    -- one Python function per C entry point
  (argument marshalling only);
* ``grouped_gemm_top_gb300.layer``  -- ``MoELayer``: buffers sized once from
  the layer shape, the fwd+bwd step as a fixed sequence of library calls, and
  optional CUDA-graph capture of that sequence;
* ``grouped_gemm_top_gb300.synth``  -- seeded synthetic inputs;
* ``grouped_gemm_top_gb300.build``  -- nvcc build of libmoe.so (sm_103a).

Importing ``ops`` or ``layer`` loads libmoe.so and fails loudly if it has not
been built; there is no CPU or library fallback.
"""
import importlib

__all__ = ["ops", "layer", "synth", "build", "MoELayer"]


def __getattr__(name):
    if name in ("ops", "layer", "synth", "build"):
        return importlib.import_module(f".{name}", __name__)
    if name == "MoELayer":
        return importlib.import_module(".layer", __name__).MoELayer
    raise AttributeError(name)
