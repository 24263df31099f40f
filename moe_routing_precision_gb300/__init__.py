"""GB300-native MoE routing + FP8 quantisation hot path.

Five operations, each a hand-written CUDA kernel for sm_103a behind the C ABI
declared in ``include/moe_route.h``:

* ``topk_gate``        top-k experts per token (ties to the lower index) and
                       the softmax weights of the k selected scores;
* ``route_map``        per-expert counts, exclusive offsets, the stable
                       expert-sorted slot of every routed copy and its inverse;
* ``expand_cast_fp8``  gather every routed copy into its expert's slot as FP8
                       E4M3 with one fp32 scale per 128 channels;
* ``swiglu_cast_fp8``  silu(gate) * up in fp32, then the same FP8 cast;
* ``combine``          the weighted sum of each token's expert outputs.

``ops`` is the thin Python binding (argument marshalling only); it loads the
in-tree shared library and raises if it is missing.  ``workloads`` draws the
seeded synthetic inputs.
"""
from . import workloads  # noqa: F401  (no CUDA needed)

__all__ = ["ops", "workloads", "build"]


def __getattr__(name):
    import importlib
    if name == "ops":
        return importlib.import_module(__name__ + ".ops")
    if name == "build":
        return importlib.import_module(__name__ + "._build").build
    raise AttributeError(name)
