"""GB300-native Gaussian Mixture Attention (GMA) forward hot path.

The compute lives in ``libgma`` (hand-written sm_103a CUDA behind a C ABI,
declared in ``include/gma.h``).  The binding in :mod:`.gma` marshals torch
tensors into that ABI; it is loaded on first use so that the seeded workload
generator (:mod:`.workloads`) can be imported on machines without a GPU.
"""
_BINDING_NAMES = (
    "gma_responsibilities", "gma_forward_bidir", "gma_forward_causal", "gma_decode_step",
    "gma_forward_causal_host", "gma_forward_bidir_profiled", "gma_decode_step_profiled",
    "gma_workspace_size", "gma_status_string", "gma_forward_causal_profiled", "Profile", "gma_decode_step_noalloc", "Shape", "GMAError", "library_path", "load",
)


def __getattr__(name):
    if name in _BINDING_NAMES:
        from . import gma
        return getattr(gma, name)
    raise AttributeError(name)
