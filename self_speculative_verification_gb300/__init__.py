"""libspecverify: the verification step of self-speculative decoding on GB300.

The compute path is the C-ABI shared library ``libspecverify.so`` (CUDA
kernels for sm_103a).  This package holds its Python binding (argument
marshalling only), the build step and the seeded workload generator.
The library is loaded lazily on first use; if it is missing, every call
raises instead of falling back to anything else.
"""

__version__ = "0.1.0"

_API = ("spec_mask_build", "spec_verify_attn", "spec_verify_attn_workspace_size",
        "spec_vocab_reduce", "spec_accept", "kv_commit", "spec_get_status",
        "spec_version")


def __getattr__(name):
    if name in _API or name in ("SpecError", "library_path", "load_library"):
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
