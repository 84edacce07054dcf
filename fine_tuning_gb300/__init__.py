"""GB300-native fused per-token layer ops for LLM fine-tuning.

RMSNorm, SwiGLU and in-place varlen QK-RoPE, forward and backward, as
hand-written sm_103a CUDA kernels behind the C ABI in include/ftk.h.

    from fine_tuning_gb300 import ftk
    y, rstd = ftk.rmsnorm_fwd(x, w, eps)

``ftk`` loads libftk.so on first use and raises ImportError if it has not
been built (``fine_tuning_gb300.build.build()``); there is no fallback.
"""
__version__ = "0.1.0"

_BINDING = ("rmsnorm_fwd", "rmsnorm_bwd", "rmsnorm_bwd_workspace_bytes", "swiglu_fwd",
            "swiglu_bwd", "qk_rope_fwd", "qk_rope_bwd", "FtkError", "library")


def __getattr__(name):
    if name in _BINDING:
        from . import ftk
        return getattr(ftk, name)
    raise AttributeError(name)
