"""Fused row-wise RMSNorm / LayerNorm, forward and backward, for GB300 (sm_103a).

The kernels live in libgbnorm.so behind the C ABI of ``include/gbnorm.h``;
``binding`` marshals torch tensors onto it.  The binding is imported on first
use of one of its names, so that ``rmsnorm_norm_fwd_gb300.inputs`` and
``rmsnorm_norm_fwd_gb300.build`` work before the library exists; any use of
the ops without the built library raises ImportError.
"""

_OPS = ("rmsnorm_fwd", "layernorm_fwd", "rmsnorm_bwd", "layernorm_bwd", "norm_bwd_workspace_size",
        "norm_fwd_ex", "norm_bwd_ex", "norm_bwd_ex_workspace_size",
        "variant_name", "force_variant", "variants", "ex_variants", "ex_force_variant", "ex_last_variant",
        "read_fault", "set_grid_limit", "GbnormError", "lib")

__all__ = list(_OPS)


def __getattr__(name):
    if name in _OPS:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
