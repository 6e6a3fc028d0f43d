"""Tensor-parallel sharded GEMMs on GB300 (sm_103a).

The compute lives in the CUDA library ``libtps.so`` built from ``csrc/``;
this package only marshals torch tensors into its C ABI (``include/tps.h``).
Importing the package does not load the library; the first call does, and
fails loudly if it is missing.
"""
__all__ = ["plan_shards", "matmul_fwd_bwd", "mlp_fwd_bwd", "vocab_ce_fwd_bwd", "inputs"]


def __getattr__(name):
    if name in ("plan_shards", "matmul_fwd_bwd", "mlp_fwd_bwd", "vocab_ce_fwd_bwd",
                "mlp_workspace_bytes", "ce_workspace_bytes", "last_device_error", "library",
                "profile", "TpsError"):
        from . import api
        return getattr(api, name)
    raise AttributeError(name)
