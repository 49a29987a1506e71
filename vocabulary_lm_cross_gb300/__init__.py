"""GB300-native (sm_103a) fused large-vocabulary LM cross-entropy.

The compute lives in ``lib/libvlmce.so`` (hand-written CUDA kernels behind the
C ABI in ``include/vlmce.h``); this package holds the build script, a thin
ctypes/PyTorch binding and the seeded synthetic workloads.
"""
from .ce import (CEResult, ce_fwd_bwd, ce_fwd_bwd_host, describe_plan, host_workspace_bytes,  # noqa: F401
                 max_vocab, workspace_bytes)
from .flce import FLCEResult, flce_fwd_bwd  # noqa: F401
