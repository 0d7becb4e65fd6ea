"""GB300-native decode-time MoE layer with FloE-style contextually sparse SwiGLU experts.

The compute runs in a CUDA library built for sm_103a (``build.py``) behind a C ABI
(``include/sparse_expert_swiglu.h``); this package is its thin Python binding plus
the seeded synthetic-input generator.
"""

from ._lib import (  # noqa: F401
    EAMC,
    EXPORTED,
    ExpertCache,
    Experts,
    Layer,
    MoeError,
    Workspace,
    eam_add_counts,
    expert_sparse_swiglu,
    expert_workspace_bytes,
    layer_decode,
    layer_decode_host_rows,
    layer_host_rows_workspace_bytes,
    layer_path,
    layer_workspace_bytes,
    lib,
    lib_path,
    pack_int2_up,
    packed_bytes,
    prefetch_experts,
    route_topk,
    route_topk_noalloc,
    route_workspace_bytes,
    unpack_int2_up,
)
from . import build as _build_module  # noqa: E402

build_library = _build_module.build
