"""GB300-native (sm_103a) MoE expert layer: router top-k, permutation, tcgen05
grouped-GEMM SwiGLU FFN, combine, and the backward pass.

The compute lives in ``libmoe_gb300.so`` (C ABI declared in
``include/moe_gb300.h``); :mod:`._lib` binds its entry points one to one and
:mod:`.layer` sequences them into the layer's forward and backward.  Importing
this package fails if the library has not been built: there is no CPU path.
"""
from ._lib import (  # noqa: F401
    MoEError, moe_combine, moe_gmm, moe_permute, moe_permute_workspace_bytes, moe_route_topk,
    moe_rows_cap, moe_tgmm, moe_unpermute_bwd, SCORE_SOFTMAX, SCORE_SIGMOID, EPI_NONE,
    EPI_SWIGLU_FWD, EPI_SWIGLU_BWD, DTYPE_BF16, DTYPE_F32,
)
from . import layer  # noqa: F401
