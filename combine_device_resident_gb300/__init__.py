"""Device-resident MoE dispatch/combine data plane for GB300 (sm_103a).

The split counts of the MoE AllToAllv are computed and kept on the GPU, tokens
are packed per destination straight into destination windows, and the expert
outputs are combined as the top-k weighted sum -- the data plane of NCCLX's
AllToAllvDynamic (Section 6.1), with R ranks emulated as R windows in one GPU's
memory.  The work runs in hand-written CUDA kernels behind the C ABI of
``include/a2av.h``; this package is its thin Python binding.
"""
from .binding import (  # noqa: F401
    A2avError,
    Config,
    DEV_BAD_EXPERT,
    DEV_WAIT_TIMEOUT,
    DEV_WINDOW_OVERFLOW,
    EXPORTED,
    FLAG_PACK_LSU,
    FLAG_SPLITS_TILED,
    FLAG_COMBINE_TMA,
    FLAG_ROUTE_FUSED,
    FLAG_ROUTE_WARP,
    ORDER_EXPERT,
    ORDER_SOURCE,
    Plan,
    Splits,
    load_library,
    library_path,
    make_config,
)
