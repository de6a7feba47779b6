"""MoE token dispatch / combine for one GB300 (sm_103a).

The compute path is the CUDA library ``libep.so`` (C ABI: include/ep.h); this
package is its Python binding.  Build the library with
``python -m combine_expert_histogram_gb300.build``.
"""
from .binding import (  # noqa: F401
    EPError,
    Layout,
    ep_combine,
    ep_dispatch,
    ep_layout,
    ep_layout_workspace_bytes,
    ep_masked_repack,
    ep_rows_capacity,
    ep_scale_cols,
    load_library,
    new_layout,
    status_str,
)
