"""Shifted-window multi-head self-attention (cyclic shift, ragged windows,
periodic seam, region and land masks, relative-position bias) for one GB300.

The compute lives in the CUDA library ``libswin_attn.so`` (C ABI in
``include/swin_attn.h``); ``swin_attn`` binds it, ``functional`` wraps it for
torch autograd, ``workloads`` holds the seeded synthetic inputs.
"""
from . import swin_attn  # noqa: F401
from .swin_attn import (Plan, SwinAttnError, make_desc, swin_attn_bwd, swin_attn_fixed_padded_extent,  # noqa: F401
                        swin_attn_fwd, swin_attn_plan, swin_attn_plan_destroy, swin_attn_plan_tables, swin_attn_status,
                        swin_attn_strerror, swin_attn_window_range, swin_attn_workspace_bytes)
