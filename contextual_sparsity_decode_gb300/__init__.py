"""GB300-native contextually sparse decode (Deja Vu) — Python side.

``binding`` is the thin ctypes layer over libdv (include/dv.h); ``stack``
orders library calls into a decoder step; ``build`` compiles libdv.so.
"""

from . import binding  # noqa: F401
from .binding import (  # noqa: F401
    DV_BF16, DV_F16, DV_F32, DV_THRESHOLD, DV_TOPK, DvError, KV, Predictor,
    dv_check, dv_kv_repair, dv_layernorm, dv_lookahead, dv_positions_advance, dv_predict,
    dv_predict_workspace_size, dv_sparse_attn, dv_sparse_attn_workspace_size, dv_sparse_mlp,
    dv_sparse_mlp_workspace_size, dv_status_str, dv_version, dv_workspace_init, workspace,
)
