"""GB300 (sm_103a) MTP draft-layer forward: Python binding of libmtpdraft.

Every entry point here marshals torch tensors into the C ABI declared in
``include/mtpdraft.h``; all arithmetic runs in the library's CUDA kernels.
"""

from .api import (  # noqa: F401
    affine4, attn_decode_sink, attn_decode_sink_noalloc, attn_geom, lmhead_argmax, moe_ffn, moe_weights, mtp_draft_chain,
    mtp_draft_forward, mtp_kv_catch_up, mtp_rope_table, mtp_workspace_init, mtp_workspace_set_wait_limit, mtp_workspace_status,
    mtp_spec_accept, mtp_spec_note_round, mtp_spec_rewind, mtp_spec_tokens_per_round,
    mtp_draft_steps, mtp_mimo_commit_layer, mtp_mimo_draft_round, mtp_mimo_plan_layer,
    qmatmul_affine4, rmsnorm_residual, verify_head_argmax, workspace,
)
from ._lib import MimoLayerState, SpecStats  # noqa: F401
from .layer import DraftLayer, DraftChain  # noqa: F401
