"""CPU oracle of the MTP draft-layer forward.

Test infrastructure, not product code: only ``tests/``, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import it.
The CUDA path never calls it and shares no code with it.
"""

from .mtp_oracle import (  # noqa: F401
    argmax_lowest, attention, dequant, draft_chain, draft_layer, moe_ffn, moe_route,
    qmatmul, rmsnorm, rope, sigmoid, silu, swiglu, topk_lowest_index, unpack_codes,
)
