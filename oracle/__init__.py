"""fp64 CPU oracle (test infrastructure; see uniprefill_oracle.py's header)."""
from .uniprefill_oracle import *  # noqa: F401,F403
from .uniprefill_oracle import (block_scores, block_scores_from_tokens, carry_forward, compact,  # noqa: F401
                                cu_blocks_of, drop_step, pack_key, phi, rank_order, select,
                                select_request, seqused, slot_mapping, token_scores, topp_kstar)
