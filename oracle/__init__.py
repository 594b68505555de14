"""Oracle package -- test infrastructure only (see dsa_oracle's header)."""
from .dsa_oracle import (positions, indexer_scores, topk_select, sparse_attn_fwd,  # noqa: F401
                         sparse_attn_bwd, indexer_kl_loss, dsa_forward)
