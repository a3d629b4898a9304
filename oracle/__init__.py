"""fp64 CPU oracle (test infrastructure; see ``oracle.attention``)."""
from .attention import (attention_one, attention_dense, attention_varlen, paged_decode,
                        paged_prefill, tile_state, merge_states, gather_paged)

__all__ = ["attention_one", "attention_dense", "attention_varlen", "paged_decode", "paged_prefill",
           "tile_state", "merge_states", "gather_paged"]
