"""fp64 CPU oracle (test infrastructure; see ``oracle.attention``)."""
from .attention import (attention_one, attention_dense, attention_varlen, paged_decode,
                        paged_prefill, tile_state, merge_states, gather_paged)
from .attention_grad import (attention_backward_one, attention_backward_dense,
                             attention_backward_varlen)

__all__ = ["attention_one", "attention_dense", "attention_varlen", "paged_decode", "paged_prefill",
           "tile_state", "merge_states", "gather_paged", "attention_backward_one",
           "attention_backward_dense", "attention_backward_varlen"]
