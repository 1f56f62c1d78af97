"""CPU oracle (test infrastructure only): see ``oracle.lf_oracle``."""
from .lf_oracle import (  # noqa: F401
    attention, attention_backward, attention_lse, attention_row_bruteforce, band_offsets,
    bf16_round, extra_block_keys, key_lists, tiles_per_class, XBLOCK,
    key_set, layer_norm, longformer_layer, mask_rows, pair_count, total_pairs,
    useful_flops,
)
