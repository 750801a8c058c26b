"""Float64 CPU oracle for the DSA forward path (test infrastructure only).

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg import
this package.  The CUDA library never does, and this package never imports
the library.
"""
from .dsa_oracle import (HiSparseLRU, attention_on_set, band_check, bf16_to_f64, cache_append, dsa_forward,
                         f32_to_f64, indexer_scores, mha_attention_on_set, mha_upproject, requested_rows, scores_for_query,
                         sparse_mha, sparse_mla, topk_select, visible_entries)

__all__ = ["HiSparseLRU", "attention_on_set", "band_check", "bf16_to_f64", "cache_append", "dsa_forward",
           "f32_to_f64", "indexer_scores", "mha_attention_on_set", "mha_upproject", "requested_rows",
           "scores_for_query", "sparse_mha", "sparse_mla", "topk_select", "visible_entries"]
