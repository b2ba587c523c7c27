"""Float64 CPU oracle (test infrastructure only; never on the product path)."""
from .verify_attention import (candidate_visibility, cohort_chunk_plan, covers_exactly_once, round_bf16,
                               verify_attention, verify_attention_streamed, visibility_table)

__all__ = ["candidate_visibility", "cohort_chunk_plan", "covers_exactly_once", "round_bf16", "verify_attention",
           "verify_attention_streamed", "visibility_table"]
