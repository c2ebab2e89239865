"""CPU float64 oracle (test infrastructure; never part of the product path)."""
from .relpos_oracle import (attention, attention_backward, attention_rows, dense_bias, fused, fused_backward,
                            fused_rows, lse2, project, project_rows, rel_index)

__all__ = ["attention", "attention_backward", "attention_rows", "dense_bias", "fused", "fused_backward",
           "fused_rows", "lse2", "project", "project_rows", "rel_index"]
