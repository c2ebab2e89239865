"""CPU float64 oracle (test infrastructure; never part of the product path)."""
from .relpos_oracle import (attention, attention_rows, dense_bias, fused, fused_rows, project, project_rows,
                            rel_index)

__all__ = ["attention", "attention_rows", "dense_bias", "fused", "fused_rows", "project", "project_rows",
           "rel_index"]
