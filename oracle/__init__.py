"""CPU fp64 oracle (test infrastructure only; see flce_oracle)."""
from .flce_oracle import (capped_logits, flce_oracle, oracle_ce_logits, oracle_grad_W_rows,  # noqa: F401
                          oracle_merge_shards, oracle_rows, oracle_shard_grad_h, oracle_shard_partials)
