"""CPU oracle for Multi-Segment Attention -- test infrastructure only.

Only the tests, the package smoke check and the benchmark's CPU-baseline leg may
import this package.  It shares no code with the CUDA path.
"""
from .msa_oracle import (attention, canonical_plan, canonical_tokens, chunk_sizes, decode,  # noqa: F401
                         gather_by_position, merge_lse, prefill, seq_units, useful_flops)
from .evict_oracle import (EvictOracle, lambda_update, marginal_cost, modelled_recompute_cost,  # noqa: F401
                           recompute_cost, reuse_estimate, turning_point)
