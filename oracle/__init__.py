"""CPU fp64 oracle of the FLARE++ mixer forward (test infrastructure only).

Imported by tests, the package smoke check and the benchmark's CPU-baseline
leg; never by the library path.
"""
from .flarepp_oracle import (EPS, decode, encode, encode_partial, flare_forward,
                             flare_forward_head, forward, forward_head, forward_simplified,
                             forward_unshared, logsumexp_rows, lse_merge, n0, routing_queries,
                             sdpa, softmax_rows, synthesis, synthesis_simplified,
                             synthesis_unshared, w_eff, NORM_NONE, NORM_N0, NORM_NA,
                             project, sdpa_backward, n0_backward, backward_head, backward)

__all__ = ["EPS", "decode", "encode", "encode_partial", "flare_forward", "flare_forward_head",
           "forward", "forward_head", "forward_simplified", "forward_unshared", "logsumexp_rows",
           "lse_merge", "n0", "routing_queries", "sdpa", "softmax_rows", "synthesis",
           "synthesis_simplified", "synthesis_unshared", "w_eff", "NORM_NONE", "NORM_N0",
           "NORM_NA", "project", "sdpa_backward", "n0_backward", "backward_head", "backward"]
