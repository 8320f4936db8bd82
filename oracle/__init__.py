"""CPU fp64 oracle for the L³ layer: test infrastructure, not part of the library.

Importable only by tests/, __graft_entry__.smoke() and bench.py's CPU legs.
"""
from .l3_oracle import (Allocation, Backward, Forward, Route, SparseBackward, allocate, allocate_from_counts,
                        attend, attend_dense_masked, backward, backward_rows,
                        backward_token, count_ids, forward,
                        forward_token, layer_norm, route, token_rows)

__all__ = ["Allocation", "Backward", "Forward", "Route", "SparseBackward", "allocate", "allocate_from_counts",
           "attend", "attend_dense_masked", "backward", "backward_rows", "backward_token", "count_ids", "forward",
           "forward_token", "layer_norm", "route", "token_rows"]
