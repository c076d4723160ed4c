"""fp64 CPU oracle of the LRM-pruned MoE expert backward (test infrastructure only).

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline / reference arm use it.
"""
from .lrm_oracle import (compact, expert_backward, expert_loads, grad_abs_scores, grad_sq_scores,  # noqa: F401
                         lrm_scores, lrm_scores_from_norms, masked_backward, plan_quotas, pruned_backward,
                         pruned_backward_recompute, recompute_saved_state,
                         route, router_grad, scatter_dx, select, swiglu_backward, swiglu_forward,
                         unpruned_backward)
