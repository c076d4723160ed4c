"""LRM-pruned MoE expert backward on one GB300 (sm_103a): C ABI (include/lrm.h) + Python binding.

Importing the package does not load the library; the first call does, and raises if
liblrm.so has not been built (python -m pruned_expert_backward_gb300.build).
"""
from .api import (HostPipeline, LrmError, PrunedBackward, lrm_compact, lrm_grouped_backward,
                  lrm_grouped_backward_gather, lrm_plan_quotas,  # noqa: F401,E501
                  lrm_recompute_forward, lrm_route, lrm_router_grad, lrm_scatter_dx, lrm_score, lrm_score_mode, lrm_score_norms,
                  lrm_select, lrm_swiglu_forward, lrm_workspace_size)
