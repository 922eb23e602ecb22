"""CPU oracle for the local MoE forward chain. Test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA library never calls it and it
never calls the CUDA library.
"""
from .moe_oracle import (  # noqa: F401
    DispatchResult,
    GroupRoutingOptions,
    RouteResult,
    check_group_options,
    combine,
    dispatch,
    experts_forward_dispatched,
    forward,
    forward_tokens,
    forward_tokens_routed,
    forward_with_routing,
    route,
    route_sigmoid_grouped,
    round_to_dtype,
    silu,
    widen,
)
from .training import (  # noqa: F401
    ExpertGrads,
    RouterWeightOptions,
    check_router_options,
    combine_backward,
    dispatch_backward,
    experts_backward,
    router_jacobian,
    selected_router_backward,
    selected_router_weights,
    training_forward_cache,
)
