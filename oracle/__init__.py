"""CPU oracle for the dropless MoE layer (forward and backward).

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or run
anything in this package: only the tests, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline leg use it.  It shares no code with the CUDA path.

Every function is plain NumPy in the float type the caller picks (fp64 by
default), written to be checked by eye against the definitions it cites.
"""
from .moe_oracle import (  # noqa: F401
    select_topk,
    route,
    dispatch,
    permute_rows,
    combine_rows,
    swiglu_expert_forward,
    moe_forward,
    moe_backward,
    route_backward,
    expert_wgrad,
    expert_wgrad_sampled,
    expert_rows,
)
from . import mx  # noqa: F401,E402
