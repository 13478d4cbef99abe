"""fp64 CPU oracle of the MoE FFN layer.  TEST INFRASTRUCTURE: used only by tests/,
``__graft_entry__.smoke()`` and bench.py's CPU-baseline leg; never by the product path."""
from .moe_oracle import *  # noqa: F401,F403
from .moe_oracle import Layer, Routing, Dispatch  # noqa: F401
