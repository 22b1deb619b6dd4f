"""fp64 CPU oracle for the sliced tensor-parallel MLP (test infrastructure only)."""
from .oracle import *  # noqa: F401,F403
from .oracle import max_rel_err, mlp_bwd, mlp_bwd_sharded, mlp_fwd, mlp_fwd_intermediates, mlp_fwd_sharded  # noqa: F401
