"""fp64 CPU oracles (test infrastructure only): the sliced tensor-parallel MLP
block (``oracle.oracle``, re-exported here) and the sliced tensor-parallel
attention block (``oracle.attention``)."""
from .oracle import *  # noqa: F401,F403
from .oracle import max_rel_err, mlp_bwd, mlp_bwd_sharded, mlp_fwd, mlp_fwd_intermediates, mlp_fwd_sharded  # noqa: F401
