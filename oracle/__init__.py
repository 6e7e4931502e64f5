"""CPU oracle for kernelized linear attention (fp64, numpy).

TEST INFRASTRUCTURE ONLY: imported by tests/, by the package smoke check and
by the benchmark's CPU-baseline leg, never by the library.  See
oracle/linear_attention.py for what each function computes and which passage
of the source pages it follows.
"""
from .linear_attention import (  # noqa: F401
    MAPS, NORMS, dpfp_nu, feature_map, feature_dim, sum_normalise, features, gram_schmidt,
    orthogonal_random_features, normalise, bidir, causal, decode_step, rescan, causal_rows, bidir_rows,
    forward, softmax_kernel_estimate, feature_map_vjp, features_vjp, backward,
)
