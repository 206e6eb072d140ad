"""POET-X transformed linear on B300 (sm_103a): a C-ABI CUDA library and its binding.

The layer's effective weight is the orthogonal equivalence transform
W = R . W0 . P of a frozen W0, applied input-centric as y = R (W0 (P x)); R and
P are permuted block-diagonal orthogonal matrices whose blocks come from packed
skew parameters by the Cayley-Neumann parameterisation ("POET-X:
Memory-efficient LLM Training by Scaling Orthogonal Transformation",
gist.science summary, section 2).  Importing this package loads nothing; the
CUDA library is loaded on first use and its absence is an error.
"""
from ._lib import (PoetxError, poetx_backward, poetx_cayley_neumann,  # noqa: F401
                   poetx_cayley_neumann_backward, poetx_check_perm, poetx_forward,
                   poetx_invert_perm, poetx_merge_w0, poetx_status_string, poetx_stream_status,
                   poetx_version, poetx_workspace_bytes)
from .layer import TransformedLinear  # noqa: F401
