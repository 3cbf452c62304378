"""In-Place TTT fast-weight layer for GB300 (sm_103a).

The layer computes Z = SiLU(H W_gate^T) * (H W_up^T) and the next-token
aligned target Vhat = CausalConv1D(X0) W_target^T, then walks the sequence in
chunks of C tokens: each chunk is applied with the fast weight accumulated
from earlier chunks (O_i = Z_i W_i^T) and then updates it
(W_{i+1} = W_i + eta Vhat_i^T Z_i).  All of it runs in hand-written CUDA
kernels behind the C-ABI library ``libittt.so``; :mod:`.ittt` is the thin
ctypes binding.  Importing this package does not load the library.
"""
from .inputs import CONFIGS, config_inputs, counted_flops, make_inputs  # noqa: F401
