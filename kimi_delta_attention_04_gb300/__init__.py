"""GB300-native Kimi Delta Attention: chunkwise forward, fused T=1 decode and the
short-T recurrent step on a state pool.

The computation lives in libkda.so (hand-written sm_103a CUDA behind the C ABI
of include/kda.h); this package is its thin Python binding. Importing the
package does not load the library; the first call does, and raises if the
library has not been built (python -m kimi_delta_attention_04_gb300.build).
"""

from ._lib import (  # noqa: F401
    KdaError,
    chunk_count,
    chunk_workspace_size,
    kda_chunk_fwd,
    kda_chunk_output,
    kda_chunk_fwd_noalloc,
    kda_decode_conv_step,
    kda_decode_step,
    kda_head_rmsnorm,
    kda_recurrent_step,
    lib_path,
    load,
    make_chunk_args,
    make_decode_args,
    make_recurrent_args,
    version,
)

__version__ = "0.1.0"
