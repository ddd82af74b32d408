"""GB300-native dual-mode (causal / bidirectional) attention forward pass for
DiffusionGemma-style block-autoregressive diffusion decoding.

The compute runs in ``lib/libdg_attn.so`` (hand-written sm_103a kernels behind
the C ABI of ``include/dg_attn.h``); ``binding`` is a thin ctypes layer over it.
"""

from .binding import (DG_MODE_BIDIRECTIONAL, DG_MODE_CAUSAL, DgAttnError,  # noqa: F401
                      accept_step, error_string, forward, load_library, status, version,
                      workspace_size)
