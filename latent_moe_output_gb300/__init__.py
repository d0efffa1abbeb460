"""GB300 (sm_103a) latent-MoE output tail.

    out[t, h] = sum_l rms_norm(sum_p routed[p, t, :], g, eps)[l] * W[h, l]
                + sum_p shared[p, t, h]

The computation runs in the CUDA library built from ``csrc/`` and exposed
through the C ABI in ``include/latent_tail.h``; ``binding`` is the thin ctypes
layer over it. Importing this package does not load the library; the first
call does, and fails loudly if it was not built.
"""

from .binding import (  # noqa: F401
    LatentTailError,
    Status,
    forward,
    forward_host,
    latent_tail_check,
    latent_tail_forward,
    latent_tail_forward_cols,
    latent_tail_forward_host,
    latent_tail_norm,
    latent_tail_project_cols,
    latent_tail_status_string,
    latent_tail_host_workspace_size,
    latent_tail_workspace_size,
    library_path,
    load_library,
)
