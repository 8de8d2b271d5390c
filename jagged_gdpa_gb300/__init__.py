"""jagged_gdpa_gb300: jagged Generalized Dot-Product Attention on GB300 (sm_103a).

The computation lives in libjgdpa.so (C ABI in include/jgdpa.h, CUDA kernels
under csrc/).  This package only builds and binds it.
"""

from ._lib import (  # noqa: F401
    ACT,
    ALU_LIB_PATH,
    LIB_PATH,
    EXPORTS,
    JgdpaError,
    jgdpa_bwd,
    jgdpa_bwd_shared_q,
    jgdpa_fwd_shared_q,
    jgdpa_shared_q_workspace_bytes,
    jgdpa_ds_scratch_bytes,
    jgdpa_eval_activation,
    jgdpa_fwd,
    jgdpa_fwd_noalloc,
    jgdpa_read_device_status,
    jgdpa_set_wait_limit_ns,
    jgdpa_status_string,
    jgdpa_workspace_bytes,
    load,
)
