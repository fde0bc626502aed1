"""GB300-native FASA decode step (frequency-aware sparse attention).

The compute lives in ``libfasa.so`` (hand-written CUDA for sm_103a, C ABI in
``include/fasa.h``).  This package is its thin Python binding: argument
marshalling from torch tensors (device pointers and the current stream) to the
C entry points of the same names.  There is no CPU fallback: if the library
is not built, every call raises.
"""

from .fasa import (  # noqa: F401
    FASA_BF16, FASA_F32, FASA_DEV_BAD_INPUT, FASA_DEV_TIMEOUT, FASA_DEV_UNDRAINED, FASA_KERNEL_CLUSTER,
    FASA_KERNEL_SINGLE_EXCHANGE, FasaDims, FasaError, dims_for, fasa_append_kdom, fasa_apply_rope_q,
    fasa_build_kdom, fasa_cluster_size, fasa_decode_step, fasa_decode_step_append, fasa_decode_step_noalloc,
    fasa_dense_attention,
    fasa_device_status, fasa_fc_agreement, fasa_fc_agreement_workspace_size,
    fasa_select_dominant_fcs, fasa_compound_agreement, fasa_test_fault_injection, fasa_step_kernel,
    fasa_build_knondom, fasa_decode_step_split, fasa_decode_step_append_split,
    fasa_focused_attention, fasa_max_budget, fasa_tip_score, fasa_topk_select, fasa_workspace_size,
    lib, library_path,
)
