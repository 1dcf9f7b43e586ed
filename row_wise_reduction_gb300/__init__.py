"""rowops: row-wise reduce-then-normalise CUDA kernels for GB300 (sm_103a).

Stable and causal softmax, split-row online softmax, fused LayerNorm -> affine ->
GELU (tanh or exact) and its backward, fused residual + bias + GELU, RMSNorm and fused residual + RMSNorm, row sums and row
maxima, exposed through the C ABI of
``librowops.so`` (``include/rowops.h``) and the thin ctypes binding in
:mod:`row_wise_reduction_gb300.rowops`.
"""
from .rowops import (  # noqa: F401
    ROWOPS_BF16,
    ROWOPS_F32,
    RowopsError,
    library,
    library_path,
    rowops_bias_residual_gelu,
    rowops_device_status,
    rowops_fused_residual_rmsnorm,
    rowops_gelu,
    rowops_layernorm_gelu,
    rowops_layernorm_gelu_backward,
    rowops_layernorm_gelu_backward_workspace_bytes,
    rowops_layernorm_gelu_erf,
    rowops_online_softmax,
    rowops_online_softmax_noalloc,
    rowops_online_softmax_status,
    rowops_online_softmax_workspace_bytes,
    rowops_rmsnorm,
    rowops_row_max,
    rowops_row_sum,
    rowops_softmax,
    rowops_softmax_causal,
    rowops_reload_tuning,
    rowops_status_string,
)
