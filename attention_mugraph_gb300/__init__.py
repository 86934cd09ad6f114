"""GB300-native fused exp-normalised GQA attention (Mirage's GQA kernel graph).

``O = (exp(Q.K) / rowsum(exp(Q.K))) . V`` with Q (B,M,d), K (B,d,N), V (B,N,d) in fp16,
computed by hand-written sm_103a kernels behind the C ABI of ``include/mg_attn.h``; the
launch-floor and exponential-rate measurements of ``include/mg_diag.h`` come with it.
The CUDA library is loaded lazily on first use; importing this package needs no GPU.
"""

from ._lib import (MG_ERR_CONFIG, MG_ERR_CUDA, MG_ERR_INSUFFICIENT_SMEM, MG_ERR_INVALID_ARG, MG_ERR_LAYOUT,
                   MG_ERR_TIMEOUT, MG_ERR_UNSUPPORTED, MG_FLAG_INJECT_TIMEOUT, MG_FLAG_ISOLATED, MG_FLAG_NO_CLUSTER, MG_FLAG_NO_EARLY_LOADS, MG_FLAG_NO_PDL, MG_FLAG_NO_Q_PAIRS, MG_FLAG_NO_STREAM_K, MG_FLAG_NO_SWAP_AB, MG_FLAG_PUSH_COMBINE, MG_FLAG_Q_PAIRS,
                   MG_FLAG_STREAM_K, MG_FLAG_SWAP_AB,
                   MG_FLAG_QK_NORM, MG_FLAG_SAFE_SOFTMAX, MG_OK,
                   MG_QKNORM_EPS, MgAttnError,
                   Plan, attention, diag_exp_rate, diag_launch_floor, load_library, mg_attn_plan, mg_attn_query,
                   run_noalloc)

__all__ = ["Plan", "attention", "run_noalloc", "load_library", "mg_attn_plan", "mg_attn_query", "MgAttnError", "MG_OK",
           "MG_ERR_INSUFFICIENT_SMEM", "MG_ERR_LAYOUT", "MG_ERR_CONFIG", "MG_ERR_INVALID_ARG", "MG_ERR_UNSUPPORTED",
           "MG_ERR_CUDA", "MG_ERR_TIMEOUT", "MG_FLAG_NO_PDL", "MG_FLAG_INJECT_TIMEOUT", "MG_FLAG_NO_CLUSTER",
           "MG_FLAG_SAFE_SOFTMAX", "MG_FLAG_QK_NORM", "MG_FLAG_Q_PAIRS", "MG_FLAG_NO_Q_PAIRS",
           "MG_FLAG_STREAM_K", "MG_FLAG_NO_STREAM_K", "MG_FLAG_SWAP_AB",
           "MG_FLAG_NO_SWAP_AB", "MG_FLAG_PUSH_COMBINE", "MG_FLAG_NO_EARLY_LOADS", "MG_FLAG_ISOLATED",
           "MG_QKNORM_EPS", "diag_launch_floor", "diag_exp_rate"]
