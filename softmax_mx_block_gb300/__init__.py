"""GB300-native MX block-scaled attention with a reformulated softmax.

The computation lives in libfsa.so (CUDA for sm_103a, C ABI in include/fsa.h);
this package is a thin binding with the same entry-point names.  See
``_binding`` for the calls: fsa_mx_quantize, fsa_mx_quantize_qkv, fsa_attention_fwd,
fsa_attention_fwd_layers, fsa_attention_fwd_host, fsa_attention_fwd_bf16,
fsa_bf16_transpose_v, fsa_mx_sizes, fsa_tune_delta, fsa_mma_peak."""
from ._binding import (  # noqa: F401
    FSA_OK, FSA_ERR_INVALID_ARG, FSA_ERR_UNSUPPORTED_FMT, FSA_ERR_LAUNCH, FSA_ERR_TIMEOUT, FSA_ERR_NO_DEVICE,
    FSA_FMT_E4M3, FSA_FMT_E2M3, FSA_FMT_E2M1, FSA_FMT_E2M1_EFQ, FSA_FMT_E3M2, FSA_FMT_NVFP4, FSA_MX_ROWS, FSA_MX_COLS_T,
    FSA_EXP_POLY, FSA_EXP_MUFU, FSA_EXP_SPLIT, FMT_BY_NAME, FsaError, MxTensor,
    fsa_mx_sizes, fsa_mx_quantize, fsa_mx_quantize_qkv, fsa_attention_fwd, fsa_attention_fwd_bf16, fsa_bf16_transpose_v,
    default_opts, new_stats, read_stats, status_string, load, library_path,
    FSA_OUT_F32, FSA_OUT_BF16, DebugDump, fsa_attention_fwd_layers, fsa_tune_delta, fsa_mma_peak,
    HostCallBuffers, fsa_attention_fwd_host,
)
from ._build import build  # noqa: F401
