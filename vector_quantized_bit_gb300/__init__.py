"""GB300-native VQ KV-cache decode attention (VecInfer's hot path).

The compute lives in ``_build/libvqkv.so`` (hand-written CUDA for sm_103a,
C ABI in ``include/vqkv.h``); this package only marshals arguments to it
(``_lib``), builds it (``_build``) and generates seeded synthetic workloads
(``synth``, ``calib``).
"""
from ._lib import (  # noqa: F401
    VQKV_MODE_VQ2,
    VQKV_MODE_VQ15,
    VQKV_MODE_VQ125,
    VQKV_MODE_VQ3,
    VQKV_MODE_VQ4,
    VQKV_ROLE_K,
    VQKV_ROLE_V,
    VqkvError,
    decode_args,
    decode_workspace,
    encode_args,
    vqkv_code_bytes,
    vqkv_decode_attn,
    vqkv_decode_num_splits,
    vqkv_decode_workspace_bytes,
    vqkv_encode,
)
