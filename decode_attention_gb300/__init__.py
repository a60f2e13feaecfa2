"""GB300 (sm_103a) decode-step attention core of the Gemma-4-31B text decoder.

The two ``attn.core`` variants of the gemma-4-31B Model Spec ("Compute-graph
nodes" table): slidingDecodeGQA (32 query / 16 KV heads, head dim 256, window of
the last 1024 positions) and decodeGQA (32 query / 4 KV heads, head dim 512, full
history), attention scale 1, over a contiguous or a 16-position paged KV cache.

The compute runs in ``libgqadecode.so`` (hand-written CUDA for sm_103a behind the
C ABI in ``include/gqa_decode.h``); this package only marshals arguments.
"""
from ._native import (  # noqa: F401
    EXPORTED_SYMBOLS,
    GQA_DEVICE_BAD_LENGTH,
    GQA_DEVICE_BAD_PAGE,
    GQA_DEVICE_WAIT_TIMEOUT,
    GQA_KERNEL_NONE,
    GQA_KERNEL_SPLIT_DECODE,
    GQA_KERNEL_TCGEN05,
    GQA_TEST_SINGLE_PIECE,
    GQA_TEST_STALL,
    GQA_MAX_QUERIES_GLOBAL,
    GQA_MAX_QUERIES_SLIDING,
    GQA_MAX_SEQ,
    GQA_ERR_CUDA,
    GQA_ERR_INVALID_ARGUMENT,
    GQA_ERR_UNSUPPORTED,
    GQA_ERR_WORKSPACE,
    GQA_OK,
    GQA_OUT_BF16,
    GQA_OUT_F32,
    PAGE_SIZE,
    GQAError,
    gqa_decode,
    gqa_decode_keqv,
    gqa_decode_keqv_kernel,
    gqa_decode_keqv_paged,
    gqa_decode_mq,
    gqa_decode_mq_paged,
    gqa_decode_noalloc,
    gqa_prepare_decode,
    gqa_prepare_decode_paged,
    gqa_decode_ring,
    gqa_decode_paged,
    gqa_check_inputs_host,
    gqa_device_status,
    gqa_get_test_mode,
    gqa_noalloc_status,
    gqa_set_test_mode,
    gqa_status_string,
    gqa_workspace_init,
    gqa_workspace_size,
    gqa_workspace_size_mq,
    library_path,
    load_library,
    new_workspace,
)
