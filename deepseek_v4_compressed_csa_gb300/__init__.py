"""One layer of DeepSeek-V4 Compressed Sparse Attention on GB300 (sm_103a).

The compute lives in libcsa.so (hand-written CUDA, C ABI in include/csa.h);
this package is its thin Python binding.  Importing it does not load the
library; the first call does, and fails loudly if it was not built.
"""
from ._binding import (  # noqa: F401
    CSA_BF16, CSA_F32, DEV_CAPACITY, DEV_RANGE, DEV_ROLLBACK, DEV_STATE, EXPORTS, FP8_ROW_BYTES, LIB_PATH,
    OP_ATTEND_DECODE, OP_ATTEND_PREFILL, OP_ATTEND_PREFILL_VARLEN, OP_COMPRESS, OP_COMPRESS_PAIR, OP_COMPRESS_VARLEN,
    OP_INDEX_TOPK, Compressor, CSAError, Layer, advance_positions, attend_decode, attend_prefill_chunk,
    attend_prefill_varlen, attend_verify, compress_append, compress_append_pair, compress_append_varlen,
    frontier_slots, index_rows_fp8, index_topk, index_topk_overlapped, index_topk_static, index_topk_verify,
    kernel_launches, load_library, static_scratch_bytes, trim, workspace_size,
)
