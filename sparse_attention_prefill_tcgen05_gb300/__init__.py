"""GB300 (sm_103a) dense prefill indexer: fp8 / fp4 MQA logits on tcgen05 tensor
cores with a ragged, causal, exactly merged per-row top-k.

The compute lives in ``libindexer.so`` (CUDA kernels behind the C ABI of
``include/indexer.h``); :mod:`._lib` is a ctypes binding with the same entry
point names, and :mod:`.workloads` draws seeded synthetic inputs.
"""
from ._lib import (  # noqa: F401
    IDX_K_FP4_E2M1_UE8M0, IDX_K_FP8_E4M3, IDX_Q_FP4_E2M1_UE8M0, IDX_Q_FP8_E4M3, IDX_OK, IDX_SELECT_AUTO, IDX_SELECT_STREAM, IndexerError, Plan, indexer_candidate_blocks,
    indexer_expand_mask, indexer_fused_topk, indexer_logits, indexer_plan, indexer_selftest_timeout,
    indexer_launch_count, indexer_profile_main_kernel, indexer_set_wait_budget, indexer_status, indexer_topk, indexer_version,
    indexer_chunk_rows, indexer_page_indices, indexer_candidate_blocks_tail,
    indexer_fused_topk_mapped, indexer_convert_fp4, indexer_fallback_rows,
    lib,
)
