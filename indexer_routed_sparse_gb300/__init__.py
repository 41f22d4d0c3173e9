"""Indexer-routed sparse GQA attention for GB300 (sm_103a).

The compute lives in libirs.so (CUDA kernels behind the C ABI of include/irs.h);
this package is its thin Python binding. Names follow the C entry points:

* ``sparse_index_score_topk(qI, kI, w, cu_seqlens, c, budget) -> route_ids``
* ``sparse_gqa_attn_fwd(q, k, v, route_ids, scale) -> (out, lse)``
* ``sparse_gqa_attn_bwd(q, k, v, route_ids, out, lse, dout, scale) -> (dq, dk, dv)``
* ``topk_from_scores(scores, cu_seqlens, c, budget) -> route_ids``
* ``compose_window_routes(route_ids, cu_seqlens, window) -> route_ids``
* ``sparse_index_score_topk_grouped`` / ``sparse_gqa_attn_fwd_grouped``: per-KV-group routes
* ``indexer_projection(hidden, weight, Hi, Di) -> (qI, kI, w)``: the indexer's projections
* ``region_summaries(kI, z, cu_seqlens, c)`` and ``sparse_index_score_topk_summaries``:
  Step-5 learned-logit region summaries and the indexer that scores them
"""
from ._binding import (  # noqa: F401
    DEVERR_CU_SEQLENS,
    DEVERR_ROUTE_ID,
    DEVERR_TIMEOUT,
    LIB_PATH,
    check_bounded_wait,
    check_device_errors,
    compose_window_routes,
    device_error_flag,
    exported_symbols,
    index_front_operands,
    index_workspace_bytes,
    indexer_projection,
    lib,
    read_device_errors,
    region_summaries,
    sparse_gqa_attn_bwd,
    sparse_gqa_attn_fwd,
    sparse_gqa_attn_fwd_grouped,
    sparse_index_score_topk,
    sparse_index_score_topk_grouped,
    sparse_index_score_topk_summaries,
    topk_from_scores,
)
