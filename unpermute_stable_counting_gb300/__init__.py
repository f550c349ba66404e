"""GB300-native MoE expert-grouped token reorder.

Two operations behind a C ABI (include/moe_reorder.h), run as hand-written
CUDA kernels for sm_103a:

* ffnwb_batching -- FFN-worker batching: stable counting sort of the slots by
  expert key, row gather (+ INT8 dynamic scale), id lookups, group_list and
  actual_token_num (flat arrays, or a ScheduleContext read on the device);
* moe_permute    -- routing-map permute, the producer of the unpermute's input;
* moe_update_expert -- logical to physical expert ids through the EPLB table,
  with threshold pruning;
* moe_unpermute  -- routing-map unpermute, four branches (padded or not, with
  or without probs), deterministic fp32 gather-reduce.

Importing the package does not load the CUDA library; the first call does,
and fails loudly if the library was not built.
"""
from .api import (DT_BF16, DT_F16, DT_F32, DT_INT8, MoeReorderError, batching_context_workspace_size,
                  batching_outputs, batching_workspace_size, ffnwb_batching, ffnwb_batching_context,
                  moe_permute, moe_unpermute, moe_update_expert, permute_workspace_size, profile_set_events,
                  unpermute_outputs, unpermute_workspace_size)

__all__ = ["ffnwb_batching", "ffnwb_batching_context", "moe_unpermute", "moe_permute", "moe_update_expert",
           "permute_workspace_size",
           "batching_context_workspace_size", "batching_workspace_size",
           "unpermute_workspace_size", "batching_outputs", "unpermute_outputs",
           "profile_set_events", "MoeReorderError", "DT_F16", "DT_BF16", "DT_INT8", "DT_F32"]
