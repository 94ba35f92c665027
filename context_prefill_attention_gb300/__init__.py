"""PCP attention for GB300 (sm_103a): the Python face of libpcp.

The functions keep the C ABI's names (include/pcp.h); they only marshal
arguments. The CUDA library must be built (``build.build()``); without it every
call raises — there is no CPU or eager fallback.
"""
from ._lib import (EXPORTS, PCP_ATTN_DECODE_SMS, PCP_ATTN_KV_SHARDS,  # noqa: F401
                   PCP_ATTN_SEPARATE_CONTEXT, PCP_ATTN_SPLIT_AT_ROW_START, PCP_ERR_ALIGN, PCP_ERR_ARG,
                   PCP_ERR_CUDA, PCP_ERR_RANGE, PCP_ERR_TIMEOUT, PCP_ERR_UNSUPPORTED, PCP_ERR_WORKSPACE,
                   PCP_OK, PCP_SPLIT_CONTIGUOUS, PCP_SPLIT_DUAL_CHUNK, ROW_FIELDS, PcpError, load,
                   pcp_attn_varlen, pcp_attn_varlen_fp8kv, pcp_attn_varlen_noalloc, pcp_attn_workspace_size,
                   pcp_build_row_plan, pcp_decode_sms, pcp_kv_cache_write, pcp_kv_cache_write_fp8,
                   pcp_lse_merge, pcp_mask_slots_for_shard, pcp_set_profile_events)
from .step import PcpStep, debug_plan, plan_summary, write_positions  # noqa: F401
