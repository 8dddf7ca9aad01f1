"""GB300-native split-KV sparse-MLA decode.

The compute path is the C-ABI library ``libsplitkv.so`` (hand-written CUDA for
sm_103a, declared in ``include/mla_split.h``); ``binding`` exposes each entry
point under its C name, and ``workloads`` draws seeded synthetic inputs.
"""
from .binding import (  # noqa: F401
    MLA_FORCE_BALANCED, MLA_OUT_BF16, MLA_OUT_E4M3, MLA_OUT_F32, MLA_STATUS_TIMEOUT, MlaPlan, SdpaPlan, SplitKVError,
    mla_abi_version, mla_decode_plan, mla_get_status, mla_selftest_wait_timeout, mla_sparse_decode,
    mla_sparse_decode_host,
    mla_sparse_decode_noalloc, mla_workspace_init, mla_plan_set_partials_bf16, mla_set_wait_limit_ns,
    mla_set_index_checks,
    mla_sparse_decode_direct, mla_sparse_decode_split, mla_split_combine, sdpa_fp8_decode,
    sdpa_fp8_decode_direct, sdpa_fp8_decode_plan, sdpa_fp8_decode_split, sdpa_split_combine,
)
