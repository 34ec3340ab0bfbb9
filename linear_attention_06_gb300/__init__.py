"""GB300-native Kimi Delta Attention (KDA): prefill and decode behind the C ABI
of libkda (include/kda.h).  This package is the thin Python side of it."""
from ._lib import (KdaError, KdaShape, kda_check_cu_seqlens, kda_decode_step,  # noqa: F401
                   kda_decode_step_gated, kda_device_status, kda_frontend, kda_prefill, kda_prefill_checkpointed,
                   kda_prefill_frontend, kda_prefill_gated, kda_prefill_split, kda_prefill_split_workspace_size, kda_selftest_timeout, lib,
                   status_string, version)
from . import workloads  # noqa: F401

__all__ = ["kda_prefill", "kda_prefill_checkpointed", "kda_prefill_frontend", "kda_prefill_gated",
           "kda_prefill_split",
           "kda_prefill_split_workspace_size", "kda_decode_step",
           "kda_decode_step_gated", "kda_frontend", "kda_check_cu_seqlens",
           "kda_device_status", "kda_selftest_timeout",
           "status_string", "version", "lib", "KdaError", "KdaShape", "workloads"]
