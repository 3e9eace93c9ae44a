"""DSpark per-round speculative-decoding sampling path on GB300 (sm_103a).

The compute lives in ``libdspark.so`` (C-ABI in include/dspark.h); this package
holds its ctypes binding (``binding``), the in-tree build (``build``) and the
seeded synthetic workloads (``workload``).
"""
from . import workload  # noqa: F401
from .binding import (  # noqa: F401
    DSparkError,
    dspark_draft_sample,
    dspark_draft_sample_rnn,
    dspark_draft_sample_rnn_w2t,
    dspark_draft_sample_w2t,
    dspark_transpose_w2,
    draft_rnn_workspace_bytes,
    dspark_profile_start,
    dspark_profile_stop,
    dspark_read_device_status,
    dspark_schedule,
    dspark_schedule_capacity,
    dspark_schedule_topk,
    dspark_schedule_threshold,
    dspark_stream_probe,
    dspark_sts_calibrate,
    dspark_verify,
    dspark_verify_packed,
    draft_workspace_bytes,
    schedule_workspace_bytes,
    sts_workspace_bytes,
    verify_workspace_bytes,
)

__all__ = [
    "dspark_draft_sample",
    "dspark_draft_sample_rnn",
    "dspark_draft_sample_rnn_w2t",
    "dspark_draft_sample_w2t",
    "dspark_transpose_w2",
    "draft_rnn_workspace_bytes",
    "dspark_schedule",
    "dspark_schedule_capacity",
    "dspark_schedule_topk",
    "dspark_schedule_threshold",
    "dspark_sts_calibrate",
    "sts_workspace_bytes",
    "dspark_verify",
    "dspark_verify_packed",
    "dspark_read_device_status",
    "dspark_profile_start",
    "dspark_profile_stop",
    "dspark_stream_probe",
    "draft_workspace_bytes",
    "schedule_workspace_bytes",
    "verify_workspace_bytes",
    "DSparkError",
    "workload",
]
