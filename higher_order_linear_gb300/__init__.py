"""Masked second-order Higher-order Linear Attention (HLA) for NVIDIA GB300.

The computation lives in ``libhla2.so`` (CUDA, sm_103a), whose C ABI is
declared in ``include/hla2.h``; ``hla2`` is the thin Python binding.
"""
from .hla2 import (  # noqa: F401
    HLA2Error,
    ahla_state_len,
    hla2_ahla_forward,
    hla2_ahla_step,
    hla2_chunk_summaries,
    hla2_decay_forward,
    hla2_decay_step,
    hla2_device_status,
    hla2_forward,
    hla2_forward_noalloc,
    hla2_forward_plan,
    hla2_forward_workspace,
    hla2_last_error_detail,
    hla2_scan,
    hla2_state_to_pform,
    hla2_step,
    hla2_step_pform,
    hla2_unmasked_forward,
    hla2_unmasked_step,
    pform_record_len,
    record_len,
    unmasked_state_len,
)
