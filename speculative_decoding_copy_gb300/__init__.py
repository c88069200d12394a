"""GB300-native SwitchSD speculate-and-verify step (gate, retrieval,
block-triangular verification attention, acceptance) behind a C-ABI library.

The C entry points are re-exported under their own names; the library is
loaded on first use and every call raises if it has not been built.
"""
from ._binding import (  # noqa: F401
    SSD_BF16, SSD_CHAIN_ALWAYS, SSD_CHAIN_NONE, SSD_CHAIN_WHEN_GATE_OFF, SSD_F32, SSD_GREEDY, SSD_LOGITS_BF16,
    SSD_LOGITS_F32, SSD_OK, SSD_PROBS_F32, SSD_SAMPLE, SsdError, launch_count, lib, ssd_accept,
    ssd_accept_workspace_size, ssd_gate_match, ssd_read_device_error, ssd_retrieve, ssd_verify_attn,
    ssd_verify_attn_workspace_size, status_string)
