"""ISD verify/accept step for B300 (sm_103a): Python binding of libidlm.so.

The binding only marshals arguments: every step of the path runs in the CUDA
kernels of ``csrc/``.  Importing the package does not load the library; the
first call does, and raises if the library was not built.
"""

from ._lib import (  # noqa: F401,E402
    IDLM_BF16, IDLM_F32, MODE_FRESH, MODE_FULL, PROPOSE_ARGMAX, PROPOSE_SAMPLE, IDLMError,
    idlm_gated_lora, idlm_gated_lora_workspace_size, idlm_gated_lora_grouped,
    idlm_gated_lora_grouped_workspace_size, idlm_isd_accept, idlm_isd_accept_noalloc,
    idlm_isd_accept_commit, idlm_isd_accept_workspace_size, idlm_isd_attention,
    idlm_isd_attention_workspace_size,
    idlm_kv_commit, idlm_synth_logits, idlm_isd_advance, idlm_risd_layer,
    idlm_risd_layer_workspace_size, idlm_lm_head_accept, idlm_lm_head_accept_workspace_size,
    layer_weights, lib, version)
