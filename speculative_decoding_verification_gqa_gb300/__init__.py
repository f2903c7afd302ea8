"""GB300-native speculative-decoding verification: GQA verify attention and greedy
acceptance as hand-written sm_103a CUDA kernels behind a C ABI (libspecverify.so).

Python entry points (argument marshalling over the C ABI; see ``api``):
``spec_verify_attn``, ``spec_verify_attn_paged``, ``spec_verify_attn_host_lengths``,
``spec_accept``, ``spec_accept_stochastic``, ``spec_draft_signals``, ``workspace_status``,
and ``plan_preview`` (the attention calls' work plan, computed on the host).
"""
from .api import (AttnDesc, SpecVerifyError, accept_workspace_bytes, load_library,
                  new_workspace, plan_preview, set_attn_kernel, set_profile_events,
                  set_unit_ctas, signals_workspace_bytes, spec_accept, spec_accept_stochastic,
                  spec_draft_signals,
                  spec_verify_attn, spec_verify_attn_host_lengths, spec_verify_attn_paged,
                  verify_workspace_bytes, workspace_status)

__all__ = ["AttnDesc", "SpecVerifyError", "accept_workspace_bytes", "load_library",
           "new_workspace", "plan_preview", "set_attn_kernel", "set_profile_events",
           "set_unit_ctas", "signals_workspace_bytes", "spec_accept", "spec_accept_stochastic",
           "spec_draft_signals",
           "spec_verify_attn", "spec_verify_attn_host_lengths", "spec_verify_attn_paged",
           "verify_workspace_bytes", "workspace_status"]
