"""Exact DeBERTa-v2/v3 disentangled attention (fused forward) for NVIDIA GB300.

The computation lives in ``libdfattn.so`` (hand-written sm_103a CUDA behind the
C ABI of ``include/df_attn.h``); ``binding`` is its ctypes marshalling layer and
``synth`` draws seeded synthetic inputs.  Build the library with
``exact_attention_deberta_gb300.build.build()``.
"""

__all__ = ["binding", "build", "synth"]


def __getattr__(name):
    if name in ("df_attn_fwd", "df_attn_plan", "df_rel_index_table", "df_attn_workspace_size",
                "df_attn_supported", "df_attn_get_device_status"):
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
