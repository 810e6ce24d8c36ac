"""Paged latent (MLA) KV-cache attention for one GB300 (sm_103a).

The compute path is the C-ABI library ``libtf_paged_mla.so`` (hand-written
CUDA, declared in ``include/tf_paged_mla.h``); ``paged_mla_kv_gb300.binding``
is its thin Python binding.  Importing this package loads nothing: the binding
loads the library on first use and raises if it has not been built.
"""

__all__ = ["binding", "synth"]
