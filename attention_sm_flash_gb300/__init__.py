"""GB300-native fused scaled-dot-product attention (forward and backward).

The compute path is the C-ABI library ``libattn.so`` built from ``csrc/`` for sm_103a;
``attention_sm_flash_gb300.attn`` is its thin ctypes binding. Importing this package
loads nothing: the binding loads the library on first use and raises if it is missing.
"""

__all__ = ["attn", "workloads", "metrics"]
