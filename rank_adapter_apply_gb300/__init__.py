"""GB300 (sm_103a) multi-LoRA delta path: C-ABI library plus a thin binding.

Importing the package loads nothing native; ``rank_adapter_apply_gb300.binding``
loads the compiled library and raises if it is missing.
"""
