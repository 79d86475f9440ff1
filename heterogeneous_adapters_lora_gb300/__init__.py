"""GB300-native multi-tenant LoRA delta (BGMV / SGMV / MoE-LoRA) behind a C ABI.

Importing the package has no side effects; ``heterogeneous_adapters_lora_gb300.lora``
loads the CUDA library (``liblora_gb300.so``) on first use and raises if it is
missing.  ``heterogeneous_adapters_lora_gb300.inputs`` draws the seeded inputs.
"""
__all__ = ["inputs", "lora"]
