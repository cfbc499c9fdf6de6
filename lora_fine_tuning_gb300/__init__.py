"""LoRA linear layer on NVIDIA GB300 (sm_103a)."""
