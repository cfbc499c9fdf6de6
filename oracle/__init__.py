"""CPU oracle for the LoRA linear layer (test infrastructure; never on the product path)."""
