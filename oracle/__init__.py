"""CPU oracle of the 4-bit MoE layer (test infrastructure only; see moe_oracle)."""
