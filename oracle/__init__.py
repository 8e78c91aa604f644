"""CPU oracle for the MoE expert-layer forward (test infrastructure only; see
moe_oracle's header for who may import it)."""
