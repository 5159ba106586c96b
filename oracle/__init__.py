"""CPU oracle of the compression pass: test infrastructure only (see zipage_oracle)."""
