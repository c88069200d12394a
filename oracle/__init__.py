"""CPU oracle of the SwitchSD speculate-and-verify step (test infrastructure only)."""
