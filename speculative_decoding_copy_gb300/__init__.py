"""GB300-native SwitchSD speculate-and-verify step (gate, retrieval,
block-triangular verification attention, acceptance) behind a C-ABI library."""
