"""libneattn binding (placeholder until the C-ABI lands)."""
