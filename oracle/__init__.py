"""CPU oracle (test infrastructure only; never called by the product path)."""
