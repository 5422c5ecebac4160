"""Plain CPU oracle of the native-sparse-attention hot path (test infrastructure only)."""
