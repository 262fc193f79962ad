"""fp64 CPU oracle for exact DeBERTa disentangled attention (test infrastructure only)."""
