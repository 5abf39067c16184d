"""fp64 CPU oracle for QSA two-stage sparse attention (test infrastructure only)."""
