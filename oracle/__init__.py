"""Float64 CPU oracle for the LOCKS decode path (test infrastructure only)."""
