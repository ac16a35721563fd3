"""fp64 CPU oracle for the KDA recurrence (test infrastructure only)."""
