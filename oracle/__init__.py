"""fp64 CPU oracle for the KDA recurrence. TEST INFRASTRUCTURE ONLY: imported by the
tests, the smoke check and the bench's CPU-baseline leg, never by the library."""
