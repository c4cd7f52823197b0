"""fp64 CPU oracle for paged decode attention -- test infrastructure only."""
