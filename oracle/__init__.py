"""fp64 CPU oracle for the MLA decode step. TEST INFRASTRUCTURE: only the tests,
__graft_entry__.smoke() and bench.py's CPU-baseline leg may import it."""
