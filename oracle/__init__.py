"""CPU oracle for the top-k dispatch / combine path.  Test infrastructure:
only the tests, the smoke check and the benchmark's CPU-baseline leg use it."""
