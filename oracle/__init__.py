"""fp64 CPU oracle for KDA.  Test infrastructure only: the product path never
imports this package."""
