"""Test infrastructure: the fp64 CPU oracle of the verify step (see vfy_oracle.py).

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may import this package.
"""
