"""CPU oracle of the MoE layer forward: TEST INFRASTRUCTURE.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline / reference
arm may import this package; the library never does.
"""
