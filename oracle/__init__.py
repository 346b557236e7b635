"""CPU oracle of the Q4_K mixture-of-experts FFN (test infrastructure only).

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg import
this package.  It is a plain C implementation (oracle.c) in fp64, loaded
through ctypes, and shares no code with the CUDA path.

Parity pins (tests/test_oracle_pins.py) tie every function here to the
Q4_K definition, closed forms, invariants, library routines and brute
force; none is "parity unpinned".
"""
from .oracle import *  # noqa: F401,F403
