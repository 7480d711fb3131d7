"""CPU oracle for the MXFP8 path (test infrastructure only).

Import restrictions: only tests/, __graft_entry__.smoke() and bench.py's
CPU-baseline and reference legs may use this package.
"""
from .mx_oracle import *  # noqa: F401,F403
