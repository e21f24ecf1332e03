"""FP64 CPU oracle of the KDA RecoverSSM step -- test infrastructure only.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline and
reference legs may import this package; the library never does.
"""
from . import kda_oracle  # noqa: F401
