"""CPU oracle for QK-Normed MLA decode (fp64 numpy).

Test infrastructure only: tests/, __graft_entry__.smoke() and bench.py's CPU
baseline leg may use it; the CUDA library never does.
"""
from .qkmla_oracle import *  # noqa: F401,F403
from .qkmla_oracle import __all__  # noqa: F401
