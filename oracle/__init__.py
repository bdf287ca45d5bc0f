"""Float64 CPU oracle for the MLA decode path (test infrastructure only).

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may use
this package.  The CUDA library never imports, links or calls it.
"""
from . import mla_oracle  # noqa: F401
