"""CPU oracle (float64 numpy) for quantized-KV decode attention.

Test infrastructure: only tests/, __graft_entry__.smoke() and bench.py's
cpu_baseline / reference leg may import it.  It shares no code with the CUDA
library and never imports it.
"""
from . import kvq_oracle  # noqa: F401
