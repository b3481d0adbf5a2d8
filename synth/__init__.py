"""Seeded synthetic inputs for the absorbed-MLA decode path.

This package only draws random numbers and lays them out (paged caches,
block tables, length mixes).  It holds none of the method's arithmetic:
values are drawn in float64 with numpy's PCG64 generator and stored in the
kernel's input dtypes with torch's own casts (bf16, float8_e4m3fn).  Both the
CUDA path and the fp64 oracle consume the very same stored bytes.
"""

from .workloads import *  # noqa: F401,F403
