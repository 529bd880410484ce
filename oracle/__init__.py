"""Float64 CPU oracle for the WaveFilter KV-filtering path (test infrastructure only).

Only tests, the package smoke check and the benchmark's CPU-baseline leg may
import this package.  It shares no code with the CUDA path.
"""
from .wavefilter_oracle import *  # noqa: F401,F403
from .wavefilter_oracle import __all__  # noqa: F401
