"""GB300-native WaveFilter KV-filtering path (DWT -> coarse Top-K -> recursive
filtering -> sparse gather -> eq. (3) attention), hand-written CUDA for sm_103a
behind a C ABI (``include/wavefilter.h``).

The CUDA library is loaded on first use by :mod:`wavelet_guided_sparse_gb300.binding`;
importing the package (or :mod:`.workloads`) does not touch the GPU.
"""

__version__ = "0.1.0"
