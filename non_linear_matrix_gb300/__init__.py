"""GB300-native M2RNN recurrence: forward and BPTT backward CUDA kernels for
sm_103a behind a C-ABI library (``libm2rnn.so``), with a thin ctypes binding.

Importing the package loads nothing; the native library is loaded on first
use by :mod:`non_linear_matrix_gb300.m2rnn` and the binding fails loudly if it
is missing.  There is no CPU fallback.
"""

__all__ = ["m2rnn", "inputs"]
