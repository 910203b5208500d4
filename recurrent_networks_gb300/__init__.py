"""GB300-native head-wise recurrent scan (LSTM, GRU, Elman, sLSTM): forward and
backward through time in hand-written sm_103a CUDA kernels behind a C ABI
(include/rnn.h, librnn_gb300.so)."""
from .functional import flashrnn  # noqa: F401

__all__ = ["flashrnn"]
