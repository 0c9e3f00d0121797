"""GB300-native (sm_103a) DSpark draft sampling and exact verification.

The computation lives in the CUDA library ``_build/libdspark.so`` (C ABI in
``include/dspark.h``); this package is its build script and a thin binding.
"""
from .binding import (BF16, F32, OP_ACCEPT_STATS, OP_MARKOV_SAMPLE, OP_RNN_SAMPLE, OP_STS_FIT, OP_VERIFY,
                      DsparkError, Workspace, accept_stats, accept_stats_grad, library_path, load, markov_launches,
                      markov_sample, rnn_launches, rnn_sample, status_string, sts_fit, verify, workspace_size)

__all__ = ["BF16", "F32", "OP_ACCEPT_STATS", "OP_MARKOV_SAMPLE", "OP_RNN_SAMPLE", "OP_STS_FIT", "OP_VERIFY",
           "DsparkError", "Workspace", "accept_stats", "accept_stats_grad", "library_path", "load", "markov_launches",
           "markov_sample", "rnn_launches", "rnn_sample", "status_string", "sts_fit", "verify", "workspace_size"]
