"""The bias GEMM's fp32-backbone epilogue, which no bf16 case reaches (the
RNN-head draft's second product runs on it): fp32 backbone rows at three
ranks and ragged batches, against the oracle.  Joins tests/test_markov_gpu.py
once it has run on a GB300."""
import numpy as np
import pytest
import torch

import synth
from test_markov_gpu import _both, _check, ds  # noqa: F401

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,V,r", [(5, 4096, 256), (33, 2056, 128), (160, 2056, 64)])
def test_markov_fp32_backbone(ds, oracle, B, V, r):
    w = synth.decode_verify_tile(V=V, B=B, r=r, H=0, seed=3001 + B)
    w.backbone = w.backbone.float().contiguous()
    _check(*_both(ds, oracle, w, with_h=False), with_h=False)
