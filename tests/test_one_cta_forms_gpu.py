"""The one-CTA kernel forms (GPU), against the fp64 oracle.

By default the prefill projections with more than 128 rows and the head_dim
256 attention run on 2-CTA clusters (tcgen05 cta_group::2); the one-CTA
kernels remain for problems or devices where that cluster shape cannot be
placed.  gqa_set_cta_pairs(0) makes every launch take the one-CTA forms, and
this module re-runs the projection and head_dim 256 parity tests that way
(the same functions as in tests/test_parity_gpu.py and tests/test_d256_gpu.py,
collected again here under the switch).

Tolerance: as in those modules (tests/parity.py).
"""
import pytest

from transformer_gqa_attention_qkv_gb300 import binding as gq
from test_d256_gpu import (test_attention_cached_d256, test_attention_stage_d256,  # noqa: F401
                           test_forward_d256_gemma3_width)
from test_parity_gpu import test_oproj_residual_stage, test_qkv_projection_stage  # noqa: F401

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def one_cta_forms():
    prev = gq.gqa_set_cta_pairs(False)
    yield
    gq.gqa_set_cta_pairs(prev)
