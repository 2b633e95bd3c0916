"""The tensor-core throughput probe computes right before its rate is used:
one round of four M = 128, N = 256 MMAs per operand kind (f16, E4M3 and
block-scaled E2M1 with unit scales) against the exact host product of the same
operands (small values, so every product and sum is exact in fp32)."""
import pytest

from sparse_attention_prefill_gb300 import peaks

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", list(peaks.KINDS))
def test_probe_products_exact(name):
    assert peaks.check(peaks.KINDS[name]) == 0.0
