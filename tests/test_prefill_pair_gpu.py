"""The bf16 / fp16 prefill in its CTA-pair form (tcgen05 cta_group::2, M = 256
over two SMs, 512-row work items), selected with pa_set_prefill_cta_pairs:
the same parity cases as the one-CTA form, against the same oracle (FlashMLA
TENSOR_SHAPES "Prefill writes into paged cache"; Modular flare_mla_prefill).
"""
import pytest

from paged_kv_attention_fwd_gb300 import binding as B

from .test_prefill_gpu import gpu  # noqa: F401  (module fixture: device and build)
from .test_prefill_gpu import (  # noqa: F401  (collected here with CTA pairs on)
    test_chunked_prefill_full_size_sampled,
    test_fp16_prefill,
    test_large_outputs_under_the_ulp_rule,
    test_mla_prefill_full_size_sampled,
    test_mla_ragged_prefill,
    test_paged_chunked_prefill,
    test_paged_prefill_poisoned_tail_rows_and_pages,
    test_persistent_work_counters_reset,
    test_prefill_deterministic,
    test_ragged_prefill,
    test_ragged_prefill_explicit_offsets,
)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cta_pairs(gpu):  # noqa: F811
    B.pa_set_prefill_cta_pairs(True)
    yield
    B.pa_set_prefill_cta_pairs(False)
