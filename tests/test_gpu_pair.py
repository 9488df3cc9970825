"""The two-CTA prefill kernel (kernel 2 of sala_gla_set_prefill_kernel) on every small and
edge case of the prefill parity suite and on the failure path.

By default sala_gla_chunk_fwd picks the kernel per call: the full varlen and long workloads of
test_gpu_parity.py run on the two-CTA kernel, the small cases there on the one-unit-per-SM
kernel. Here the two-CTA kernel is forced, so both kernels meet every ragged length, empty
and one-token sequence, exact-route chunk (g = -30), zero gate, initial state and head count,
and the headline workload, against the same fp64 oracle and tolerances.
"""
import pytest

from test_gpu_parity import (  # noqa: F401  (fixture and tests collected here again)
    sg, test_full_sala_layer, test_packed_equals_separate_calls, test_prefill_batched_rows,
    test_prefill_g_very_negative, test_prefill_g_zero, test_prefill_h0_only,
    test_prefill_head_counts, test_prefill_mixed_segment_shapes, test_prefill_ragged_lengths,
    test_prefill_tiny_workload, test_prefill_varlen_with_empty_and_short,
    test_prefill_without_final_state, test_prefill_zero_tokens_returns_h0,
    test_split_call_equals_single_call, test_one_token_prefill_equals_decode_step,
    test_decode_steps_equal_prefill, test_bad_cu_seqlens_reported_and_skipped)
from test_gpu_failure import test_withheld_hand_off_times_out_then_next_call_is_correct  # noqa: F401

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def two_cta_kernel(sg):  # noqa: F811
    sg.set_prefill_kernel(2)
    yield
    sg.set_prefill_kernel(0)


def test_kernel_choice_rejects_unknown_values(sg):  # noqa: F811
    with pytest.raises(sg.SalaError):
        sg.set_prefill_kernel(3)
